// A chain of dependent Q4_K dequant-GEMVs in one persistent launch
// (epq_gemv_chain): the decode step of a dense decoder is such a chain --
// every projection reads the output of the one before it.
//
// [H] "速度上限：带宽 ÷ 权重字节数": decode streams every packed weight once
// per token, so a step is bounded by HBM bandwidth / weight bytes.  Issued as
// one kernel per matrix, every matrix boundary drains the HBM stream: the
// next kernel's CTAs cannot load a byte before the previous kernel's CTAs
// leave the SMs.  Here one CTA per SM (a cooperative launch, so all are
// resident) walks the whole chain:
//   * its shared-memory ring streams the weights of its row range of every
//     matrix in chain order -- weights depend on nothing, so the copies for
//     matrix k+1 are already in flight (or landed) while matrix k finishes;
//   * between matrices a grid-wide barrier (one atomic counter and a
//     generation word in the caller's workspace, bounded waits) makes matrix
//     k's output visible before matrix k+1 reads it as x;
//   * each matrix runs the tensor-core dot products of gemv_tc.cu with all
//     16 warps on every 8-row block (warp w takes superblocks w, w+16, ...),
//     the last-arriving warp of a stage reducing the partial sums and
//     refilling the ring slot with the next stage of the chain.
// A ring slot holds 8 rows of a SwiGLU pair (gate and up) or up to three
// 8-row blocks; matrices whose 8 rows do not fit (wide rows, e.g. a down
// projection of 14336 columns) are streamed as 4-row stages, and one 8-row
// MMA block then reads its rows from two consecutive slots.  A CTA whose row
// range is shorter than the longest one runs empty stages, so the stage
// numbering is the same in every CTA and is computed on the host.
#include <algorithm>
#include <type_traits>

#include "gemv_tc_core.cuh"

namespace epq {
namespace {

using namespace tc;

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kNSB = 4;   // superblocks per warp: rows of up to 64 superblocks
constexpr int kMaxNbs = 3;
constexpr uint32_t kWarpArea = kFragWarpBytes;  // per-warp staging (prologue) / partial sums (stages)

struct ChainOp {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int rows_out, up_rows, row_bytes;  // rows_out <= 2^30
  int x_stride, y_stride;
  int cols, nsb, nbs, nst, stage0;
  int half;    // 1: 4-row stages, an 8-row block spans two of them
  int cfg;     // warp geometry: 0 (16 k-parts, 4 superblocks), 1/3 (8, 2), 2 (8, 1)
  int rq, rr;  // CTA b owns rows [b*rq + min(b, rr), ...), rq + (b < rr) of them
  int swiglu, rms;
  float rms_eps;
  int x_group, x_head_dim;
};

struct ChainParams {
  int nops, nv, stages, nsb_max;
  uint32_t slot_bytes;
  unsigned *bar;  // [0] arrivals, [1] generation
  unsigned *err;
  ChainOp ops[EPQ_CHAIN_MAX_OPS];
};

struct ChainLayout {
  uint32_t full, cnt, cbar, area, xs, scratch, total;
};

__host__ __device__ inline uint32_t al16c(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline ChainLayout chain_layout(int stages, uint32_t slot_bytes, int nsb_max) {
  ChainLayout L;
  uint32_t o = al16c(static_cast<uint32_t>(stages) * slot_bytes);
  L.full = o;
  o += 8u * stages;
  L.cbar = o;  // CTA barrier of the grid barrier: [0] warps arrived, [1] released
  o += 16u;
  L.cnt = o;  // per ring slot: warps done with it (monotonic)
  o = al16c(o + 4u * stages);
  L.area = o;  // per warp: x staging / partial sums [slot][block][row 8][vector 2][gate/up]
  o += kWarpArea * kWarps;
  L.xs = o;  // [group][superblock][t 4][vector 2][sub-block pair 2]: sums of x
  o = al16c(o + 4u * nsb_max * 16);  // nsb_max here: the largest groups x superblocks
  L.scratch = o;  // [warp][vector 2]: sums of squares
  o = al16c(o + 4u * 2 * kWarps);
  L.total = o;
  return L;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_relaxed_gpu(unsigned *p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) gemv_chain_kernel(const __grid_constant__ ChainParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const ChainLayout L = chain_layout(p.stages, p.slot_bytes, p.nsb_max);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
  uint64_t *cbar = reinterpret_cast<uint64_t *>(smem + L.cbar);
  unsigned *cnt = reinterpret_cast<unsigned *>(smem + L.cnt);
  float *xsum = reinterpret_cast<float *>(smem + L.xs);
  float *scratch = reinterpret_cast<float *>(smem + L.scratch);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.stages;

  const int bx = blockIdx.x;
  // global stage h (ring slot s) -> its matrix (a forward scan from `k`) and its copies
  auto issue = [&](int h, int s, int k) {
    while (k + 1 < p.nops && h >= p.ops[k + 1].stage0) ++k;
    const ChainOp &op = p.ops[k];
    const int rb = bx * op.rq + min(bx, op.rr);
    const int nrows = op.rq + (bx < op.rr ? 1 : 0);
    const int T = op.half ? 4 : 8 * op.nbs;
    const int r0 = (h - op.stage0) * T;
    const int nr = max(0, min(T, nrows - r0));
    const uint32_t rbytes = static_cast<uint32_t>(op.row_bytes);
    const uint32_t bytes = static_cast<uint32_t>(nr) * rbytes;
    uint8_t *dst = smem + static_cast<uint32_t>(s) * p.slot_bytes;
    mbar_arrive_expect_tx(&full[s], op.swiglu ? 2 * bytes : bytes);
    if (bytes) {
      const uint8_t *src = op.W + static_cast<int64_t>(rb + r0) * rbytes;
      bulk_g2s(dst, src, bytes, &full[s]);
      if (op.swiglu)
        bulk_g2s(dst + static_cast<uint32_t>(T) * rbytes, src + static_cast<int64_t>(op.up_rows) * rbytes, bytes,
                 &full[s]);
    }
  };
  const int total = p.ops[p.nops - 1].stage0 + p.ops[p.nops - 1].nst;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      cnt[s] = 0u;
    }
    mbar_init(&cbar[0], kWarps);
    mbar_init(&cbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int h = 0; h < min(S, total); ++h) issue(h, h, 0);  // weights depend on nothing upstream

  const int g = lane >> 2, t = lane & 3;
  const int cv = t & 1;
  uint32_t bq[kNSB][8][2];  // x operands of this warp's superblocks (the op's first NSB used)
  float fsc[kNSB];
  uint32_t magic = kH1024;
  asm volatile("" : "+r"(magic));
  const uint32_t csel = t == 0 ? 0x10u : (t == 1 ? 0x21u : (t == 2 ? 0x43u : 0x54u));
  const uint32_t ksel = t == 0 ? 0x32u : (t == 1 ? 0x43u : (t == 2 ? 0x65u : 0x76u));
  const int nsh = (t & 1) * 4;
  uint8_t *area = smem + L.area + warp * kWarpArea;
  pdl_wait();  // the first x is produced upstream

  for (int k = 0; k < p.nops; ++k) {
    const ChainOp &op = p.ops[k];
    // ---------------------------------------------------------------- grid barrier
    if (k > 0) {
      const unsigned par = (k - 1) & 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&cbar[0]);  // this warp's outputs of matrix k-1 are written
      if (tid == 0) {
        if (mbar_wait_poll(&cbar[0], par, p.err, DEVERR_RED_WAIT, k)) {
          // acq_rel at GPU scope (cumulative: it also releases the writes
          // this thread acquired from the CTA's warps through cbar[0])
          const unsigned gen0 = ld_acquire_gpu(&p.bar[1]);
          const unsigned old = atom_add_acq_rel_gpu(&p.bar[0], 1u);
          if (old == gridDim.x - 1) {
            st_relaxed_gpu(&p.bar[0], 0u);
            atom_add_acq_rel_gpu(&p.bar[1], 1u);  // release: the reset precedes the new generation
          } else {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(&p.bar[1]) == gen0) {
              if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_error(p.err, DEVERR_RED_WAIT, 0x10000u + k);
                break;
              }
            }
          }
        }
        mbar_arrive(&cbar[1]);
      }
      if (!warp_wait_poll(&cbar[1], par, p.err, DEVERR_RED_WAIT, k)) return;
    }

    // ---------------------------------------------------------------- the op
    // prologue and stages, compiled per warp geometry (KP warps per 8-row
    // block, NB = 16/KP groups alternating stages, NSB superblocks per warp)
    auto run = [&](auto kp_tag, auto nsb_tag, auto full_tag) -> bool {
      constexpr int KP = decltype(kp_tag)::value;
      constexpr int NSB = decltype(nsb_tag)::value;
      constexpr bool FULL = decltype(full_tag)::value;
      constexpr int NB = kWarps / KP;
      const int kq = warp % KP, grp = warp / KP;
      const XGather xg{op.x_group, op.x_head_dim};
      const int o_nsb = op.nsb;
      float *gxsum = xsum + grp * o_nsb * 16;
      uint32_t(&bqn)[NSB][8][2] = reinterpret_cast<uint32_t(&)[NSB][8][2]>(bq);
      float(&fscn)[NSB] = reinterpret_cast<float(&)[NSB]>(fsc);
      // x operands of this warp's superblocks (see gemv_tc.cu): one global
      // round trip, the superblock scales, sums of x per sub-block and of x^2
      {
        uint2 *frag = reinterpret_cast<uint2 *>(area);
        const int sub = lane >> 2, wi = lane & 3;
        const int tp = sub >> 1, jj = 4 * (sub & 1) + wi;
        float4 xr[NSB][2][2];
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          if (v < p.nv) {
            const float *xv = op.x + v * op.x_stride;
#pragma unroll
            for (int i = 0; i < NSB; ++i) {
              const int sb = FULL ? kq + i * KP : min(kq + i * KP, o_nsb - 1);
              const float *src = xv + xg.src(256 * sb + 8 * lane);
              // written by the previous op of this launch: coherent loads
              xr[i][v][0] = *reinterpret_cast<const float4 *>(src);
              xr[i][v][1] = *reinterpret_cast<const float4 *>(src + 4);
            }
          } else {
#pragma unroll
            for (int i = 0; i < NSB; ++i) xr[i][v][0] = xr[i][v][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        float ssq[2] = {0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < NSB; ++i) {
          const int sb = kq + i * KP;
          if (!FULL && sb >= o_nsb) {
#pragma unroll
            for (int j = 0; j < 8; ++j) bqn[i][j][0] = bqn[i][j][1] = 0u;
            fscn[i] = 0.0f;
            continue;
          }
          float fs[2] = {0.0f, 0.0f};
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            if (v >= p.nv) {  // no such vector: zero operands, nothing to convert
              if (wi == 0) gxsum[((sb * 4 + tp) * 2 + v) * 2 + (sub & 1)] = 0.0f;
              fs[v] = 0.0f;
            #pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int l0 = 4 * (4 * h + 2 * v) + tp;
                frag[jj * kFragRow + l0] = frag[jj * kFragRow + l0 + 4] = make_uint2(0u, 0u);
              }
              continue;
            }
            const float q0[8] = {xr[i][v][0].x, xr[i][v][0].y, xr[i][v][0].z, xr[i][v][0].w,
                                 xr[i][v][1].x, xr[i][v][1].y, xr[i][v][1].z, xr[i][v][1].w};
            float amax = 0.0f, s8 = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              amax = fmaxf(amax, fabsf(q0[e]));
              ssq[v] = fmaf(q0[e], q0[e], ssq[v]);
              s8 += q0[e];
            }
            amax = warp_max_all(amax);
            s8 += __shfl_xor_sync(0xffffffffu, s8, 1);
            s8 += __shfl_xor_sync(0xffffffffu, s8, 2);
            if (wi == 0) gxsum[((sb * 4 + tp) * 2 + v) * 2 + (sub & 1)] = s8;
            const int sig = min(126, max(-112, 15 - bound_exponent(amax)));
            fs[v] = exp2i(14 - sig);
            const float up = exp2i(sig);
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = q0[e] * up;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint2 hi, lo;
              hi.x = split_pair(q[h], q[h + 4], false);
              lo.x = split_pair(q[h], q[h + 4], true);
              hi.y = split_pair(q[h + 2], q[h + 6], false);
              lo.y = split_pair(q[h + 2], q[h + 6], true);
              const int l0 = 4 * (4 * h + 2 * v) + tp;
              frag[jj * kFragRow + l0] = hi;
              frag[jj * kFragRow + l0 + 4] = lo;
            }
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint2 r = frag[j * kFragRow + lane];
            bqn[i][j][0] = r.x;
            bqn[i][j][1] = r.y;
          }
          fscn[i] = cv ? fs[1] : fs[0];
          __syncwarp();
        }
        const float s0 = warp_sum_xor<32>(ssq[0]), s1 = warp_sum_xor<32>(ssq[1]);
        if (lane == 0) {
          scratch[warp * 2] = s0;
          scratch[warp * 2 + 1] = s1;
        }
        __syncwarp();
      }

      // stages of this group: h = stage0 + grp + j*NB (4-row stages only
      // with NB == 1, where a pass takes two consecutive stages)
      const int rb = bx * op.rq + min(bx, op.rr);
      const int re = rb + op.rq + (bx < op.rr ? 1 : 0);
      const int nblocks = (re - rb + 7) / 8;
      const int o_half = op.half, o_nbs = op.nbs, o_nst = op.nst, o_stage0 = op.stage0;
      const int M = op.swiglu ? 2 : 1;
      const uint32_t rbytes = static_cast<uint32_t>(op.row_bytes);
      const int step = o_half ? 2 : NB;       // stages per pass (of the whole CTA)
      const int bps = o_half ? 1 : o_nbs;     // 8-row blocks per stage pass
      const int T = o_half ? 4 : 8 * o_nbs;   // rows per stage
      float *myred = reinterpret_cast<float *>(area);  // [slot][block][row][vector][gate/up]
      // ring position of this warp's first stage
      int h = o_stage0 + (o_half ? 0 : grp);
      int cs = h % S;
      unsigned cph = static_cast<unsigned>(h / S) & 1u;
      for (; h < o_stage0 + o_nst; h += step) {
        const int s = cs;
        const int s2 = o_half ? (cs + 1 == S ? 0 : cs + 1) : cs;
        bool ok = warp_wait_poll(&full[s], cph, p.err, DEVERR_FULL_WAIT, h);
        if (ok && o_half) ok = warp_wait_poll(&full[s2], s2 == 0 ? cph ^ 1u : cph, p.err, DEVERR_FULL_WAIT, h + 1);
        if (!ok) return false;
        const uint8_t *sb0 = smem + static_cast<uint32_t>(s) * p.slot_bytes;
        const uint8_t *sb1 = smem + static_cast<uint32_t>(s2) * p.slot_bytes;
        const int i = h - o_stage0;
        const int blk0 = o_half ? i / 2 : i * o_nbs;  // first 8-row block of the stage
        const int nbl = max(0, min(bps, nblocks - blk0));
        for (int bi = 0; bi < nbl; ++bi) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            if (m == 1 && M == 1) break;
            float acc = 0.0f, am0 = 0.0f, am1 = 0.0f;
            const uint8_t *row = o_half ? (g < 4 ? sb0 + static_cast<uint32_t>(m * T + g) * rbytes
                                                 : sb1 + static_cast<uint32_t>(m * T + g - 4) * rbytes)
                                        : sb0 + static_cast<uint32_t>(m * T + 8 * bi + g) * rbytes;
            block_dot<KP, NSB, FULL>(row, kq, o_nsb, t, magic, csel, ksel, nsh, bqn, fscn, gxsum, acc, am0, am1);
            float p0 = (cv == 0 ? acc : 0.0f) - am0;
            float p1 = (cv == 1 ? acc : 0.0f) - am1;
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            if (t < 2) myred[(((s2 * kMaxNbs + bi) * 8 + g) * 2 + t) * 2 + m] = t == 0 ? p0 : p1;
          }
        }
        __syncwarp();
        const int nsl = o_half ? 2 : 1;
        for (int u = 0; u < nsl; ++u) {
          const int su = u == 0 ? s : s2;
          unsigned old = 0u;
          if (lane == 0) old = atom_add_acq_rel(&cnt[su], 1u);
          old = __shfl_sync(0xffffffffu, old, 0);
          __syncwarp();
          if (old + 1u != static_cast<unsigned>(KP)) continue;
          // last warp of the group on this slot; on the pass's last slot it
          // writes the outputs; then it resets the count and refills the slot
          if (u == nsl - 1) {
            float osc0 = 1.0f, osc1 = 1.0f;
            if (op.rms) {
              float q0 = 0.0f, q1 = 0.0f;
              for (int w = grp * KP; w < grp * KP + KP; ++w) {
                q0 += scratch[w * 2];
                q1 += scratch[w * 2 + 1];
              }
              osc0 = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q0, static_cast<float>(op.cols)), op.rms_eps)));
              osc1 = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q1, static_cast<float>(op.cols)), op.rms_eps)));
            }
            for (int o = lane; o < nbl * 16; o += 32) {
              const int bi = o >> 4, gg = (o >> 1) & 7, v = o & 1;
              const int row = rb + 8 * (blk0 + bi) + gg;
              if (row < re && v < p.nv) {
                float sg = 0.0f, su2 = 0.0f;
                const float *r = reinterpret_cast<const float *>(smem + L.area + grp * KP * kWarpArea) +
                                 (((s2 * kMaxNbs + bi) * 8 + gg) * 2 + v) * 2;
#pragma unroll
                for (int q = 0; q < KP; ++q) sg += r[q * (kWarpArea / 4)];
                if (M == 2) {
#pragma unroll
                  for (int q = 0; q < KP; ++q) su2 += r[q * (kWarpArea / 4) + 1];
                }
                const float os = v ? osc1 : osc0;
                float val = sg * os;
                if (M == 2) val = silu(val) * (su2 * os);
                if (op.residual) val += op.residual[v * op.y_stride + row];
                op.y[v * op.y_stride + row] = val;
              }
            }
            __syncwarp();
          }
          if (lane == 0) {
            cnt[su] = 0u;  // the slot's next users arrive only after its refill
            if (h + u + S < total) {
              fence_proxy_async();  // this CTA's reads of the slot precede the refill
              issue(h + u + S, su, k);
            }
          }
        }
        // advance by the pass's stages
        cs += step;
        while (cs >= S) {
          cs -= S;
          cph ^= 1u;
        }
      }
      return true;
    };
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    using I4 = std::integral_constant<int, 4>;
    using I8 = std::integral_constant<int, 8>;
    using I16 = std::integral_constant<int, 16>;
    bool ok = true;
    switch (op.cfg) {
      case 0: ok = run(I16{}, I4{}, std::false_type{}); break;   // 17..64 superblocks
      case 1: ok = run(I8{}, I2{}, std::true_type{}); break;     // 16 superblocks
      case 2: ok = run(I8{}, I1{}, std::false_type{}); break;    // 1..8 superblocks
      case 3: ok = run(I8{}, I2{}, std::false_type{}); break;    // 9..15 superblocks
      default: ok = run(I16{}, I2{}, std::false_type{}); break;  // (unused)
    }
    if (!ok) {
      // leave no copy in flight into this CTA's shared memory (bounded waits)
      if (lane == 0)
        for (int j = 0; j < S; ++j) mbar_wait(&full[j], 0u, p.err, DEVERR_DRAIN_WAIT, j);
      return;
    }
  }
}

}  // namespace

size_t gemv_chain_smem(int stages, uint32_t slot_bytes, int nsb_max) {
  return chain_layout(stages, slot_bytes, nsb_max).total;
}

}  // namespace epq

using namespace epq;

extern "C" size_t epq_gemv_chain_workspace_bytes(void) { return 256; }

extern "C" epq_status epq_gemv_chain(epq_fmt fmt, const epq_gemv_op *ops, int nops, int nvec, void *ws,
                                     size_t ws_bytes, epq_stream_t stream) {
  if (fmt != EPQ_Q4_K) return EPQ_ERR_FORMAT;
  if (!ops || nops < 1 || nops > EPQ_CHAIN_MAX_OPS || nvec < 1 || nvec > 2) return EPQ_ERR_ARG;
  if (!ws || ws_bytes < epq_gemv_chain_workspace_bytes()) return EPQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return EPQ_ERR_ALIGN;
  DeviceInfo dev;
  if (!current_device(&dev) || dev.major * 10 + dev.minor < 100) return EPQ_ERR_DEVICE;
  unsigned *err = device_error_slot();
  if (!err) return EPQ_ERR_DEVICE;

  ChainParams p;
  p.nops = nops;
  p.nv = nvec;
  p.bar = static_cast<unsigned *>(ws);
  p.err = err;
  const unsigned grid = static_cast<unsigned>(dev.sm_count);
  // ring slot: at least 36 KB, 8 rows of every SwiGLU pair, 4 rows of every
  // other matrix
  int64_t slot = 36864;
  int nsb_max = 1;
  for (int k = 0; k < nops; ++k) {
    const epq_gemv_op &o = ops[k];
    if (!o.blocks || !o.x || !o.y) return EPQ_ERR_ARG;
    if (o.rows < 1 || o.rows > (int64_t(1) << 30) || o.cols < 256 || o.cols > 16384 || o.cols % 256)
      return EPQ_ERR_SHAPE;
    if (o.swiglu && (o.rows % 2)) return EPQ_ERR_SHAPE;
    const int xg = o.x_group > 1 ? o.x_group : 1;
    if (xg > 1 && (o.x_head_dim <= 0 || o.x_head_dim % 32 || o.cols % (o.x_head_dim * xg))) return EPQ_ERR_SHAPE;
    if (!aligned16(o.blocks) || !aligned16(o.x) || !aligned16(o.y) || (o.residual && !aligned16(o.residual)))
      return EPQ_ERR_ALIGN;
    if (o.rms_prenorm && !(o.rms_eps >= 0.0f)) return EPQ_ERR_ARG;
    if (o.x_ld < 0 || o.x_ld > (int64_t(1) << 30) || (o.x_ld && (o.x_ld % 4 || o.x_ld < o.cols / xg)))
      return EPQ_ERR_ARG;
    slot = std::max<int64_t>(slot, (o.swiglu ? 16 : 4) * epq_row_bytes(fmt, o.cols));
    // sums of x: one copy per warp group (two groups below 17 superblocks)
    nsb_max = std::max(nsb_max, static_cast<int>(o.cols / 256) * (o.cols / 256 > 16 ? 1 : 2));
  }
  slot = (slot + 15) & ~int64_t(15);
  // partial sums of every slot fit each warp's area: stages * 3 blocks * 32 floats
  int stages = static_cast<int>(kWarpArea / (kMaxNbs * 32 * 4));
  while (stages >= 2 && gemv_chain_smem(stages, static_cast<uint32_t>(slot), nsb_max) >
                            static_cast<size_t>(dev.max_smem_optin))
    --stages;
  if (stages < 2) return EPQ_ERR_SHAPE;
  p.stages = stages;
  p.slot_bytes = static_cast<uint32_t>(slot);
  p.nsb_max = nsb_max;
  int h = 0;
  for (int k = 0; k < nops; ++k) {
    const epq_gemv_op &o = ops[k];
    ChainOp &c = p.ops[k];
    const int64_t rb = epq_row_bytes(fmt, o.cols);
    const int64_t rows_out = o.swiglu ? o.rows / 2 : o.rows;
    const int64_t block = 8 * rb * (o.swiglu ? 2 : 1);
    const int xg = o.x_group > 1 ? o.x_group : 1;
    c.W = static_cast<const uint8_t *>(o.blocks);
    c.x = o.x;
    c.y = o.y;
    c.residual = o.residual;
    c.rows_out = static_cast<int>(rows_out);
    c.up_rows = o.swiglu ? static_cast<int>(rows_out) : 0;
    c.row_bytes = static_cast<int>(rb);
    c.x_stride = static_cast<int>(o.x_ld ? o.x_ld : o.cols / xg);
    c.y_stride = static_cast<int>(rows_out);
    c.cols = static_cast<int>(o.cols);
    c.nsb = static_cast<int>(o.cols / 256);
    const int64_t rows_cta = (rows_out + grid - 1) / grid;
    c.rq = static_cast<int>(rows_out / grid);
    c.rr = static_cast<int>(rows_out % grid);
    c.cfg = c.nsb > 16 ? 0 : (c.nsb == 16 ? 1 : (c.nsb <= 8 ? 2 : 3));
    c.half = block > slot ? 1 : 0;  // only rows of > 16 superblocks (cfg 0, one group)
    c.nbs = c.half ? 1 : static_cast<int>(std::min<int64_t>(kMaxNbs, slot / block));
    c.nst = c.half ? static_cast<int>(2 * ((rows_cta + 7) / 8))
                   : static_cast<int>(((rows_cta + 7) / 8 + c.nbs - 1) / c.nbs);
    c.stage0 = h;
    h += c.nst;
    c.swiglu = o.swiglu ? 1 : 0;
    c.rms = o.rms_prenorm;
    c.rms_eps = o.rms_eps;
    c.x_group = xg;
    c.x_head_dim = o.x_head_dim;
  }
  const size_t smem = gemv_chain_smem(stages, p.slot_bytes, nsb_max);
  cudaError_t e = cudaFuncSetAttribute(gemv_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_chain_kernel, p);
  if (e != cudaSuccess) return cuda_fail(e);
  return EPQ_OK;
}

// Tensor-core dequant-GEMV for Q4_K weights (epq_gemv / epq_gemv_ex, one or
// two vectors per weight pass).
//
// [H] "速度上限：带宽 ÷ 权重字节数": batch-1 decode streams every packed weight
// once per token, so the kernel is an HBM stream.  [H] "GGUF 的量化格式" fixes
// the Q4_K superblock: 256 weights, fp16 d and dmin, eight 6-bit scale codes
// c_s and eight 6-bit min codes k_s, 4-bit codes n; w = d*c_s*n - dmin*k_s.
//
// Why tensor cores for a matrix-vector product.  On this SM the logic pipe
// (LOP3/SHF/SEL) issues 16 lanes per clock per sub-partition, half the rate
// of the FP32 pipe.  Turning each nibble into an fp32 operand costs one
// logic op per weight, which caps a CUDA-core kernel near half of HBM speed.
// Here one AND isolates two nibbles as two fp16 subnormals (the bit pattern
// n read as fp16 is n * 2^-24, exact and linear), one packed fp16 multiply by
// the sub-block scale code gives c*n*2^-14 (exact: c*n <= 945, a normal
// number), and mma.sync does the products and the float32 sums.  x is split
// into fp16 hi + lo parts (both pre-scaled by a power of two), so the
// products keep ~22 bits of x and the result stays within ~1e-6 of the
// float64 value, far inside the 1e-4 bound.
//
// MMA layout (m16n8k16, A row-major, B column-major):
//   * the 16 "rows" of A are 8 weight rows x two halves of the k-slots, so
//     one MMA consumes 8 rows x 32 weights and every C entry a lane holds
//     is useful;
//   * the 8 columns of B are (half h, vector v, hi/lo): x of vector v at the
//     positions of half h, split into its fp16 hi and lo parts;
//   * lane (g, t) of a warp owns weight row g and sub-blocks 2t, 2t+1 of each
//     superblock: its 32-bit code word j gives the four A registers of MMA j
//     (positions {0,4} {1,5} {2,6} {3,7} of the word's eight nibbles).
// Per superblock the C entries are scaled by d and added to a float32
// accumulator; the min term dmin * sum_s k_s * sum(x over sub-block s) is
// formed from per-sub-block sums of x computed once per CTA.  Every
// superblock of x gets its own power-of-two scale (its largest entry maps to
// just below 2^15), so the fp16 parts keep their precision wherever x is
// large relative to its neighbours.
//
// CTA organisation (persistent, one CTA per SM, 16 warps, no producer warp):
//   * CTA b owns output rows [b*R/G, (b+1)*R/G); a stage holds nbs blocks of
//     8 whole rows (gate and up rows with SwiGLU), moved by one bulk copy
//     (two with SwiGLU) into a ring of shared-memory stages;
//   * the warps form NB = 16/KP groups of KP warps; stage i belongs to group
//     i % NB (the ring depth is a multiple of NB, so a ring slot always serves
//     the same group); warp kq of a group handles superblocks kq, kq + KP, ...
//     of every row block of its stages, and the x operands of those
//     superblocks stay in its registers for the whole kernel.  Each warp
//     converts its own x operands (one global round trip, no CTA barrier);
//   * each warp leaves its partial row sums of a stage in shared memory and
//     bumps the stage's acq_rel counter; the warp that arrives last adds the
//     KP partials in k-part order (deterministic), writes the outputs and
//     issues the bulk copy that refills the slot.  Nobody waits for a free
//     slot and there is no producer warp, so every thread may use 128
//     registers (a 17th warp would cap them at 96).
#include <algorithm>

#include "gemv_tc.cuh"
#include "gemv_tc_core.cuh"

namespace epq {
namespace {

using namespace tc;

constexpr int kTcWarps = 16;
constexpr int kTcThreads = kTcWarps * 32;

struct TcParams {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows_out;
  int64_t up_rows;     // swiglu: row distance gate -> up
  int64_t row_bytes;
  int cols, nsb;       // weights per row, superblocks per row
  int nbs;             // 8-row blocks per stage
  int stages;          // ring depth (a multiple of NB)
  uint32_t stage_bytes;
  int nv;              // vectors in this launch (1 or 2)
  int64_t x_stride, y_stride;
  int rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early_weights;  // stages issued before the grid-dependency wait
  unsigned *err;
};

struct TcLayout {
  uint32_t full, cnt, red, xs, scratch, frag, total;
  int held;  // ring slots whose memory holds the x fragments during the prologue
};

__host__ __device__ inline uint32_t al16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline TcLayout tc_layout(int stages, uint32_t stage_bytes, int nbs, int kp, bool swiglu,
                                              int nsb) {
  TcLayout L;
  const int ngroups = 16 / kp;
  uint32_t o = al16(static_cast<uint32_t>(stages) * stage_bytes);
  L.full = o;
  o += 8u * stages;
  L.cnt = o;  // per ring slot: warps done with it (monotonic); then the staging counter
  o = al16(o + 4u * (stages + 1));
  L.red = o;  // [slot][block nbs][k-part][row 8][vector 2][gate/up]
  o = al16(o + 4u * stages * nbs * kp * 16 * (swiglu ? 2 : 1));
  L.xs = o;  // [group][superblock][t 4][vector 2][sub-block pair 2]: sums of x
  o = al16(o + 4u * ngroups * nsb * 16);
  L.scratch = o;  // [warp][vector 2]: sums of squares over the warp's superblocks
  o = al16(o + 4u * 2 * 16);
  // per-warp staging of one superblock's x operands in consumer lane order,
  // [warp][j 8][lane 32][2]; it lives in the last ring slots while they are
  // not yet filled (small rings get a separate area)
  const uint32_t fb = 16u * kFragWarpBytes;
  const int held = static_cast<int>((fb + stage_bytes - 1) / stage_bytes);
  if (held < stages) {
    L.held = held;
    L.frag = static_cast<uint32_t>(stages - held) * stage_bytes;
  } else {
    L.held = 0;
    L.frag = o;
    o += fb;
  }
  L.total = al16(o);
  return L;
}

template <int KP, int NSB, bool FULL, bool SWIGLU>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_q4k_tc_kernel(const TcParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int M = SWIGLU ? 2 : 1;
  constexpr int NB = kTcWarps / KP;
  const TcLayout L = tc_layout(p.stages, p.stage_bytes, p.nbs, KP, SWIGLU, p.nsb);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
  unsigned *cnt = reinterpret_cast<unsigned *>(smem + L.cnt);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *xsum = reinterpret_cast<float *>(smem + L.xs);
  float *scratch = reinterpret_cast<float *>(smem + L.scratch);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * p.rows_out) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * p.rows_out) / gridDim.x;
  const int nblocks = static_cast<int>((re - rb + 7) / 8);
  const int T = 8 * p.nbs;  // rows per stage
  const int nst = (nblocks + p.nbs - 1) / p.nbs;

  // stage i: rows [rb + i*T, ...) of the gate matrix (and of the up matrix)
  auto issue = [&](int i) {
    const int s = i % p.stages;
    const int64_t r0 = rb + static_cast<int64_t>(i) * T;
    const int64_t nr = min(static_cast<int64_t>(T), re - r0);
    const uint32_t bytes = static_cast<uint32_t>(nr * p.row_bytes);
    uint8_t *dst = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    mbar_arrive_expect_tx(&full[s], SWIGLU ? 2 * bytes : bytes);
    bulk_g2s(dst, p.W + r0 * p.row_bytes, bytes, &full[s]);
    if (SWIGLU)
      bulk_g2s(dst + static_cast<uint32_t>(T * p.row_bytes), p.W + (p.up_rows + r0) * p.row_bytes, bytes,
               &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      cnt[s] = 0u;
    }
    cnt[p.stages] = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  // Weights may stream before the grid-dependency wait, but few stages (four
  // by default, p.early_weights): the x loads issued after the wait would
  // otherwise queue behind this SM's whole ring of weight copies (~200 KB,
  // several microseconds).  The other stages are issued once every warp has
  // issued its x loads.
  const int npre = min(p.early_weights, min(p.stages - L.held, nst));
  if (tid == 0)
    for (int i = 0; i < npre; ++i) issue(i);

  // ------------------------------------------------------------------ prologue
  // Each warp converts the x operands of its own superblocks: lane l loads
  // columns 8l .. 8l+7 of the superblock (one code word's positions) for
  // both vectors (all loads issued before any use: one global round trip),
  // the warp finds the superblock's max |x| (its scale), the sums of x over
  // each 32-column sub-block and of x^2, writes the fp16 hi/lo operands to
  // its staging area in consumer lane order and reads back its registers.
  pdl_wait();  // x and the residual are produced upstream
  const XGather xg{p.x_group, p.x_head_dim};
  const int g = lane >> 2, t = lane & 3;
  const int kq = warp % KP, grp = warp / KP;
  const int cv = t & 1;  // vector of this lane's C entries
  float *gxsum = xsum + grp * p.nsb * 16;
  uint32_t bq[NSB][8][2];
  float fsc[NSB];
  {
    uint2 *frag = reinterpret_cast<uint2 *>(smem + L.frag) + warp * (kFragWarpBytes / 8);
    const int sub = lane >> 2, wi = lane & 3;          // sub-block and word of this lane's columns
    const int tp = sub >> 1, jj = 4 * (sub & 1) + wi;   // consumer lane group t' and MMA index j
    // every load of a vector is issued before any is used (one round trip);
    // superblocks past the row end read the last one and are zeroed later
    float4 xr[NSB][2][2];
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      if (v < p.nv) {
        const float *xv = p.x + v * p.x_stride;
#pragma unroll
        for (int i = 0; i < NSB; ++i) {
          const int sb = FULL ? kq + i * KP : min(kq + i * KP, p.nsb - 1);
          const float *src = xv + xg.src(256 * sb + 8 * lane);
          xr[i][v][0] = ldg4(src);
          xr[i][v][1] = ldg4(src + 4);
        }
      } else {
#pragma unroll
        for (int i = 0; i < NSB; ++i) xr[i][v][0] = xr[i][v][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // the x loads are in flight: now the rest of the initial weight copies
    named_sync(2, kTcThreads);  // prologue only: no warp has left yet
    if (tid == 0)
      for (int i = npre; i < min(p.stages - L.held, nst); ++i) issue(i);
    if (!FULL) {
#pragma unroll
      for (int i = 0; i < NSB; ++i)
        if (kq + i * KP >= p.nsb)
          xr[i][0][0] = xr[i][0][1] = xr[i][1][0] = xr[i][1][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ssq[2] = {0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < NSB; ++i) {
      const int sb = kq + i * KP;
      float fs[2] = {0.0f, 0.0f};
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        if (v >= p.nv) {  // no such vector: zero operands, nothing to convert
          if (wi == 0 && (FULL || sb < p.nsb)) gxsum[((sb * 4 + tp) * 2 + v) * 2 + (sub & 1)] = 0.0f;
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
        if (wi == 0 && (FULL || sb < p.nsb)) gxsum[((sb * 4 + tp) * 2 + v) * 2 + (sub & 1)] = s8;
        // |x| < 2^E: x * 2^(15 - E) stays below 2^15; the A operands carry
        // 2^-14, so the code sums come back with 2^(14 - sig)
        const int sig = min(126, max(-112, 15 - bound_exponent(amax)));
        fs[v] = exp2i(14 - sig);
        const float up = exp2i(sig);
        float q[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = q0[e] * up;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // consumer lane (g', t') with g' = 4h + 2v + hilo holds positions
          // {h, h+4} (register 0) and {h+2, h+6} (register 1) of this word
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
        bq[i][j][0] = r.x;
        bq[i][j][1] = r.y;
      }
      fsc[i] = cv ? fs[1] : fs[0];
      __syncwarp();
    }
    const float s0 = warp_sum_xor<32>(ssq[0]), s1 = warp_sum_xor<32>(ssq[1]);
    if (lane == 0) {
      scratch[warp * 2] = s0;
      scratch[warp * 2 + 1] = s1;
    }
    __syncwarp();
  }
  // the ring slots that held the staging areas can be filled once every warp
  // is done with them
  if (L.held > 0 && p.stages - L.held < nst) {
    if (lane == 0) atom_add_acq_rel(&cnt[p.stages], 1u);  // staging-free counter
    if (tid == 0) {
      // bounded wait for all warps (each arrives right after its own prologue)
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_shared(&cnt[p.stages]) < static_cast<unsigned>(kTcWarps)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          record_error(p.err, DEVERR_RED_WAIT, 0);
          break;
        }
      }
      fence_proxy_async();  // the staging reads and writes precede the copies into it
      for (int i = p.stages - L.held; i < min(p.stages, nst); ++i) issue(i);
    }
  }
  // byte permutes of the scale / min code pairs of sub-blocks 2t, 2t+1
  const uint32_t csel = t == 0 ? 0x10u : (t == 1 ? 0x21u : (t == 2 ? 0x43u : 0x54u));
  const uint32_t ksel = t == 0 ? 0x32u : (t == 1 ? 0x43u : (t == 2 ? 0x65u : 0x76u));
  const int nsh = (t & 1) * 4;
  uint32_t magic = kH1024;
  asm volatile("" : "+r"(magic));  // keep the constant in a register
  const uint32_t rbytes = static_cast<uint32_t>(p.row_bytes);

  // ------------------------------------------------------------------ main loop
  for (int i = grp; i < nst; i += NB) {
    const int s = i % p.stages;
    if (!warp_wait(&full[s], (i / p.stages) & 1, p.err, DEVERR_FULL_WAIT, i)) {
      // leave no copy of this group in flight into this CTA's shared memory
      if (lane == 0)
        for (int j = i; j < min(nst, i + p.stages); j += NB)
          mbar_wait(&full[j % p.stages], (j / p.stages) & 1, p.err, DEVERR_DRAIN_WAIT, j);
      return;
    }
    const uint8_t *sbase = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    float *rs = red + static_cast<uint32_t>(s * p.nbs * KP * 16 * M);
    const int nbl = min(p.nbs, nblocks - i * p.nbs);  // blocks in this stage
    for (int bi = 0; bi < nbl; ++bi) {
      float pv[2][M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float acc = 0.0f, am0 = 0.0f, am1 = 0.0f;
        const uint8_t *row = sbase + static_cast<uint32_t>(m * T + 8 * bi + g) * rbytes;
        block_dot<KP, NSB, FULL>(row, kq, p.nsb, t, magic, csel, ksel, nsh, bq, fsc, gxsum, acc, am0, am1);
        pv[0][m] = (cv == 0 ? acc : 0.0f) - am0;
        pv[1][m] = (cv == 1 ? acc : 0.0f) - am1;
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          pv[v][m] += __shfl_xor_sync(0xffffffffu, pv[v][m], 1);
          pv[v][m] += __shfl_xor_sync(0xffffffffu, pv[v][m], 2);
        }
        if (t < 2) rs[(((bi * KP + kq) * 8 + g) * 2 + t) * M + m] = t == 0 ? pv[0][m] : pv[1][m];
      }
    }
    __syncwarp();
    unsigned old = 0u;
    if (lane == 0) old = atom_add_acq_rel(&cnt[s], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    __syncwarp();
    if (((old + 1u) & (KP - 1)) == 0u) {
      // last warp of the group on this stage: outputs, then refill the slot.
      // The RMS factor comes from the group's sums of squares (its k-parts
      // cover the row; each was written before its warp's first arrival).
      float osc0 = 1.0f, osc1 = 1.0f;
      if (p.rms) {
        float q0 = 0.0f, q1 = 0.0f;
        for (int w = grp * KP; w < grp * KP + KP; ++w) {
          q0 += scratch[w * 2];
          q1 += scratch[w * 2 + 1];
        }
        osc0 = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q0, static_cast<float>(p.cols)), p.rms_eps)));
        osc1 = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q1, static_cast<float>(p.cols)), p.rms_eps)));
      }
      for (int o = lane; o < nbl * 16; o += 32) {
        const int bi = o >> 4, gg = (o >> 1) & 7, v = o & 1;
        const int64_t row = rb + 8 * (i * p.nbs + bi) + gg;
        if (row < re && v < p.nv) {
          float sg = 0.0f, su = 0.0f;
#pragma unroll
          for (int q = 0; q < KP; ++q) {
            sg += rs[(((bi * KP + q) * 8 + gg) * 2 + v) * M];
            if (SWIGLU) su += rs[(((bi * KP + q) * 8 + gg) * 2 + v) * M + 1];
          }
          const float os = v ? osc1 : osc0;
          float val = sg * os;
          if (SWIGLU) val = silu(val) * (su * os);
          if (p.residual) val += p.residual[v * p.y_stride + row];
          p.y[v * p.y_stride + row] = val;
        }
      }
      __syncwarp();
      if (lane == 0 && i + p.stages < nst) {
        fence_proxy_async();  // this CTA's reads of the slot precede the refill
        issue(i + p.stages);
      }
    }
  }
}

template <int KP, int NSB, bool FULL, bool SW>
cudaError_t launch_tc(const TcParams &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  auto k = gemv_q4k_tc_kernel<KP, NSB, FULL, SW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(kTcThreads), smem, s, p);
}

// (KP, NSB) pairs with a compiled kernel
bool tc_combo(int kp, int nsbw) {
  switch (kp) {
    case 1: case 2: return nsbw == 1;
    case 4: return nsbw == 1 || nsbw == 2 || nsbw == 4;
    case 8: return nsbw == 1 || nsbw == 2;
    case 16: return nsbw == 1 || nsbw == 2 || nsbw == 4;
  }
  return false;
}

}  // namespace

bool gemv_tc_plan(int64_t row_bytes, int cols, int64_t rows_out, bool swiglu, const DeviceInfo &dev,
                  TcPlan *pl) {
  if (cols % 256 || cols < 256 || cols > 16384) return false;
  const int nsb = cols / 256;
  const int64_t g = std::min<int64_t>(dev.sm_count, (rows_out + 7) / 8);
  pl->grid = static_cast<unsigned>(std::max<int64_t>(1, g));
  const int64_t blocks_cta = ((rows_out + pl->grid - 1) / pl->grid + 7) / 8;
  // superblocks per warp and row block: more when a CTA has many blocks (the
  // per-block reduction is then shared by more work), fewer for short CTAs
  // (more warps on each block)
  // (measured on the dense decode step: 8 warps per block for rows of up to
  // 32 superblocks beat 4 and 16; wider rows keep 16)
  const int want = blocks_cta >= 24 ? 4 : (blocks_cta >= 6 ? 2 : 1);
  int kp = 1;
  while (kp < kTcWarps && (nsb + kp - 1) / kp > want) kp *= 2;
  if (nsb <= 32 && nsb >= 8) kp = 8;
  if (tune_tc_split() > 0 && (nsb + tune_tc_split() - 1) / tune_tc_split() <= 4) kp = tune_tc_split();
  int nsbw = (nsb + kp - 1) / kp;
  nsbw = nsbw <= 1 ? 1 : (nsbw <= 2 ? 2 : 4);
  while (!tc_combo(kp, nsbw) && kp < kTcWarps) {
    kp *= 2;
    nsbw = (nsb + kp - 1) / kp;
    nsbw = nsbw <= 1 ? 1 : (nsbw <= 2 ? 2 : 4);
  }
  if (!tc_combo(kp, nsbw)) return false;
  pl->nsb_tmpl = nsbw;
  pl->kp = kp;
  pl->nb = kTcWarps / kp;
  pl->full = nsb == kp * nsbw;
  const int64_t block_bytes = 8 * row_bytes * (swiglu ? 2 : 1);
  // ring: a multiple of the group count deep (<= 16 slots), preferring two
  // blocks per stage only when every group still gets three slots
  auto depth = [&](int nbs) {
    const int64_t stages_cta = (blocks_cta + nbs - 1) / nbs;
    int st = static_cast<int>(std::min<int64_t>(16, std::max<int64_t>(stages_cta, 2)));
    st = std::max(pl->nb, (st + pl->nb - 1) / pl->nb * pl->nb);
    for (; st >= pl->nb; st -= pl->nb) {
      const TcLayout L = tc_layout(st, static_cast<uint32_t>(nbs * block_bytes), nbs, kp, swiglu, nsb);
      if (L.total <= static_cast<uint32_t>(dev.max_smem_optin)) break;
    }
    return st;
  };
  int nbs = (blocks_cta >= 2 && block_bytes < tune_tile_bytes()) ? 2 : 1;
  int st = depth(nbs);
  if (nbs == 2 && st < 3 * pl->nb) {
    nbs = 1;
    st = depth(1);
  }
  if (st < pl->nb || st < 1) return false;
  pl->nbs = nbs;
  pl->stage_bytes = static_cast<uint32_t>(nbs * block_bytes);
  pl->stages = st;
  pl->smem = tc_layout(st, pl->stage_bytes, nbs, kp, swiglu, nsb).total;
  return true;
}

cudaError_t gemv_tc_launch(const TcPlan &pl, const TcArgs &a, cudaStream_t s) {
  TcParams p;
  p.W = a.W;
  p.x = a.x;
  p.y = a.y;
  p.residual = a.residual;
  p.rows_out = a.rows_out;
  p.up_rows = a.swiglu ? a.rows_out : 0;
  p.row_bytes = a.row_bytes;
  p.cols = a.cols;
  p.nsb = a.cols / 256;
  p.nbs = pl.nbs;
  p.stages = pl.stages;
  p.stage_bytes = pl.stage_bytes;
  p.nv = a.nv;
  p.x_stride = a.x_stride;
  p.y_stride = a.y_stride;
  p.rms = a.rms;
  p.rms_eps = a.rms_eps;
  p.x_group = a.x_group;
  p.x_head_dim = a.x_head_dim;
  p.early_weights = a.early_weights ? tune_early_stages() : 0;
  p.err = a.err;
  const bool sw = a.swiglu != 0;
#define EPQ_TC_CASE(KP, NSB)                                                                        \
  if (pl.kp == KP && pl.nsb_tmpl == NSB) {                                                          \
    if (pl.full)                                                                                    \
      return sw ? launch_tc<KP, NSB, true, true>(p, pl.grid, pl.smem, s)                            \
                : launch_tc<KP, NSB, true, false>(p, pl.grid, pl.smem, s);                          \
    return sw ? launch_tc<KP, NSB, false, true>(p, pl.grid, pl.smem, s)                             \
              : launch_tc<KP, NSB, false, false>(p, pl.grid, pl.smem, s);                           \
  }
  EPQ_TC_CASE(1, 1)
  EPQ_TC_CASE(2, 1)
  EPQ_TC_CASE(4, 1)
  EPQ_TC_CASE(4, 2)
  EPQ_TC_CASE(4, 4)
  EPQ_TC_CASE(8, 1)
  EPQ_TC_CASE(8, 2)
  EPQ_TC_CASE(16, 1)
  EPQ_TC_CASE(16, 2)
  EPQ_TC_CASE(16, 4)
#undef EPQ_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace epq

// Tensor-core Q4_K expert kernels of the MoE layer, one or two tokens per
// call.
//
// "Flash-MoE：在笔记本上运行 397B 参数大模型", section "每层流水线": the selected
// experts' gate/up projections with SwiGLU, then the down projections and
// the weighted combine with the residual.  The products use the tensor-core
// Q4_K decode of the dense GEMV (gemv_tc.cu: each nibble pair read as two
// fp16 subnormals and scaled by the sub-block code, x split into fp16 hi +
// lo parts with one power-of-two scale per superblock, m16n8k16 MMAs, d and
// the min term applied per superblock).  The two MMA vectors are the two
// tokens.  What differs from the dense kernel is where rows and x come from:
//   * gate/up (moe_gateup_tc_kernel): every CTA first routes all tokens from
//     the router's logits (route_tokens, as the CUDA-core kernels do), so
//     the expert copies need no grid-wide step.  The virtual rows slot*I + i
//     (the selected experts in ascending order, then the shared expert) are
//     split evenly over the grid.  A stage is 8 virtual rows of gate and the
//     matching 8 up rows, copied in two pieces when the rows cross a slot
//     boundary.  A row of slot s writes h = silu(g r_t) * (u r_t) for each
//     entry (token t, choice k) of the slot, r_t the token's RMS factor.
//   * down (moe_down_tc_kernel): the output rows are split over the grid and
//     a stage holds 8 rows of every slot's down matrix (one copy per slot).
//     The x operand of token t is the concatenation over the slots of
//     coef * h, coef being the routing weight (or the shared gate), and zero
//     where t does not use the slot.  One dot per row and token is then the
//     whole combine: y = x + dot.
// Warp organisation as in gemv_tc.cu: 16 warps in NB = 16/KP groups of KP
// k-parts, stage i belongs to group i % NB, partial sums go through shared
// memory, and the last warp of a group to finish a stage adds them in
// k-part order (deterministic), writes the outputs and refills the slot.
#include <algorithm>

#include "gemv_tc_core.cuh"
#include "moe_tc.cuh"

namespace epq {
namespace {

using namespace tc;

constexpr int kMtWarps = 16;
constexpr int kMtThreads = kMtWarps * 32;

__host__ __device__ inline uint32_t mt_al16(uint32_t v) { return (v + 15u) & ~15u; }

struct MtParams {
  MoeArgs a;
  int stages;
  uint32_t stage_bytes;
  int nsbx;      // superblocks of the x operand (gate/up: H/256; down: max slots * I/256)
  int frag_sep;  // 1: the x staging area has its own space (else the last ring slots)
};

// Shared memory: the ring, its barriers and counters, the partial sums,
// the sub-block sums of x, the routing copy, and the per-warp staging of
// the x operands (in the last ring slots while they are not yet filled).
struct MtLayout {
  uint32_t full, cnt, red, xs, meta, frag, total;
  int held;
};

__host__ __device__ inline MtLayout mt_layout(int stages, uint32_t stage_bytes, int kp, int m, int nsbx, int ntok,
                                              int topk, bool sep) {
  MtLayout L;
  uint32_t o = mt_al16(static_cast<uint32_t>(stages) * stage_bytes);
  L.full = o;
  o += 8u * stages;
  L.cnt = o;  // per slot: warps done with it (monotonic); then the staging counter
  o = mt_al16(o + 4u * (stages + 1));
  L.red = o;  // [slot][k-part][row 8][vector 2][gate/up]
  o = mt_al16(o + 4u * stages * kp * 16 * m);
  L.xs = o;  // [group][superblock][t 4][vector 2][sub-block pair 2]
  o = mt_al16(o + 4u * (kMtWarps / kp) * nsbx * 16);
  L.meta = o;
  o = mt_al16(o + 4u * meta_words(ntok, topk));
  const uint32_t fb = 16u * kFragWarpBytes;
  const int held = static_cast<int>((fb + stage_bytes - 1) / stage_bytes);
  if (!sep && held < stages) {
    L.held = held;
    L.frag = static_cast<uint32_t>(stages - held) * stage_bytes;
  } else {
    L.held = 0;
    L.frag = o;
    o += fb;
  }
  L.total = mt_al16(o);
  return L;
}

// The x operands of this warp's superblocks kq, kq + KP, ... from xr (the
// eight columns 8*lane .. of each superblock for vectors 0 and 1, zeros for
// absent vectors): per superblock and vector a power-of-two scale from the
// superblock's max |x|, the sums of x over each 32-column sub-block (for the
// min term), and the fp16 hi/lo split staged through `frag` into consumer
// lane order.  Superblocks at or past nsb get zero operands.
template <int KP, int NSB, bool FULL>
__device__ __forceinline__ void convert_x(const float4 (&xr)[NSB][2][2], int nv, int kq, int nsb, int lane, int cv,
                                          uint2 *frag, float *gxsum, uint32_t (&bq)[NSB][8][2],
                                          float (&fsc)[NSB]) {
  const int sub = lane >> 2, wi = lane & 3;         // sub-block and word of this lane's columns
  const int tp = sub >> 1, jj = 4 * (sub & 1) + wi;  // consumer lane group t' and MMA index j
#pragma unroll
  for (int i = 0; i < NSB; ++i) {
    const int sb = kq + i * KP;
    if (!FULL && sb >= nsb) {  // warp-uniform: never read by the dot products
#pragma unroll
      for (int j = 0; j < 8; ++j) bq[i][j][0] = bq[i][j][1] = 0u;
      fsc[i] = 0.0f;
      continue;
    }
    float fs[2] = {0.0f, 0.0f};
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      if (v >= nv) {  // no such vector: zero operands
        if (wi == 0) gxsum[((sb * 4 + tp) * 2 + v) * 2 + (sub & 1)] = 0.0f;
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
        s8 += q0[e];
      }
      amax = warp_max_all(amax);
      s8 += __shfl_xor_sync(0xffffffffu, s8, 1);
      s8 += __shfl_xor_sync(0xffffffffu, s8, 2);
      if (wi == 0) gxsum[((sb * 4 + tp) * 2 + v) * 2 + (sub & 1)] = s8;
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
}

// block_dot of gemv_tc_core.cuh with the superblock i of row g at
// row + off[i] (the down stage keeps each slot's rows in its own segment).
template <int KP, int NSB>
__device__ __forceinline__ void block_dot_seg(const uint8_t *row, const uint32_t (&off)[NSB], int kq, int nsb,
                                              int t, uint32_t magic, uint32_t csel, uint32_t ksel, int nsh,
                                              const uint32_t (&bq)[NSB][8][2], const float (&fsc)[NSB],
                                              const float *xsum, float &acc, float &am0, float &am1) {
#pragma unroll
  for (int i = 0; i < NSB; ++i) {
    const int sb = kq + i * KP;
    if (sb >= nsb) break;  // warp-uniform
    const uint8_t *sp = row + off[i];
    const uint4 hd = *reinterpret_cast<const uint4 *>(sp);
    const uint4 qa = *reinterpret_cast<const uint4 *>(sp + 16 + 32 * t);
    const uint4 qb = *reinterpret_cast<const uint4 *>(sp + 32 + 32 * t);
    const float4 X = *reinterpret_cast<const float4 *>(xsum + (sb * 4 + t) * 4);
    const uint32_t cc = __byte_perm(hd.y, hd.z, csel) >> nsh;
    const uint32_t kk = __byte_perm(hd.z, hd.w, ksel) >> nsh;
    const SubMul ma = sub_mul(cc & 63u, magic), mb = sub_mul((cc >> 6) & 63u, magic);
    float Ca[4] = {0.f, 0.f, 0.f, 0.f}, Cb[4] = {0.f, 0.f, 0.f, 0.f};
    mma_word(qa.x, ma, bq[i][0][0], bq[i][0][1], Ca);
    mma_word(qa.y, ma, bq[i][1][0], bq[i][1][1], Cb);
    mma_word(qa.z, ma, bq[i][2][0], bq[i][2][1], Ca);
    mma_word(qa.w, ma, bq[i][3][0], bq[i][3][1], Cb);
    mma_word(qb.x, mb, bq[i][4][0], bq[i][4][1], Ca);
    mma_word(qb.y, mb, bq[i][5][0], bq[i][5][1], Cb);
    mma_word(qb.z, mb, bq[i][6][0], bq[i][6][1], Ca);
    mma_word(qb.w, mb, bq[i][7][0], bq[i][7][1], Cb);
    const float s = t < 2 ? (Ca[0] + Cb[0]) + (Ca[1] + Cb[1]) : (Ca[2] + Cb[2]) + (Ca[3] + Cb[3]);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hd.x));  // d, dmin
    acc = fmaf(dd.x, s * fsc[i], acc);
    const float ka = u6_to_float(kk & 63u), kb = u6_to_float((kk >> 6) & 63u);
    am0 = fmaf(dd.y, fmaf(ka, X.x, kb * X.y), am0);
    am1 = fmaf(dd.y, fmaf(ka, X.z, kb * X.w), am1);
  }
}

// Entry k of token v in slot sl (the choice index, topk for the shared
// expert), or -1 when v does not use the slot.
__device__ __forceinline__ int slot_entry(const Meta &m, int ntok, int sl, int v) {
  int k = -1;
  const int n = m.cnt[sl];
  for (int j = 0; j < n; ++j) {
    const int ent = m.list[sl * ntok + j];
    if ((ent >> 5) == v) k = ent & 31;
  }
  return k;
}

// Staging-area release shared by both kernels: every warp arrives after its
// conversion; thread 0 waits (bounded) for all of them, then fills the ring
// slots that held the staging areas.
template <typename Issue>
__device__ __forceinline__ void release_held(const MtLayout &L, int stages, int nst, unsigned *cnt, int lane,
                                             int tid, unsigned *err, Issue &&issue) {
  if (L.held > 0 && stages - L.held < nst) {
    if (lane == 0) atom_add_acq_rel(&cnt[stages], 1u);
    if (tid == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_shared(&cnt[stages]) < static_cast<unsigned>(kMtWarps)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          record_error(err, DEVERR_RED_WAIT, 0);
          break;
        }
      }
      fence_proxy_async();  // the staging reads and writes precede the copies into it
      for (int i = stages - L.held; i < min(stages, nst); ++i) issue(i);
    }
  }
}

// ------------------------------------------------------------------ gate/up + SwiGLU
template <int KP, int NSB, bool FULL>
__global__ void __launch_bounds__(kMtThreads, 1) moe_gateup_tc_kernel(const MtParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NB = kMtWarps / KP;
  const MoeArgs &a = p.a;
  const MtLayout L = mt_layout(p.stages, p.stage_bytes, KP, 2, p.nsbx, a.ntok, a.topk, p.frag_sep);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
  unsigned *cnt = reinterpret_cast<unsigned *>(smem + L.cnt);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *xsum = reinterpret_cast<float *>(smem + L.xs);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nsb = p.nsbx, I = a.I;
  const uint32_t rbytes = static_cast<uint32_t>(a.gu_row_bytes);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      cnt[s] = 0u;
    }
    cnt[p.stages] = 0u;
    fence_mbar_init();
  }
  Meta m(smem + L.meta, a.ntok, a.topk);
  m.clear(tid, blockDim.x);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // logits and x statistics come from the router kernel, x from upstream

  const int g = lane >> 2, t = lane & 3, cv = t & 1;
  const int kq = warp % KP, grp = warp / KP;
  // x of this warp's superblocks, in flight while the CTA routes
  float4 xr[NSB][2][2];
#pragma unroll
  for (int v = 0; v < 2; ++v) {
#pragma unroll
    for (int i = 0; i < NSB; ++i) {
      if (v < a.ntok) {
        const int sb = FULL ? kq + i * KP : min(kq + i * KP, nsb - 1);
        const float *src = a.x + static_cast<int64_t>(v) * a.H + 256 * sb + 8 * lane;
        xr[i][v][0] = ldg4(src);
        xr[i][v][1] = ldg4(src + 4);
      } else {
        xr[i][v][0] = xr[i][v][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  // routing scratch: the start of the ring (no copy is issued before the
  // experts are known); route_tokens ends with a CTA barrier
  route_tokens(a, m, reinterpret_cast<uint32_t *>(smem), blockIdx.x == 0);

  const int nslots = *m.nslots, nact = *m.nact;
  const int64_t total = static_cast<int64_t>(nslots) * I;
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * total) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * total) / gridDim.x;
  const int nst = static_cast<int>((re - rb + 7) / 8);
  // stage i: virtual rows [rb + 8i, +8) of gate, then the same rows of up
  auto issue = [&](int i) {
    const int s = i % p.stages;
    const int64_t r0 = rb + 8ll * i;
    const int nr = static_cast<int>(min(static_cast<int64_t>(8), re - r0));
    uint8_t *dst = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    mbar_arrive_expect_tx(&full[s], 2u * static_cast<uint32_t>(nr) * rbytes);
    for (int d = 0; d < nr;) {  // one piece per slot the rows touch (two at most: I >= 256)
      const int64_t r = r0 + d;
      const int sl = static_cast<int>(r / I);
      const int ii = static_cast<int>(r - static_cast<int64_t>(sl) * I);
      const int n = min(nr - d, I - ii);
      const int e = sl < nact ? m.active[sl] : -1;
      const uint8_t *base = e >= 0 ? a.gate_up + static_cast<int64_t>(e) * a.gu_stride : a.sh_gate_up;
      const uint32_t bytes = static_cast<uint32_t>(n) * rbytes;
      bulk_g2s(dst + static_cast<uint32_t>(d) * rbytes, base + static_cast<int64_t>(ii) * rbytes, bytes, &full[s]);
      bulk_g2s(dst + static_cast<uint32_t>(8 + d) * rbytes, base + static_cast<int64_t>(I + ii) * rbytes, bytes,
               &full[s]);
      d += n;
    }
  };
  // The first stage's copies go out at once; the other free slots are
  // filled by warps 1, 2, ... right after their own x conversion: issuing
  // ~100 KB of copies stalls the issuing thread for microseconds while
  // every SM's requests drain, and one thread issuing them all delayed its
  // warp's conversion, which the staging release below waits for.
  const int first_n = min(p.stages - L.held, nst);
  if (tid == 0 && first_n > 0) {
    fence_proxy_async();  // the routing scratch writes precede the copies into the ring
    issue(0);
  }

  float *gxsum = xsum + grp * nsb * 16;
  uint32_t bq[NSB][8][2];
  float fsc[NSB];
  {
    uint2 *frag = reinterpret_cast<uint2 *>(smem + L.frag) + warp * (kFragWarpBytes / 8);
    if (!FULL) {
#pragma unroll
      for (int i = 0; i < NSB; ++i)
        if (kq + i * KP >= nsb) xr[i][0][0] = xr[i][0][1] = xr[i][1][0] = xr[i][1][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    convert_x<KP, NSB, FULL>(xr, a.ntok, kq, nsb, lane, cv, frag, gxsum, bq, fsc);
  }
  if (lane == 0) {
    bool fenced = false;
    for (int i = warp == 0 ? kMtWarps : warp; i < first_n; i += kMtWarps) {
      if (!fenced) fence_proxy_async();
      fenced = true;
      issue(i);
    }
  }
  release_held(L, p.stages, nst, cnt, lane, tid, a.err, issue);

  const uint32_t csel = t == 0 ? 0x10u : (t == 1 ? 0x21u : (t == 2 ? 0x43u : 0x54u));
  const uint32_t ksel = t == 0 ? 0x32u : (t == 1 ? 0x43u : (t == 2 ? 0x65u : 0x76u));
  const int nsh = (t & 1) * 4;
  uint32_t magic = kH1024;
  asm volatile("" : "+r"(magic));

  for (int i = grp; i < nst; i += NB) {
    const int s = i % p.stages;
    if (!warp_wait(&full[s], (i / p.stages) & 1, a.err, DEVERR_FULL_WAIT, i)) {
      // leave no copy of this group in flight into this CTA's shared memory
      if (lane == 0)
        for (int j = i; j < min(nst, i + p.stages); j += NB)
          mbar_wait(&full[j % p.stages], (j / p.stages) & 1, a.err, DEVERR_DRAIN_WAIT, j);
      return;
    }
    const uint8_t *sbase = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    float *rs = red + s * KP * 16 * 2;
    float pv[2][2];
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      float acc = 0.0f, am0 = 0.0f, am1 = 0.0f;
      const uint8_t *row = sbase + static_cast<uint32_t>(mm * 8 + g) * rbytes;
      block_dot<KP, NSB, FULL>(row, kq, nsb, t, magic, csel, ksel, nsh, bq, fsc, gxsum, acc, am0, am1);
      pv[0][mm] = (cv == 0 ? acc : 0.0f) - am0;
      pv[1][mm] = (cv == 1 ? acc : 0.0f) - am1;
    }
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        pv[v][mm] += __shfl_xor_sync(0xffffffffu, pv[v][mm], 1);
        pv[v][mm] += __shfl_xor_sync(0xffffffffu, pv[v][mm], 2);
      }
      if (t < 2) rs[((kq * 8 + g) * 2 + t) * 2 + mm] = t == 0 ? pv[0][mm] : pv[1][mm];
    }
    __syncwarp();
    unsigned old = 0u;
    if (lane == 0) old = atom_add_acq_rel(&cnt[s], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    __syncwarp();
    if (((old + 1u) & (KP - 1)) == 0u) {
      // last warp of the group on this stage: h of every entry, then the refill
      if (lane < 16) {
        const int gg = lane >> 1, v = lane & 1;
        const int64_t row = rb + 8ll * i + gg;
        if (row < re && v < a.ntok) {
          float sg = 0.0f, su = 0.0f;
#pragma unroll
          for (int q = 0; q < KP; ++q) {
            sg += rs[((q * 8 + gg) * 2 + v) * 2];
            su += rs[((q * 8 + gg) * 2 + v) * 2 + 1];
          }
          const int sl = static_cast<int>(row / I);
          const int ii = static_cast<int>(row - static_cast<int64_t>(sl) * I);
          const int k = slot_entry(m, a.ntok, sl, v);
          if (k >= 0) {
            const float r = m.rms[v];
            a.h[static_cast<int64_t>(v * (a.topk + 1) + k) * I + ii] = silu(sg * r) * (su * r);
          }
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

// ------------------------------------------------------------------ down + combine
template <int KP, int NSB>
__global__ void __launch_bounds__(kMtThreads, 1) moe_down_tc_kernel(const MtParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NB = kMtWarps / KP;
  const MoeArgs &a = p.a;
  const MtLayout L = mt_layout(p.stages, p.stage_bytes, KP, 1, p.nsbx, a.ntok, a.topk, p.frag_sep);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
  unsigned *cnt = reinterpret_cast<unsigned *>(smem + L.cnt);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *xsum = reinterpret_cast<float *>(smem + L.xs);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int I = a.I, H = a.H, spb = a.I / 256;
  const uint32_t rbytes = static_cast<uint32_t>(a.dn_row_bytes);
  const uint32_t seg = 8u * rbytes;  // one slot's rows in a stage
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * H) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * H) / gridDim.x;
  const int nst = static_cast<int>((re - rb + 7) / 8);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      cnt[s] = 0u;
    }
    cnt[p.stages] = 0u;
    fence_mbar_init();
  }
  Meta m(smem + L.meta, a.ntok, a.topk);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // h and the routing come from the gate/up kernel
  load_meta(a, m, tid, blockDim.x);
  __syncthreads();
  const int nslots = *m.nslots, nact = *m.nact;
  const int nsb = nslots * spb;  // superblocks of the virtual x

  // stage i: rows [rb + 8i, +8) of every slot's down matrix, slot-major
  auto issue = [&](int i) {
    const int s = i % p.stages;
    const int64_t r0 = rb + 8ll * i;
    const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(8), re - r0)) * rbytes;
    uint8_t *dst = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    mbar_arrive_expect_tx(&full[s], bytes * static_cast<uint32_t>(nslots));
    for (int sl = 0; sl < nslots; ++sl) {
      const int e = sl < nact ? m.active[sl] : -1;
      const uint8_t *base = e >= 0 ? a.down + static_cast<int64_t>(e) * a.dn_stride : a.sh_down;
      bulk_g2s(dst + static_cast<uint32_t>(sl) * seg, base + r0 * rbytes, bytes, &full[s]);
    }
  };
  // first stage now, the other free slots by warps 1, 2, ... after their
  // conversion (as in the gate/up kernel)
  const int first_n = min(p.stages - L.held, nst);
  if (tid == 0 && first_n > 0) issue(0);

  const int g = lane >> 2, t = lane & 3, cv = t & 1;
  const int kq = warp % KP, grp = warp / KP;
  // x operand: superblock sb of token v is coef * h[v, k] over columns
  // 256 (sb mod spb) .. of the entry (v, k) that slot sb / spb serves
  float4 xr[NSB][2][2];
  float coef[NSB][2];
  uint32_t off[NSB];
#pragma unroll
  for (int i = 0; i < NSB; ++i) {
    const int sb = kq + i * KP;
    const int sl = sb / spb, sbl = sb - sl * spb;
    off[i] = static_cast<uint32_t>(sl) * seg + static_cast<uint32_t>(sbl) * 144u;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      xr[i][v][0] = xr[i][v][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      coef[i][v] = 0.0f;
      if (sb < nsb && v < a.ntok) {
        const int k = slot_entry(m, a.ntok, sl, v);
        if (k >= 0) {
          const float *src = a.h + static_cast<int64_t>(v * (a.topk + 1) + k) * I + 256 * sbl + 8 * lane;
          xr[i][v][0] = ldg4(src);
          xr[i][v][1] = ldg4(src + 4);
          coef[i][v] = k < a.topk ? m.w[v * a.topk + k] : m.gs[v];
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NSB; ++i)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const float c = coef[i][v];
      xr[i][v][0] = make_float4(xr[i][v][0].x * c, xr[i][v][0].y * c, xr[i][v][0].z * c, xr[i][v][0].w * c);
      xr[i][v][1] = make_float4(xr[i][v][1].x * c, xr[i][v][1].y * c, xr[i][v][1].z * c, xr[i][v][1].w * c);
    }
  float *gxsum = xsum + grp * p.nsbx * 16;
  uint32_t bq[NSB][8][2];
  float fsc[NSB];
  {
    uint2 *frag = reinterpret_cast<uint2 *>(smem + L.frag) + warp * (kFragWarpBytes / 8);
    convert_x<KP, NSB, false>(xr, a.ntok, kq, nsb, lane, cv, frag, gxsum, bq, fsc);
  }
  if (lane == 0)
    for (int i = warp == 0 ? kMtWarps : warp; i < first_n; i += kMtWarps) issue(i);
  release_held(L, p.stages, nst, cnt, lane, tid, a.err, issue);

  const uint32_t csel = t == 0 ? 0x10u : (t == 1 ? 0x21u : (t == 2 ? 0x43u : 0x54u));
  const uint32_t ksel = t == 0 ? 0x32u : (t == 1 ? 0x43u : (t == 2 ? 0x65u : 0x76u));
  const int nsh = (t & 1) * 4;
  uint32_t magic = kH1024;
  asm volatile("" : "+r"(magic));

  for (int i = grp; i < nst; i += NB) {
    const int s = i % p.stages;
    if (!warp_wait(&full[s], (i / p.stages) & 1, a.err, DEVERR_FULL_WAIT, i)) {
      if (lane == 0)
        for (int j = i; j < min(nst, i + p.stages); j += NB)
          mbar_wait(&full[j % p.stages], (j / p.stages) & 1, a.err, DEVERR_DRAIN_WAIT, j);
      return;
    }
    const uint8_t *sbase = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    float *rs = red + s * KP * 16;
    float acc = 0.0f, am0 = 0.0f, am1 = 0.0f;
    block_dot_seg<KP, NSB>(sbase + static_cast<uint32_t>(g) * rbytes, off, kq, nsb, t, magic, csel, ksel, nsh, bq,
                           fsc, gxsum, acc, am0, am1);
    float p0 = (cv == 0 ? acc : 0.0f) - am0;
    float p1 = (cv == 1 ? acc : 0.0f) - am1;
    p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
    p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
    if (t < 2) rs[(kq * 8 + g) * 2 + t] = t == 0 ? p0 : p1;
    __syncwarp();
    unsigned old = 0u;
    if (lane == 0) old = atom_add_acq_rel(&cnt[s], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    __syncwarp();
    if (((old + 1u) & (KP - 1)) == 0u) {
      // last warp of the group on this stage: y = x + the combined dot
      if (lane < 16) {
        const int gg = lane >> 1, v = lane & 1;
        const int64_t row = rb + 8ll * i + gg;
        if (row < re && v < a.ntok) {
          float sum = 0.0f;
#pragma unroll
          for (int q = 0; q < KP; ++q) sum += rs[(q * 8 + gg) * 2 + v];
          const int64_t o = static_cast<int64_t>(v) * H + row;
          a.y[o] = a.x[o] + sum;
        }
      }
      __syncwarp();
      if (lane == 0 && i + p.stages < nst) {
        fence_proxy_async();
        issue(i + p.stages);
      }
    }
  }
}

template <typename K>
cudaError_t mt_launch(K kernel, const MtParams &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(grid), dim3(kMtThreads), smem, s, p);
}

// k-parts and superblocks per warp for an operand of n superblocks: one
// superblock per warp up to 16, then 2 or 4 per warp (0: too wide)
void mt_split(int n, int *kp, int *nsbw) {
  int k = 1;
  while (k < kMtWarps && k < n) k *= 2;
  const int w = (n + k - 1) / k;
  *kp = k;
  *nsbw = w <= 1 ? 1 : (w <= 2 ? 2 : (w <= 4 ? 4 : 0));
}

// Deepest ring (a multiple of the group count, <= 16, at least min_stages)
// that fits shared memory, 0 when none does; *sep: whether the x staging
// area gets its own space at that depth (preferred: with it in the ring, the
// slots it occupies are filled only after every warp's conversion).
int mt_depth(int want, int min_stages, uint32_t stage_bytes, int kp, int m, int nsbx, int ntok, int topk,
             const DeviceInfo &dev, int *sep) {
  const int nb = kMtWarps / kp;
  int st = std::max(std::max(want, min_stages), 2);
  st = std::min(16, (st + nb - 1) / nb * nb);
  st = std::max(st, nb);
  const uint32_t cap = static_cast<uint32_t>(dev.max_smem_optin);
  for (; st >= nb; st -= nb) {
    if (st < min_stages) return 0;
    for (int sp = 1; sp >= 0; --sp) {
      if (mt_layout(st, stage_bytes, kp, m, nsbx, ntok, topk, sp != 0).total <= cap) {
        *sep = sp;
        return st;
      }
    }
  }
  return 0;
}

}  // namespace

bool moe_tc_plan(const MoeArgs &a, int max_slots, const DeviceInfo &dev, MoeTcPlan *pl) {
  if (a.ntok < 1 || a.ntok > 2 || a.H % 256 || a.I % 256 || a.H > 16384 || a.I > 16384) return false;
  pl->grid = static_cast<unsigned>(dev.sm_count);
  const int64_t grid = dev.sm_count;
  // gate/up
  mt_split(a.H / 256, &pl->g_kp, &pl->g_nsbw);
  if (!pl->g_nsbw) return false;
  pl->g_full = a.H / 256 == pl->g_kp * pl->g_nsbw;
  pl->g_stage_bytes = static_cast<uint32_t>(16 * a.gu_row_bytes);
  const int64_t g_rows = (static_cast<int64_t>(max_slots) * a.I + grid - 1) / grid;
  // the routing scratch lives in the ring
  const int g_min = static_cast<int>((4u * kSelScratchWords + pl->g_stage_bytes - 1) / pl->g_stage_bytes);
  pl->g_stages = mt_depth(static_cast<int>((g_rows + 7) / 8), g_min, pl->g_stage_bytes, pl->g_kp, 2, a.H / 256,
                          a.ntok, a.topk, dev, &pl->g_sep);
  if (!pl->g_stages) return false;
  pl->g_smem = mt_layout(pl->g_stages, pl->g_stage_bytes, pl->g_kp, 2, a.H / 256, a.ntok, a.topk, pl->g_sep).total;
  // down
  pl->d_nsbx = max_slots * (a.I / 256);
  mt_split(pl->d_nsbx, &pl->d_kp, &pl->d_nsbw);
  if (!pl->d_nsbw) return false;
  pl->d_stage_bytes = static_cast<uint32_t>(max_slots * 8 * a.dn_row_bytes);
  if (static_cast<int64_t>(pl->d_stage_bytes) >= (1 << 20)) return false;  // one barrier's transaction count
  const int64_t d_rows = (a.H + grid - 1) / grid;
  pl->d_stages = mt_depth(static_cast<int>((d_rows + 7) / 8), 1, pl->d_stage_bytes, pl->d_kp, 1, pl->d_nsbx,
                          a.ntok, a.topk, dev, &pl->d_sep);
  if (!pl->d_stages) return false;
  pl->d_smem =
      mt_layout(pl->d_stages, pl->d_stage_bytes, pl->d_kp, 1, pl->d_nsbx, a.ntok, a.topk, pl->d_sep).total;
  return true;
}

cudaError_t moe_tc_gateup_launch(const MoeTcPlan &pl, const MoeArgs &a, cudaStream_t s) {
  MtParams p;
  p.a = a;
  p.stages = pl.g_stages;
  p.stage_bytes = pl.g_stage_bytes;
  p.nsbx = a.H / 256;
  p.frag_sep = pl.g_sep;
  const unsigned gr = pl.grid;
  const uint32_t sm = pl.g_smem;
  const int kp = pl.g_kp, w = pl.g_nsbw;
  if (pl.g_full) {
    if (w == 1) switch (kp) {
        case 1: return mt_launch(moe_gateup_tc_kernel<1, 1, true>, p, gr, sm, s);
        case 2: return mt_launch(moe_gateup_tc_kernel<2, 1, true>, p, gr, sm, s);
        case 4: return mt_launch(moe_gateup_tc_kernel<4, 1, true>, p, gr, sm, s);
        case 8: return mt_launch(moe_gateup_tc_kernel<8, 1, true>, p, gr, sm, s);
        case 16: return mt_launch(moe_gateup_tc_kernel<16, 1, true>, p, gr, sm, s);
      }
    if (kp == 16 && w == 2) return mt_launch(moe_gateup_tc_kernel<16, 2, true>, p, gr, sm, s);
    if (kp == 16 && w == 4) return mt_launch(moe_gateup_tc_kernel<16, 4, true>, p, gr, sm, s);
  } else {
    if (w == 1) switch (kp) {
        case 2: return mt_launch(moe_gateup_tc_kernel<2, 1, false>, p, gr, sm, s);
        case 4: return mt_launch(moe_gateup_tc_kernel<4, 1, false>, p, gr, sm, s);
        case 8: return mt_launch(moe_gateup_tc_kernel<8, 1, false>, p, gr, sm, s);
        case 16: return mt_launch(moe_gateup_tc_kernel<16, 1, false>, p, gr, sm, s);
      }
    if (kp == 16 && w == 2) return mt_launch(moe_gateup_tc_kernel<16, 2, false>, p, gr, sm, s);
    if (kp == 16 && w == 4) return mt_launch(moe_gateup_tc_kernel<16, 4, false>, p, gr, sm, s);
  }
  return cudaErrorInvalidConfiguration;
}

cudaError_t moe_tc_down_launch(const MoeTcPlan &pl, const MoeArgs &a, cudaStream_t s) {
  MtParams p;
  p.a = a;
  p.stages = pl.d_stages;
  p.stage_bytes = pl.d_stage_bytes;
  p.nsbx = pl.d_nsbx;
  p.frag_sep = pl.d_sep;
  const unsigned gr = pl.grid;
  const uint32_t sm = pl.d_smem;
  const int kp = pl.d_kp, w = pl.d_nsbw;
  if (w == 1) switch (kp) {
      case 1: return mt_launch(moe_down_tc_kernel<1, 1>, p, gr, sm, s);
      case 2: return mt_launch(moe_down_tc_kernel<2, 1>, p, gr, sm, s);
      case 4: return mt_launch(moe_down_tc_kernel<4, 1>, p, gr, sm, s);
      case 8: return mt_launch(moe_down_tc_kernel<8, 1>, p, gr, sm, s);
      case 16: return mt_launch(moe_down_tc_kernel<16, 1>, p, gr, sm, s);
    }
  if (kp == 16 && w == 2) return mt_launch(moe_down_tc_kernel<16, 2>, p, gr, sm, s);
  if (kp == 16 && w == 4) return mt_launch(moe_down_tc_kernel<16, 4>, p, gr, sm, s);
  return cudaErrorInvalidConfiguration;
}

}  // namespace epq

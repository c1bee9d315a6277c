// Mixture-of-experts layer (epq_moe_forward).
//
// "Flash-MoE：在笔记本上运行 397B 参数大模型", section "每层流水线": router
// matvec, softmax + top-K, then the selected experts' forward and the
// combine.  Here all of it stays on the GPU in three kernels on one stream:
//
//   1. router_kernel   logits = R xin (+bias) for every token (warp per
//                      expert row, the row's first loads issued before the
//                      grid-dependency wait), plus max|x| and the RMS factor.
//   2. gateup_kernel   every CTA first routes all tokens on its own from the
//                      logits (softmax + top-K per token, then grouping: the
//                      distinct experts in ascending order become "slots",
//                      each with its list of (token, choice) entries; the
//                      shared expert is the last slot and serves every
//                      token), so no grid-wide step sits between the router
//                      and the expert weights.  Then a persistent staged
//                      dequant-GEMV over the virtual rows slot*I + i: each
//                      tile stages the gate rows and the matching up rows of
//                      one expert; every token entry of the slot reuses the
//                      staged bytes; the epilogue writes h = silu(g) * u and
//                      records max|h| per (token, slot).  CTA 0 publishes the
//                      routing for the down kernel and the caller.
//   3. down_kernel     persistent over hidden rows: for each tile of rows the
//                      down rows of every slot are staged in turn, applied to
//                      each entry's h, weighted and accumulated per token in
//                      shared memory; then y = x + accumulated sum.
//
// Each expert's weights are read once per layer however many tokens use it.
#include <algorithm>
#include <mutex>

#include "gemv_core.cuh"

#include "moe_common.cuh"
#include "moe_k16.cuh"
#include "moe_tc.cuh"

namespace epq {
namespace {

// ------------------------------------------------------------------ 1. router
constexpr int kRouterWarps = kRouterThreads / 32;
constexpr int kRouterXSmem = 40 * 1024;  // stage x in shared memory up to this size (static smem stays < 48 KB)
constexpr int kRouterChunk = 16;         // 16-byte loads of a router row in flight per lane
constexpr int64_t kRouterStageMax = 200 * 1024;  // staged router: shared memory for the CTA's rows and x

// chunk j0.. of router row r (zeros past the row or for r >= r_end)
__device__ __forceinline__ void router_chunk(const MoeArgs &a, int r, int r_end, int j0, int lane,
                                             float4 (&wv)[kRouterChunk]) {
  const int n4 = a.H / 4;
  const float4 *wrow = reinterpret_cast<const float4 *>(r < a.E ? a.R + static_cast<int64_t>(r) * a.H : a.gvec);
#pragma unroll
  for (int u = 0; u < kRouterChunk; ++u) {
    const int j = j0 + u * 32 + lane;
    wv[u] = (r < r_end && j < n4) ? __ldcs(wrow + j) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Router logits of every token (NT >= ntok): warp per row of R; the rows
// E.. hold the shared-expert gate vector as one extra row.  The first chunk
// of each warp's first row is requested before the grid-dependency wait (R
// is a weight: nothing upstream writes it).  CTA 0 publishes max|x| and the
// RMS factor per token and clears the max|h| accumulators of the gate/up
// kernel.
//
// STAGED: the CTA's rows of R (all but the gate-vector row) arrive in
// dynamic shared memory through one bulk copy issued before the wait, so the
// whole router matrix streams while the previous kernel finishes; the dot
// products then read the same values in the same order from shared memory.
template <int NT, bool STAGED>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const MoeArgs a) {
  extern __shared__ __align__(16) uint8_t r_rows[];  // STAGED: [rows of this CTA][H]
  __shared__ float s_part[2][kRouterWarps][NT];
  __shared__ float s_rms[NT];
  __shared__ __align__(16) float s_x[STAGED ? 4 : kRouterXSmem / 4];  // STAGED: x follows the rows
  __shared__ __align__(8) uint64_t r_bar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nrows = a.E + (a.gvec ? 1 : 0);
  const int r_begin = static_cast<int>((static_cast<int64_t>(blockIdx.x) * nrows) / gridDim.x);
  const int r_end = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * nrows) / gridDim.x);
  const int n4 = a.H / 4;  // multiple of 64
  float4 wv[kRouterChunk];
  if (STAGED) {
    if (tid == 0) {
      mbar_init(&r_bar, 1);
      fence_mbar_init();
      const int nr = max(0, min(r_end, a.E) - r_begin);
      const uint32_t bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(a.H) * 4u;
      mbar_arrive_expect_tx(&r_bar, bytes);
      if (bytes) bulk_g2s(r_rows, a.R + static_cast<int64_t>(r_begin) * a.H, bytes, &r_bar);
    }
  } else {
    router_chunk(a, r_begin + warp, r_end, 0, lane, wv);
  }
  pdl_launch_dependents();
  pdl_wait();

  // x staged in shared memory; per-token sum of squares and max |x|
  const bool xs = STAGED || static_cast<int64_t>(a.ntok) * a.H * 4 <= kRouterXSmem;
  float *xsm = STAGED ? reinterpret_cast<float *>(r_rows) + static_cast<int64_t>(max(0, min(r_end, a.E) - r_begin)) * a.H
                      : s_x;
  for (int t = 0; t < a.ntok; ++t) {
    float ss = 0.0f, mx = 0.0f;
    const float4 *src = reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(t) * a.H);
#pragma unroll 4
    for (int j = tid; j < n4; j += kRouterThreads) {
      const float4 v = src[j];
      if (xs) reinterpret_cast<float4 *>(xsm + t * a.H)[j] = v;
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    ss = warp_sum_xor<32>(ss);
    mx = warp_max_all(mx);
    if (lane == 0) {
      s_part[0][warp][t] = ss;
      s_part[1][warp][t] = mx;
    }
  }
  __syncthreads();
  if (tid < a.ntok) {
    float tot = 0.0f, m = 0.0f;
    for (int w = 0; w < kRouterWarps; ++w) {
      tot += s_part[0][w][tid];
      m = fmaxf(m, s_part[1][w][tid]);
    }
    const float r = a.rms ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, static_cast<float>(a.H)), a.eps)))
                          : 1.0f;
    s_rms[tid] = r;
    if (blockIdx.x == 0) {
      a.xstat[2 * tid] = m;
      a.xstat[2 * tid + 1] = r;
    }
  }
  if (blockIdx.x == 0)
    for (int i = tid; i < a.ntok * (a.topk + 1); i += kRouterThreads) a.hmax[i] = 0u;
  __syncthreads();
  const float *xbase = xs ? xsm : a.x;
  if (STAGED && !warp_wait(&r_bar, 0, a.err, DEVERR_FULL_WAIT, 0)) {
    if (lane == 0) mbar_wait(&r_bar, 0, a.err, DEVERR_DRAIN_WAIT, 0);  // no copy in flight at exit
    return;
  }

  bool preloaded = !STAGED;
  for (int r = r_begin + warp; r < r_end; r += kRouterWarps) {
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    for (int j0 = 0; j0 < n4; j0 += 32 * kRouterChunk) {
      if (STAGED && r < a.E) {
        const float4 *wrow = reinterpret_cast<const float4 *>(r_rows) + static_cast<int64_t>(r - r_begin) * n4;
#pragma unroll
        for (int u = 0; u < kRouterChunk; ++u) {
          const int j = j0 + u * 32 + lane;
          wv[u] = j < n4 ? wrow[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      } else if (!preloaded) {
        router_chunk(a, r, r_end, j0, lane, wv);
      }
      preloaded = false;
#pragma unroll
      for (int u = 0; u < kRouterChunk; ++u) {
        const int j = j0 + u * 32 + lane;
        if (j < n4) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t < a.ntok) {
              const float4 xv = reinterpret_cast<const float4 *>(xbase + static_cast<int64_t>(t) * a.H)[j];
              acc[t] = fmaf(wv[u].x, xv.x, fmaf(wv[u].y, xv.y, fmaf(wv[u].z, xv.z, fmaf(wv[u].w, xv.w, acc[t]))));
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < a.ntok) {
        const float v = warp_sum_xor<32>(acc[t]) * s_rms[t];
        if (lane == 0) {
          if (r < a.E) {
            a.logits[static_cast<int64_t>(t) * a.E + r] = v + (a.bias ? a.bias[r] : 0.0f);
          } else {
            a.gshared[t] = __fdiv_rn(1.0f, 1.0f + expf(-v));
          }
        }
      }
    }
  }
}

// Routing alone, for a call that runs the router stage without the gate/up
// stage: one CTA computes and publishes what the gate/up kernel would.
constexpr int kSelectThreads = 256;
__global__ void __launch_bounds__(kSelectThreads) select_kernel(const MoeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_sel[];
  Meta m(smem_sel, a.ntok, a.topk);
  uint32_t *scratch = reinterpret_cast<uint32_t *>(smem_sel + ((4u * meta_words(a.ntok, a.topk) + 15u) & ~15u));
  m.clear(threadIdx.x, blockDim.x);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  route_tokens(a, m, scratch, true);
}

// ------------------------------------------------------------------ engine plan
constexpr int kRedRing = 4;
constexpr int kHSmemMax = 64 * 1024;  // stage all SwiGLU outputs in smem up to this size

struct EnginePlan {
  int tpr, groups, rpg, tile_rows, stages;
  uint32_t stage_bytes, smem, bar_off, red_off, meta_off, hs_off, acc_off;
  int stage_h;  // down: all of h staged in shared memory
};

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// largest down RPG the per-token accumulators allow (RPG * NT <= 32)
inline int down_max_rpg(int ntok) { return ntok <= 4 ? 8 : 2; }

constexpr int64_t kMoeTileBytes = 96 * 1024;  // a tile may hold all of a CTA's decode-sized share

// cols: weights per row; per_row: staged bytes per output row; rows_hint:
// output rows a CTA is expected to own (the tile grows until it covers
// them, within kMoeTileBytes).  Down: a thread takes every tpr-th column
// block (tpr <= 32) and RPG is bounded by its per-token accumulators.
bool engine_plan(int cols, int64_t per_row, bool swiglu, int64_t rows_hint, int ntok, int topk, int I_for_h,
                 bool down, const DeviceInfo &dev, EnginePlan *pl) {
  const int nblk = cols / 32;
  pl->tpr = down ? std::min(32, std::max(8, next_pow2(nblk)))
                 : (nblk <= 32 ? std::max(8, next_pow2(nblk)) : ((nblk + 31) / 32) * 32);
  if (pl->tpr > kMaxConsumers) return false;
  pl->groups = std::max(1, kMaxConsumers / pl->tpr);
  const int rmax = down ? std::min(8, down_max_rpg(ntok)) : std::min(8, std::min(pl->tpr, 32));
  auto tile_rows_of = [&](int r) { return static_cast<int64_t>(pl->groups) * (swiglu ? r / 2 : r); };
  const int64_t tile_cap = std::max<int64_t>(tune_tile_bytes(), kMoeTileBytes);
  int rpg = swiglu ? 2 : 1;
  while (rpg * 2 <= rmax && tile_rows_of(rpg * 2) * per_row <= tile_cap &&
         tile_rows_of(rpg * 2) <= std::max<int64_t>(rows_hint, tile_rows_of(rpg)))
    rpg *= 2;
  pl->rpg = rpg;
  pl->tile_rows = static_cast<int>(tile_rows_of(rpg));
  pl->stage_bytes = static_cast<uint32_t>((pl->tile_rows * per_row + 15) & ~int64_t(15));
  const int wpg = pl->tpr > 32 ? pl->tpr / 32 : 1;
  const uint32_t red_bytes = down ? 0u : 4u * kRedRing * pl->groups * rpg * wpg;
  const uint32_t meta_bytes = 4u * meta_words(ntok, topk);
  const int64_t hbytes = 4ll * ntok * (topk + 1) * I_for_h;
  pl->stage_h = down && hbytes <= kHSmemMax;
  // staged h: the scaled values plus one scaled column sum per 32 values
  const uint32_t hs_bytes = pl->stage_h ? static_cast<uint32_t>(hbytes + hbytes / 32) : 0u;
  const uint32_t acc_bytes = 0u;
  pl->stages = static_cast<int>(
      std::max<int64_t>(2, std::min<int64_t>(down ? 16 : 8, tune_ring_bytes() / pl->stage_bytes)));
  for (;;) {
    uint32_t o = pl->stages * pl->stage_bytes + 16;
    o = (o + 15) & ~15u;
    pl->bar_off = o;
    o += 16u * pl->stages + 16u * kRedRing;
    pl->red_off = o;
    o += red_bytes;
    o = (o + 15) & ~15u;
    pl->meta_off = o;
    o += meta_bytes;
    o = (o + 15) & ~15u;
    pl->hs_off = o;
    o += hs_bytes;
    pl->acc_off = o;
    o += acc_bytes;
    pl->smem = (o + 15) & ~15u;
    if (pl->smem <= static_cast<uint32_t>(dev.max_smem_optin) || pl->stages <= 2) break;
    --pl->stages;
  }
  return pl->smem <= static_cast<uint32_t>(dev.max_smem_optin);
}

// One-shot down form (down_flat_kernel): every slot's rows of a CTA staged
// at once.  Returns false when the shapes need the pipelined form.
bool flat_down_plan(int I, int64_t row_bytes, int H, unsigned grid, int max_slots, int ntok, int topk,
                    const DeviceInfo &dev, EnginePlan *pl) {
  if (ntok > 4) return false;
  const int nblk = I / 32;
  const int64_t hbytes = 4ll * ntok * (topk + 1) * I;
  if (hbytes > kHSmemMax) return false;
  pl->tpr = std::min(32, std::max(8, next_pow2(nblk)));
  pl->groups = kMaxConsumers / pl->tpr;
  pl->rpg = 1;
  pl->tile_rows = static_cast<int>((H + grid - 1) / grid);
  pl->stage_bytes = static_cast<uint32_t>((pl->tile_rows * row_bytes + 15) & ~int64_t(15));
  pl->stages = max_slots;
  pl->stage_h = 1;
  const int nt = ntok <= 1 ? 1 : 4;
  uint32_t o = static_cast<uint32_t>(max_slots) * pl->stage_bytes;
  o = (o + 15) & ~15u;
  pl->bar_off = o;
  o += 16;
  pl->red_off = o;
  pl->meta_off = o;
  o += 4u * meta_words(ntok, topk);
  o = (o + 15) & ~15u;
  pl->hs_off = o;
  o += static_cast<uint32_t>(hbytes + hbytes / 32);
  o = (o + 15) & ~15u;
  pl->acc_off = o;
  o += 4u * max_slots * pl->tile_rows * nt;
  pl->smem = (o + 15) & ~15u;
  return pl->smem <= static_cast<uint32_t>(dev.max_smem_optin);
}

// One-shot gate/up form (gateup_flat_kernel): a CTA's whole share of gate
// and up rows staged at once.  Returns false when the shapes need the
// pipelined form.
bool flat_gateup_plan(int H, int64_t row_bytes, int I, unsigned grid, int max_slots, int ntok, int topk,
                      const DeviceInfo &dev, EnginePlan *pl) {
  if (ntok > 4) return false;
  const int nblk = H / 32;
  pl->tpr = std::min(32, std::max(8, next_pow2(nblk)));
  pl->groups = kMaxConsumers / pl->tpr;
  pl->rpg = 2;
  pl->tile_rows = static_cast<int>((static_cast<int64_t>(max_slots) * I + grid - 1) / grid);
  pl->stage_bytes = static_cast<uint32_t>((2 * pl->tile_rows * row_bytes + 15) & ~int64_t(15));
  if (pl->stage_bytes < 4u * kSelScratchWords) pl->stage_bytes = 4u * kSelScratchWords;  // routing scratch
  pl->stages = 1;
  pl->stage_h = 0;
  uint32_t o = pl->stage_bytes;
  pl->bar_off = o;
  o += 16;
  pl->red_off = o;
  pl->meta_off = o;
  o += 4u * meta_words(ntok, topk);
  o = (o + 15) & ~15u;
  pl->hs_off = o;  // scaled x pairs and column sums
  o += static_cast<uint32_t>(4ll * ntok * H + 4ll * ntok * nblk);
  o = (o + 15) & ~15u;
  pl->acc_off = o;  // per-CTA max|h|
  o += 4u * ntok * (topk + 1);
  pl->smem = (o + 15) & ~15u;
  return pl->smem <= static_cast<uint32_t>(dev.max_smem_optin);
}

struct EngineArgs {
  MoeArgs a;
  int tpr, groups, tile_rows, stages, stage_h;
  uint32_t stage_bytes, bar_off, red_off, meta_off, hs_off, acc_off;
};

// h of every (token, slot) for the down kernels' shared-memory copy: the
// float4 loads are issued first (with the routing loads), the scaling into
// pairs waits for the exponents.  hbytes <= kHSmemMax, 512 consumers.
constexpr int kHStage4 = kHSmemMax / 16 / kMaxConsumers;  // float4 per thread

__device__ __forceinline__ void load_h(const MoeArgs &a, int n4, int tid, int lane, int nthreads,
                                       float4 (&hv)[kHStage4]) {
#pragma unroll
  for (int k = 0; k < kHStage4; ++k) {
    const int q = (tid - lane) + k * nthreads + lane;
    hv[k] = q < n4 ? reinterpret_cast<const float4 *>(a.h)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// pair i of column c of slot vector hsi at pairs[(hsi*16 + i)*nblk + c]
// (neighbouring threads read neighbouring pairs); scaled column sums in
// hsum[hsi*nblk + c].  8 consecutive threads hold one 32-float column.
template <int FMT>
__device__ __forceinline__ void stage_h(const float4 (&hv)[kHStage4], const Meta &m, int I, int nblk, int n4, int tid,
                                        int lane, int nthreads, f2_t *pairs, float *hsum) {
#pragma unroll
  for (int k = 0; k < kHStage4; ++k) {
    const int q0 = (tid - lane) + k * nthreads;
    if (q0 >= n4) break;  // warp-uniform; n4 is a multiple of 64
    const int q = q0 + lane;
    const float4 v = hv[k];
    const int hsi = (4 * q) / I;
    const int col = ((4 * q) - hsi * I) >> 5;
    const int j = (4 * q) & 31;
    const int E = m.expo[hsi];
    float sum = (v.x + v.y) + (v.z + v.w);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    const int base = (hsi * 16 + j / 2) * nblk + col;
    pairs[base] = f2_pack(scale_pow2(v.x, 126 - E - Fmt<FMT>::shift(j)),
                          scale_pow2(v.y, 126 - E - Fmt<FMT>::shift(j + 1)));
    pairs[base + nblk] = f2_pack(scale_pow2(v.z, 126 - E - Fmt<FMT>::shift(j + 2)),
                                 scale_pow2(v.w, 126 - E - Fmt<FMT>::shift(j + 3)));
    if (j == 0) hsum[hsi * nblk + col] = scale_pow2(sum, -23 - E);
  }
}

// Row reduction of one (unit, entry) for RPG partials: in-warp reduce-scatter,
// then either the row holder (groups within a warp) returns its row, or the
// warp hands its partials to the finisher through ring buffer `b`.
template <int RPG>
__device__ __forceinline__ int reduce_or_hand_off(float (&part)[1][RPG], const EngineArgs &p, int g, int c,
                                                  int lane, float *red, uint64_t *rfull, uint64_t *rempty, int use,
                                                  bool &ok) {
  const int W = p.tpr < 32 ? p.tpr : 32;
  const int ri = reduce_scatter<RPG, 1>(part, W, lane % W);
  if (p.tpr > 32) {
    const int wpg = p.tpr / 32;
    const int b = use % kRedRing;
    if (use >= kRedRing && !warp_wait(&rempty[b], ((use / kRedRing) - 1) & 1, p.a.err, DEVERR_RED_WAIT, use)) {
      ok = false;
      return -1;
    }
    float *rbuf = red + b * p.groups * RPG * wpg;
    if ((lane % (32 / RPG)) == 0) rbuf[(g * RPG + ri) * wpg + (c >> 5)] = part[0][0];
    __syncwarp();
    if (lane == 0) mbar_arrive(&rfull[b]);
    return -1;
  }
  return (((lane % W) % (W / RPG)) == 0) ? ri : -1;
}

// Finisher side of the hand-off: wait for ring buffer of `use`, sum the
// warp partials of slot row `r` (0..groups*RPG-1).
__device__ __forceinline__ float fin_row(const float *rbuf, int r, int wpg) {
  float acc = 0.0f;
  for (int w = 0; w < wpg; ++w) acc += rbuf[r * wpg + w];
  return acc;
}


// Producer warp: expert id of `slot` (slot >= nact means the shared expert,
// returned as -1).  The ids are fetched once, 32 per lane-parallel load, so
// the producer never waits on a global load between bulk copies.
struct SlotIds {
  int ids[ (kMaxTok * kMaxTopk + 1 + 31) / 32 ];  // one id per lane per chunk
  int nact;
  __device__ void load(const MoeArgs &a, int lane) {
    nact = __ldcg(a.meta);
#pragma unroll
    for (int c = 0; c < (kMaxTok * kMaxTopk + 1 + 31) / 32; ++c) {
      const int s = c * 32 + lane;
      ids[c] = s < nact ? __ldcg(a.active + s) : -1;
    }
  }
  // all lanes of the warp must call this
  __device__ int get(int slot) const {
    int v = -1;
#pragma unroll
    for (int c = 0; c < (kMaxTok * kMaxTopk + 1 + 31) / 32; ++c)
      if (slot / 32 == c) v = __shfl_sync(0xffffffffu, ids[c], slot & 31);
    return slot < nact ? v : -1;
  }
};

// ------------------------------------------------------------------ 2. gate/up
// Virtual rows [rb, re) of CTA b out of G when each row of slot s costs
// max(1, cnt[s]) units: the CTAs get equal shares of the total, and every
// CTA evaluates the same monotonic map, so the ranges tile the rows exactly.
__device__ __forceinline__ void weighted_rows(const Meta &m, int I, int nslots, int b, int G, int64_t &rb,
                                              int64_t &re) {
  int64_t W = 0;
  for (int s = 0; s < nslots; ++s) W += static_cast<int64_t>(I) * max(1, m.cnt[s]);
  auto row_at = [&](int64_t w) -> int64_t {  // first row whose work starts at or after w
    int64_t acc = 0;
    for (int s = 0; s < nslots; ++s) {
      const int64_t c = max(1, m.cnt[s]);
      if (w < acc + static_cast<int64_t>(I) * c) return static_cast<int64_t>(s) * I + (w - acc + c - 1) / c;
      acc += static_cast<int64_t>(I) * c;
    }
    return static_cast<int64_t>(nslots) * I;
  };
  rb = row_at(W * b / G);
  re = row_at(W * (b + 1) / G);
}

template <int FMT, int RPG>
__global__ void __launch_bounds__(kMaxConsumers + 64, 1) gateup_kernel(const EngineArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const MoeArgs &a = p.a;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);
  uint64_t *empty = full + p.stages;
  uint64_t *rfull = empty + p.stages;
  uint64_t *rempty = rfull + kRedRing;
  float *red = reinterpret_cast<float *>(smem + p.red_off);
  const int nthreads = p.groups * p.tpr;
  const int nwarps = nthreads / 32;
  const bool has_fin = p.tpr > 32;
  const int wpg = has_fin ? p.tpr / 32 : 1;
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int RH = RPG / 2;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nwarps);
    }
    for (int b = 0; b < kRedRing; ++b) {
      mbar_init(&rfull[b], nwarps);
      mbar_init(&rempty[b], 1);
    }
    fence_mbar_init();
  }
  Meta m(smem + p.meta_off, a.ntok, a.topk);
  m.clear(tid, blockDim.x);
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // logits and x statistics come from the router kernel

  // consumer coordinates (the x column is loaded once the routing is done)
  const int g = tid / p.tpr, c = tid % p.tpr;
  const int nblk = a.H / 32;
  const bool active = tid < nthreads && c < nblk;
  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  XCol<1> xc;
  float xs[1] = {0.0f};
  int cur_t = -1;
  if (active && g == 0)  // token 0's x lines, into L1 while the routing runs
    prefetch_l1(a.x + 32 * c);
  route_tokens(a, m, reinterpret_cast<uint32_t *>(smem), blockIdx.x == 0);  // the ring is free until routed

  const int I = a.I;
  const int nact = *m.nact;
  // every entry of a slot is one more dot product per row: equal shares of
  // rows x entries, not of rows (the shared expert serves every token)
  int64_t rb, re;
  weighted_rows(m, I, *m.nslots, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), rb, re);
  auto tile_len = [&](int64_t r0) {
    const int64_t lim = min(re, (r0 / I + 1) * I);
    return static_cast<int>(min(static_cast<int64_t>(p.tile_rows), lim - r0));
  };

  if (tid >= nthreads && tid < nthreads + 32) {
    // producer: one thread issues two bulk copies per tile (gate rows, up rows)
    if (tid != nthreads) return;
    int issued = 0;
    bool ok = true;
    int t = 0;
    for (int64_t r0 = rb; r0 < re; r0 += tile_len(r0), ++t) {
      const int s = t % p.stages;
      const int slot = static_cast<int>(r0 / I);
      const int e = slot < nact ? m.active[slot] : -1;
      if (t >= p.stages && !mbar_wait(&empty[s], ((t / p.stages) - 1) & 1, a.err, DEVERR_EMPTY_WAIT, t)) {
        ok = false;
        break;
      }
      const int nr = tile_len(r0);
      const int i0 = static_cast<int>(r0 % I);
      const uint8_t *base = e >= 0 ? a.gate_up + static_cast<int64_t>(e) * a.gu_stride : a.sh_gate_up;
      const uint32_t bytes = static_cast<uint32_t>(nr * a.gu_row_bytes);
      uint8_t *dst = smem + static_cast<uint32_t>(s) * p.stage_bytes;
      mbar_arrive_expect_tx(&full[s], 2 * bytes);
      bulk_g2s(dst, base + static_cast<int64_t>(i0) * a.gu_row_bytes, bytes, &full[s]);
      bulk_g2s(dst + p.tile_rows * a.gu_row_bytes, base + static_cast<int64_t>(I + i0) * a.gu_row_bytes, bytes,
               &full[s]);
      ++issued;
    }
    if (!ok) {
      // drain: wait (bounded) for every copy still in flight before leaving
      for (int u = max(0, issued - p.stages); u < issued; ++u)
        mbar_wait(&full[u % p.stages], (u / p.stages) & 1, a.err, DEVERR_DRAIN_WAIT, u);
    }
    return;
  }

  const bool is_fin = tid >= nthreads + 32;
  if (is_fin) {
    int use = 0, t = 0;
    for (int64_t r0 = rb; r0 < re; r0 += tile_len(r0), ++t) {
      const int nr = tile_len(r0);
      const int slot = static_cast<int>(r0 / I);
      const int i0 = static_cast<int>(r0 % I);
      const int ne = m.cnt[slot];
      for (int j = 0; j < ne; ++j, ++use) {
        const int b = use % kRedRing;
        if (!warp_wait(&rfull[b], (use / kRedRing) & 1, a.err, DEVERR_RED_WAIT, use)) return;
        const float *rbuf = red + b * p.groups * RPG * wpg;
        const int ent = m.list[slot * a.ntok + j];
        const int tok = ent >> 5, k = ent & 31;
        const int E = m.expo[tok];
        const float r = m.rms[tok];
        const int hs = tok * (a.topk + 1) + k;
        unsigned hm = 0u;
        for (int o = lane; o < nr; o += 32) {
          const int gg = o / RH, kk = o % RH;
          const float gv = unscale(fin_row(rbuf, gg * RPG + kk, wpg), E) * r;
          const float uv = unscale(fin_row(rbuf, gg * RPG + RH + kk, wpg), E) * r;
          const float hv = silu(gv) * uv;
          a.h[static_cast<int64_t>(hs) * I + i0 + o] = hv;
          hm = max(hm, __float_as_uint(fabsf(hv)));
        }
        hm = __reduce_max_sync(0xffffffffu, hm);
        if (lane == 0 && hm) atomicMax(a.hmax + hs, hm);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[b]);
      }
    }
    return;
  }

  float xr[32];
  int use = 0, t = 0;
  for (int64_t r0 = rb; r0 < re; r0 += tile_len(r0), ++t) {
    const int s = t % p.stages;
    if (!warp_wait(&full[s], (t / p.stages) & 1, a.err, DEVERR_FULL_WAIT, t)) return;
    const int nr = tile_len(r0);
    const int slot = static_cast<int>(r0 / I);
    const int i0 = static_cast<int>(r0 % I);
    const uint8_t *stage = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    const int ne = m.cnt[slot];
    bool ok = true;
    for (int j = 0; j < ne; ++j, ++use) {
      const int ent = m.list[slot * a.ntok + j];
      const int tok = ent >> 5, k = ent & 31;
      if (tok != cur_t) {
        cur_t = tok;
        if (active) {
          load_column(a.x + static_cast<int64_t>(tok) * a.H + 32 * c, xr);
          xs[0] = scale_column<FMT>(xr, m.expo[tok], xc.p[0]);
        }
      }
      float part[1][RPG];
#pragma unroll
      for (int q = 0; q < RPG; ++q) {
        const int lr = g * RH + (q % RH);
        float pr[1] = {0.0f};
        if (active && lr < nr) {
          const uint8_t *row = stage + static_cast<uint32_t>(lr) * a.gu_row_bytes;
          if (q >= RH) row += p.tile_rows * a.gu_row_bytes;
          column_dot<FMT, 1>(row, cc, xc, xs, pr);
        }
        part[0][q] = pr[0];
      }
      if (j == ne - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage is no longer read
      }
      const int row_k = reduce_or_hand_off<RPG>(part, p, g, c, lane, red, rfull, rempty, use, ok);
      if (__any_sync(0xffffffffu, !ok)) return;
      if (!has_fin) {
        const int W = p.tpr < 32 ? p.tpr : 32;
        const float up = __shfl_xor_sync(0xffffffffu, part[0][0], W / 2);
        const int hs = tok * (a.topk + 1) + k;  // the same entry for the whole warp
        unsigned hm = 0u;
        if (row_k >= 0 && row_k < RH) {
          const int lr = g * RH + row_k;
          if (lr < nr) {
            const int E = m.expo[tok];
            const float r = m.rms[tok];
            const float hv = silu(unscale(part[0][0], E) * r) * (unscale(up, E) * r);
            a.h[static_cast<int64_t>(hs) * I + i0 + lr] = hv;
            hm = __float_as_uint(fabsf(hv));
          }
        }
        hm = __reduce_max_sync(0xffffffffu, hm);
        if (lane == 0 && hm) atomicMax(a.hmax + hs, hm);
      }
    }
  }
}

// ------------------------------------------------------------------ 2b. gate/up, one-shot form
// Used when a CTA's whole share of gate and up rows fits shared memory at
// once (decode).  While the last warps select the experts, the other warps
// stage x of every token in scaled form; after routing the producer copies
// the CTA's rows (per slot segment: the gate rows, then the matching up
// rows) on one barrier.  Group g takes virtual rows g, g + groups, ...: for
// every entry of the row's slot it forms the gate and up dots over its
// column blocks, reduces them inside the group and writes
// h = silu(g) * u.  max|h| is reduced per CTA before one global atomic per
// (token, slot).  NT >= ntok.
template <int FMT, int NT>
__global__ void __launch_bounds__(kMaxConsumers, 1) gateup_flat_kernel(const EngineArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const MoeArgs &a = p.a;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);
  uint64_t *done = full + 1;
  f2_t *xpairs = reinterpret_cast<f2_t *>(smem + p.hs_off);  // [ntok][16][nblk]
  const int nthreads = p.groups * p.tpr;
  const int nwarps_c = nthreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int H = a.H, I = a.I;
  const int nblk = H / 32;
  float *xsum = reinterpret_cast<float *>(xpairs + static_cast<int64_t>(a.ntok) * 16 * nblk);  // [ntok][nblk]
  unsigned *hmax_cta = reinterpret_cast<unsigned *>(smem + p.acc_off);  // [ntok * (topk + 1)]

  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(done, nwarps_c);
    fence_mbar_init();
  }
  Meta m(smem + p.meta_off, a.ntok, a.topk);
  m.clear(tid, blockDim.x);
  for (int i = tid; i < a.ntok * (a.topk + 1); i += blockDim.x) hmax_cta[i] = 0u;
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // logits, x statistics and x come from the router kernel and before

  // x of every token, scaled, by the warps that do not start the selection
  const int nch = (a.E + 31) / 32;
  const int xwarps = nwarps - min(nwarps - 1, a.ntok * nch);
  if (warp < xwarps) {
    const int n4 = a.ntok * H / 4;  // a multiple of 64: whole warps
    int Ex[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) Ex[t] = t < a.ntok ? bound_exponent(__ldcg(a.xstat + 2 * t)) : 0;
    const int stride = xwarps * 32;
#pragma unroll 1
    for (int q0 = tid - lane; q0 < n4; q0 += 4 * stride) {
      float4 xv[4];  // four loads in flight before the first store
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + u * stride + lane;
        xv[u] = q < n4 ? reinterpret_cast<const float4 *>(a.x)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (q0 + u * stride >= n4) break;  // warp-uniform
        const int q = q0 + u * stride + lane;
        const float4 v = xv[u];
        const int t = (4 * q) / H;
        const int col = ((4 * q) - t * H) >> 5;
        const int j = (4 * q) & 31;
        const int E = t == 0 ? Ex[0] : (t == 1 ? Ex[1] : (t == 2 ? Ex[2] : Ex[3]));
        float sum = (v.x + v.y) + (v.z + v.w);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        const int base = (t * 16 + j / 2) * nblk + col;
        xpairs[base] = f2_pack(scale_pow2(v.x, 126 - E - Fmt<FMT>::shift(j)),
                               scale_pow2(v.y, 126 - E - Fmt<FMT>::shift(j + 1)));
        xpairs[base + nblk] = f2_pack(scale_pow2(v.z, 126 - E - Fmt<FMT>::shift(j + 2)),
                                      scale_pow2(v.w, 126 - E - Fmt<FMT>::shift(j + 3)));
        if (j == 0) xsum[t * nblk + col] = scale_pow2(sum, -23 - E);
      }
    }
  }
  route_tokens(a, m, reinterpret_cast<uint32_t *>(smem), blockIdx.x == 0);  // the stage area is free until routed

  const int nact = *m.nact;
  const int64_t total = static_cast<int64_t>(*m.nslots) * I;
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * total) / gridDim.x;
  const int nrows = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * total) / gridDim.x - rb);  // <= tile_rows
  uint8_t *gate_s = smem;
  uint8_t *up_s = smem + static_cast<uint32_t>(p.tile_rows) * a.gu_row_bytes;

  {
    // the last thread issues, per slot segment of this CTA's rows, the gate
    // rows and the up rows (there is no separate producer warp)
    if (tid == nthreads - 1 && nrows > 0) {
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(2 * nrows * a.gu_row_bytes));
      int64_t r0 = rb;
      const int64_t re = rb + nrows;
#pragma unroll 1
      while (r0 < re) {
        const int slot = static_cast<int>(r0 / I);
        const int64_t r1 = min(re, static_cast<int64_t>(slot + 1) * I);
        const int e = slot < nact ? m.active[slot] : -1;
        const uint8_t *base = e >= 0 ? a.gate_up + static_cast<int64_t>(e) * a.gu_stride : a.sh_gate_up;
        const int64_t i0 = r0 - static_cast<int64_t>(slot) * I;
        const uint32_t bytes = static_cast<uint32_t>((r1 - r0) * a.gu_row_bytes);
        const uint32_t off = static_cast<uint32_t>((r0 - rb) * a.gu_row_bytes);
        bulk_g2s(gate_s + off, base + i0 * a.gu_row_bytes, bytes, full);
        bulk_g2s(up_s + off, base + (I + i0) * a.gu_row_bytes, bytes, full);
        r0 = r1;
      }
    }
  }

  const int g = tid / p.tpr, c = tid % p.tpr;
  const bool active = c < nblk;
  const int cb_bytes = FMT == EPQ_Q4_K ? p.tpr * 144 / 8 : p.tpr * Fmt<FMT>::kBlockBytes;
  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  XCol<1> xc;
  float xs[1] = {0.0f};
  if (nrows > 0 && !warp_wait(full, 0, a.err, DEVERR_FULL_WAIT, 0)) return;
  const int iters = (nrows + p.groups - 1) / p.groups;  // the same for every warp
  const int ncb = (nblk + p.tpr - 1) / p.tpr;
  if (NT == 1 && ncb <= 2 && iters <= 4) {
    // one token: this lane's x column blocks are loaded once; the group's
    // rows (gate and up dots) are independent of each other
    XCol<1> x1;
    float xs1[1] = {0.0f};
    const bool two = ncb == 2 && c + p.tpr < nblk;
    if (active) {
#pragma unroll
      for (int q = 0; q < 16; ++q) xc.p[0][q] = xpairs[q * nblk + c];
      xs[0] = xsum[c];
      if (two) {
#pragma unroll
        for (int q = 0; q < 16; ++q) x1.p[0][q] = xpairs[q * nblk + c + p.tpr];
        xs1[0] = xsum[c + p.tpr];
      }
    }
    float pg[4], pu[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      pg[it] = 0.0f;
      pu[it] = 0.0f;
      const int v = g + it * p.groups;
      if (it < iters && v < nrows && active) {
        const uint8_t *grow = gate_s + static_cast<uint32_t>(v) * a.gu_row_bytes;
        const uint8_t *urow = up_s + static_cast<uint32_t>(v) * a.gu_row_bytes;
        float pr[1] = {0.0f};
        column_dot<FMT, 1>(grow, cc, xc, xs, pr);
        pg[it] = pr[0];
        pr[0] = 0.0f;
        column_dot<FMT, 1>(urow, cc, xc, xs, pr);
        pu[it] = pr[0];
        if (two) {
          pr[0] = 0.0f;
          column_dot<FMT, 1>(grow + cb_bytes, cc, x1, xs1, pr);
          pg[it] += pr[0];
          pr[0] = 0.0f;
          column_dot<FMT, 1>(urow + cb_bytes, cc, x1, xs1, pr);
          pu[it] += pr[0];
        }
      }
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      if (it < iters) {
        float gv = pg[it], uv = pu[it];
        for (int o = p.tpr / 2; o > 0; o >>= 1) {
          gv += __shfl_xor_sync(0xffffffffu, gv, o);
          uv += __shfl_xor_sync(0xffffffffu, uv, o);
        }
        const int v = g + it * p.groups;
        if (c == 0 && v < nrows) {
          const int64_t rv = rb + v;
          const int slot = static_cast<int>(rv / I);
          const int i = static_cast<int>(rv - static_cast<int64_t>(slot) * I);
          const int k = m.list[slot] & 31;
          const int E = m.expo[0];
          const float r = m.rms[0];
          const float hv = silu(unscale(gv, E) * r) * (unscale(uv, E) * r);
          a.h[static_cast<int64_t>(k) * I + i] = hv;
          atomicMax(hmax_cta + k, __float_as_uint(fabsf(hv)));
        }
      }
    }
  } else {
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int v = g + it * p.groups;
    const bool have = v < nrows;
    const int64_t rv = rb + (have ? v : 0);
    const int slot = static_cast<int>(rv / I);
    const int i = static_cast<int>(rv - static_cast<int64_t>(slot) * I);
    const int ne = have ? m.cnt[slot] : 0;
    const int ne_max = __reduce_max_sync(0xffffffffu, ne);
    const uint8_t *grow = gate_s + static_cast<uint32_t>(have ? v : 0) * a.gu_row_bytes;
    const uint8_t *urow = up_s + static_cast<uint32_t>(have ? v : 0) * a.gu_row_bytes;
#pragma unroll 1
    for (int jj = 0; jj < ne_max; ++jj) {
      const bool on = jj < ne;
      const int ent = on ? m.list[slot * a.ntok + jj] : 0;
      const int tok = ent >> 5, k = ent & 31;
      float pg = 0.0f, pu = 0.0f;
      if (on && active) {
#pragma unroll 1
        for (int cb = c, ib = 0; cb < nblk; cb += p.tpr, ++ib) {
#pragma unroll
          for (int q = 0; q < 16; ++q) xc.p[0][q] = xpairs[(tok * 16 + q) * nblk + cb];
          xs[0] = xsum[tok * nblk + cb];
          float pr[1] = {0.0f};
          column_dot<FMT, 1>(grow + ib * cb_bytes, cc, xc, xs, pr);
          pg += pr[0];
          pr[0] = 0.0f;
          column_dot<FMT, 1>(urow + ib * cb_bytes, cc, xc, xs, pr);
          pu += pr[0];
        }
      }
      for (int o = p.tpr / 2; o > 0; o >>= 1) {
        pg += __shfl_xor_sync(0xffffffffu, pg, o);
        pu += __shfl_xor_sync(0xffffffffu, pu, o);
      }
      if (on && c == 0) {
        const int E = m.expo[tok];
        const float r = m.rms[tok];
        const float hv = silu(unscale(pg, E) * r) * (unscale(pu, E) * r);
        const int hs = tok * (a.topk + 1) + k;
        a.h[static_cast<int64_t>(hs) * I + i] = hv;
        atomicMax(hmax_cta + hs, __float_as_uint(fabsf(hv)));
      }
    }
  }
  }
  // one global max|h| update per (token, slot) and CTA
  __syncwarp();
  if (lane == 0) mbar_arrive(done);
  if (warp == 0) {
    if (!warp_wait(done, 0, a.err, DEVERR_RED_WAIT, 0)) return;
#pragma unroll 1
    for (int q = lane; q < a.ntok * (a.topk + 1); q += 32)
      if (hmax_cta[q]) atomicMax(a.hmax + q, hmax_cta[q]);
  }
}

// ------------------------------------------------------------------ 3. down + combine
// Rows of y are split over the CTAs.  A unit is the CTA's rows (one tile of
// them) of one slot's down matrix; the units of a tile are staged slot by
// slot.  Row group g owns tile rows g*RPG .. g*RPG+RPG-1 for every slot: its
// threads accumulate w * (partial dot) per token in registers across all
// slots and entries, and the group reduces once per tile, when the tile's
// last slot is in, to write y = x + sum.  NT >= ntok.
template <int FMT, int RPG, int NT>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) down_kernel(const EngineArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const MoeArgs &a = p.a;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);
  uint64_t *empty = full + p.stages;
  float *hs_smem = reinterpret_cast<float *>(smem + p.hs_off);
  const int nthreads = p.groups * p.tpr;
  const int tid = threadIdx.x, lane = tid & 31;
  const int H = a.H, I = a.I;
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * H) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * H) / gridDim.x;
  const int ntiles = static_cast<int>((re - rb + p.tile_rows - 1) / p.tile_rows);
  // warps whose groups own rows of the first (largest) tile do the units;
  // the others only help stage h
  const int nr0 = static_cast<int>(min(static_cast<int64_t>(p.tile_rows), re - rb));
  const int work_groups = min(p.groups, (nr0 + RPG - 1) / RPG);
  const int work_warps = (work_groups * p.tpr + 31) / 32;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], work_warps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // h, routing and hmax come from the previous kernels

  if (tid >= nthreads) {
    // producer warp: the expert ids are held by the warp; one lane issues a
    // bulk copy per unit
    const int plane = tid - nthreads;
    const int nslots = __ldcg(a.meta + 1);
    SlotIds ids;
    ids.load(a, plane);
    const int nunits = ntiles * nslots;
    int issued = 0;
    bool ok = true;
    for (int u = 0; u < nunits; ++u) {
      const int s = u % p.stages;
      const int tile = u / nslots, slot = u % nslots;
      const int e = ids.get(slot);
      if (u >= p.stages && !warp_wait(&empty[s], ((u / p.stages) - 1) & 1, a.err, DEVERR_EMPTY_WAIT, u)) {
        ok = false;
        break;
      }
      const int64_t r0 = rb + static_cast<int64_t>(tile) * p.tile_rows;
      const int nr = static_cast<int>(min(static_cast<int64_t>(p.tile_rows), re - r0));
      const uint8_t *base = e >= 0 ? a.down + static_cast<int64_t>(e) * a.dn_stride : a.sh_down;
      const uint32_t bytes = static_cast<uint32_t>(nr * a.dn_row_bytes);
      if (plane == 0) {
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(smem + static_cast<uint32_t>(s) * p.stage_bytes, base + r0 * a.dn_row_bytes, bytes, &full[s]);
      }
      ++issued;
    }
    if (!ok && plane == 0) {
      for (int u = max(0, issued - p.stages); u < issued; ++u)
        mbar_wait(&full[u % p.stages], (u / p.stages) & 1, a.err, DEVERR_DRAIN_WAIT, u);
    }
    return;
  }

  // consumers: routing metadata (and all of h) into shared memory
  Meta m(smem + p.meta_off, a.ntok, a.topk);
  const int nblk = I / 32;
  const int nh = a.ntok * (a.topk + 1);
  const int n4 = p.stage_h ? nh * I / 4 : 0;
  float4 hv[kHStage4];
  load_h(a, n4, tid, lane, nthreads, hv);  // issued together with the routing loads
  load_meta(a, m, tid, nthreads);
  f2_t *pairs = reinterpret_cast<f2_t *>(hs_smem);
  float *hsum = hs_smem + static_cast<int64_t>(nh) * I;  // [nh][nblk]
  named_sync(1, nthreads);  // the h exponents are in m.expo
  if (p.stage_h) {
    stage_h<FMT>(hv, m, I, nblk, n4, tid, lane, nthreads, pairs, hsum);
    named_sync(1, nthreads);
  }
  const int nslots = *m.nslots;
  const int nunits = ntiles * nslots;
  if (tid >= work_warps * 32) return;

  // thread c of a group takes the column blocks c, c + tpr, ... (tpr <= 32,
  // so a row's reduction stays inside one warp)
  const int g = tid / p.tpr, c = tid % p.tpr;
  const bool active = c < nblk;
  // bytes of tpr column blocks (tpr is a multiple of 8: whole Q4_K superblocks)
  const int cb_bytes = FMT == EPQ_Q4_K ? p.tpr * 144 / 8 : p.tpr * Fmt<FMT>::kBlockBytes;
  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  float xr[32];
  XCol<1> xc;
  float xs[1] = {0.0f};
  float acc[RPG][NT];
#pragma unroll
  for (int q = 0; q < RPG; ++q)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[q][t] = 0.0f;
  for (int u = 0; u < nunits; ++u) {
    const int s = u % p.stages;
    if (!warp_wait(&full[s], (u / p.stages) & 1, a.err, DEVERR_FULL_WAIT, u)) return;
    const int tile = u / nslots, slot = u % nslots;
    const int64_t r0 = rb + static_cast<int64_t>(tile) * p.tile_rows;
    const int nr = static_cast<int>(min(static_cast<int64_t>(p.tile_rows), re - r0));
    const uint8_t *stage = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    const bool rows_here = active && g * RPG < nr;  // this group has rows in the tile
    const int ne = m.cnt[slot];
    for (int j = 0; j < ne; ++j) {
      const int ent = m.list[slot * a.ntok + j];
      const int tok = ent >> 5, k = ent & 31;
      const int hsi = tok * (a.topk + 1) + k;
      if (!rows_here) continue;
      const int E = m.expo[hsi];
      const float wk = k < a.topk ? m.w[tok * a.topk + k] : m.gs[tok];
      float part[RPG];
#pragma unroll
      for (int q = 0; q < RPG; ++q) part[q] = 0.0f;
      for (int cb = c, ib = 0; cb < nblk; cb += p.tpr, ++ib) {
        if (p.stage_h) {
#pragma unroll
          for (int i = 0; i < 16; ++i) xc.p[0][i] = pairs[(hsi * 16 + i) * nblk + cb];
          xs[0] = hsum[hsi * nblk + cb];
        } else {
          load_column(a.h + static_cast<int64_t>(hsi) * I + 32 * cb, xr);
          xs[0] = scale_column<FMT>(xr, E, xc.p[0]);
        }
#pragma unroll
        for (int q = 0; q < RPG; ++q) {
          const int lr = g * RPG + q;
          if (lr < nr) {
            float pr[1] = {0.0f};
            column_dot<FMT, 1>(stage + static_cast<uint32_t>(lr) * a.dn_row_bytes + ib * cb_bytes, cc, xc, xs, pr);
            part[q] += pr[0];
          }
        }
      }
#pragma unroll
      for (int q = 0; q < RPG; ++q) {
        const float v = wk * unscale(part[q], E);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t == tok) acc[q][t] += v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the stage is no longer read
    if (slot != nslots - 1) continue;

    // all slots of this tile are in: reduce each (row, token) over the group
    // and write y = x + weighted expert sum
#pragma unroll
    for (int q = 0; q < RPG; ++q) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float v = acc[q][t];
        for (int o = p.tpr / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int lr = g * RPG + q;
        if (c == 0 && t < a.ntok && lr < nr) {
          const int64_t o = static_cast<int64_t>(t) * H + r0 + lr;
          a.y[o] = a.x[o] + v;
        }
        acc[q][t] = 0.0f;
      }
    }
  }
}

// ------------------------------------------------------------------ 3b. down + combine, one-shot form
// Used when every slot's rows of a CTA fit shared memory at once (decode:
// a few KB per slot).  The producer stages them with one bulk copy per slot
// on a single barrier; the consumers then work on (slot, row) pairs with no
// per-unit synchronisation: group g takes pairs g, g + groups, ...; a pair's
// dot per entry is reduced inside the group and its weighted value per
// token is stored in contrib[(slot * rows + row) * NT + t]; after a bounded
// CTA barrier one thread per (row, token) adds the slots in order, so the
// result does not depend on timing.  NT >= ntok.
template <int FMT, int NT>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) down_flat_kernel(const EngineArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const MoeArgs &a = p.a;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);
  uint64_t *done = full + 1;
  float *hs_smem = reinterpret_cast<float *>(smem + p.hs_off);
  float *contrib = reinterpret_cast<float *>(smem + p.acc_off);
  const int nthreads = p.groups * p.tpr;
  const int nwarps = nthreads / 32;
  const int tid = threadIdx.x, lane = tid & 31;
  const int H = a.H, I = a.I;
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * H) / gridDim.x;
  const int nr = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * H) / gridDim.x - rb);  // <= tile_rows

  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(done, nwarps);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // h, routing and hmax come from the previous kernels

  if (tid >= nthreads) {
    // producer warp: every slot's rows of this CTA, one bulk copy each
    const int plane = tid - nthreads;
    const int nslots = __ldcg(a.meta + 1);
    SlotIds ids;
    ids.load(a, plane);
    const uint32_t bytes = static_cast<uint32_t>(nr * a.dn_row_bytes);
    if (plane == 0) mbar_arrive_expect_tx(full, bytes * static_cast<uint32_t>(nslots));
#pragma unroll 1
    for (int s = 0; s < nslots; ++s) {
      const int e = ids.get(s);
      const uint8_t *base = e >= 0 ? a.down + static_cast<int64_t>(e) * a.dn_stride : a.sh_down;
      if (plane == 0)
        bulk_g2s(smem + static_cast<uint32_t>(s) * p.stage_bytes, base + rb * a.dn_row_bytes, bytes, full);
    }
    return;
  }

  // consumers: routing metadata and all of h into shared memory
  Meta m(smem + p.meta_off, a.ntok, a.topk);
  const int nblk = I / 32;
  const int nh = a.ntok * (a.topk + 1);
  const int n4 = nh * I / 4;
  float4 hv[kHStage4];
  load_h(a, n4, tid, lane, nthreads, hv);
  load_meta(a, m, tid, nthreads);
  f2_t *pairs = reinterpret_cast<f2_t *>(hs_smem);
  float *hsum = hs_smem + static_cast<int64_t>(nh) * I;  // [nh][nblk]
  named_sync(1, nthreads);  // the h exponents are in m.expo
  stage_h<FMT>(hv, m, I, nblk, n4, tid, lane, nthreads, pairs, hsum);
  named_sync(1, nthreads);
  const int nslots = *m.nslots;

  const int g = tid / p.tpr, c = tid % p.tpr;
  const bool active = c < nblk;
  const int cb_bytes = FMT == EPQ_Q4_K ? p.tpr * 144 / 8 : p.tpr * Fmt<FMT>::kBlockBytes;
  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  XCol<1> xc;
  float xs[1] = {0.0f};
  if (!warp_wait(full, 0, a.err, DEVERR_FULL_WAIT, 0)) return;
  const int gps = max(1, p.groups / nslots);  // groups per slot (single-token path)
  const int rows_per = (nr + gps - 1) / gps;
  if (NT == 1 && nblk <= p.tpr && rows_per <= 8 && nslots <= p.groups) {
    // one token: group g takes rows part, part + gps, ... of slot g / gps;
    // the slot's h column is loaded once and the rows' dots are independent
    const int sl = g / gps, part = g - sl * gps;
    const bool grp_on = sl < nslots && active;
    const int k = grp_on ? (m.list[sl] & 31) : 0;
    float dv[8];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) dv[rr] = 0.0f;
    if (grp_on) {
#pragma unroll
      for (int i = 0; i < 16; ++i) xc.p[0][i] = pairs[(k * 16 + i) * nblk + c];
      xs[0] = hsum[k * nblk + c];
      const uint8_t *srow = smem + static_cast<uint32_t>(sl) * p.stage_bytes;
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = part + rr * gps;
        if (rr < rows_per && r < nr) {
          float pr[1] = {0.0f};
          column_dot<FMT, 1>(srow + static_cast<uint32_t>(r) * a.dn_row_bytes, cc, xc, xs, pr);
          dv[rr] = pr[0];
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      if (rr < rows_per) {
        float v = dv[rr];
        for (int o = p.tpr / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int r = part + rr * gps;
        if (grp_on && c == 0 && r < nr)
          contrib[sl * p.tile_rows + r] = (k < a.topk ? m.w[k] : m.gs[0]) * unscale(v, m.expo[k]);
      }
    }
  } else {
  const int npairs = nslots * nr;
  const int iters = (npairs + p.groups - 1) / p.groups;  // the same for every warp
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int pi = g + it * p.groups;
    const bool have = pi < npairs;
    const int s = have ? pi / nr : 0, r = have ? pi - s * nr : 0;
    const int ne = have ? m.cnt[s] : 0;
    const int ne_max = __reduce_max_sync(0xffffffffu, ne);  // uniform trip count for the shuffles
    float accp[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) accp[t] = 0.0f;
    const uint8_t *row = smem + static_cast<uint32_t>(s) * p.stage_bytes + static_cast<uint32_t>(r) * a.dn_row_bytes;
#pragma unroll 1
    for (int jj = 0; jj < ne_max; ++jj) {
      const bool on = jj < ne;
      const int ent = on ? m.list[s * a.ntok + jj] : 0;
      const int tok = ent >> 5, k = ent & 31;
      const int hsi = tok * (a.topk + 1) + k;
      float part = 0.0f;
      if (on && active) {
#pragma unroll 1
        for (int cb = c, ib = 0; cb < nblk; cb += p.tpr, ++ib) {
#pragma unroll
          for (int i = 0; i < 16; ++i) xc.p[0][i] = pairs[(hsi * 16 + i) * nblk + cb];
          xs[0] = hsum[hsi * nblk + cb];
          float pr[1] = {0.0f};
          column_dot<FMT, 1>(row + ib * cb_bytes, cc, xc, xs, pr);
          part += pr[0];
        }
      }
      for (int o = p.tpr / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (on) {
        const float v = (k < a.topk ? m.w[tok * a.topk + k] : m.gs[tok]) * unscale(part, m.expo[hsi]);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t == tok) accp[t] += v;
      }
    }
    if (have && c == 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t) contrib[(s * p.tile_rows + r) * NT + t] = accp[t];
    }
  }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(done);
  // y = x + sum over slots, one thread per (row, token), slots in order
  if (tid < ((nr * a.ntok + 31) & ~31)) {
    if (!warp_wait(done, 0, a.err, DEVERR_RED_WAIT, 0)) return;
    if (tid < nr * a.ntok) {
      const int r = tid / a.ntok, t = tid - r * a.ntok;
      float v = 0.0f;
#pragma unroll 1
      for (int s = 0; s < nslots; ++s) v += contrib[(s * p.tile_rows + r) * NT + t];
      const int64_t o = static_cast<int64_t>(t) * H + rb + r;
      a.y[o] = a.x[o] + v;
    }
  }
}

// block: consumers + the producer warp (+ the finisher warp when `fin`)
template <typename K>
cudaError_t launch_engine(K kernel, const EngineArgs &p, unsigned grid, uint32_t smem, cudaStream_t s, bool fin) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 block(p.groups * p.tpr + 32 + (fin ? 32 : 0));
  return launch_pdl(kernel, dim3(grid), block, smem, s, p);
}

template <int FMT>
cudaError_t launch_gateup(const EngineArgs &p, int rpg, unsigned grid, uint32_t smem, cudaStream_t s) {
  const bool fin = p.tpr > 32;
  switch (rpg) {
    case 2: return launch_engine(gateup_kernel<FMT, 2>, p, grid, smem, s, fin);
    case 4: return launch_engine(gateup_kernel<FMT, 4>, p, grid, smem, s, fin);
    case 8: return launch_engine(gateup_kernel<FMT, 8>, p, grid, smem, s, fin);
  }
  return cudaErrorInvalidValue;
}

// NT: token accumulators per thread (>= ntok); RPG * NT <= 32 registers
template <int FMT, int NT>
cudaError_t launch_down_nt(const EngineArgs &p, int rpg, unsigned grid, uint32_t smem, cudaStream_t s) {
  switch (rpg) {
    case 1: return launch_engine(down_kernel<FMT, 1, NT>, p, grid, smem, s, false);
    case 2: return launch_engine(down_kernel<FMT, 2, NT>, p, grid, smem, s, false);
    case 4: if (NT <= 8) return launch_engine(down_kernel<FMT, (NT <= 8 ? 4 : 1), NT>, p, grid, smem, s, false); break;
    case 8: if (NT <= 4) return launch_engine(down_kernel<FMT, (NT <= 4 ? 8 : 1), NT>, p, grid, smem, s, false); break;
  }
  return cudaErrorInvalidValue;
}

template <int FMT>
cudaError_t launch_gateup_flat(const EngineArgs &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  auto k = p.a.ntok <= 1 ? gateup_flat_kernel<FMT, 1> : gateup_flat_kernel<FMT, 4>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(p.groups * p.tpr), smem, s, p);  // consumers only
}

template <int FMT>
cudaError_t launch_down_flat(const EngineArgs &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  if (p.a.ntok <= 1) return launch_engine(down_flat_kernel<FMT, 1>, p, grid, smem, s, false);
  return launch_engine(down_flat_kernel<FMT, 4>, p, grid, smem, s, false);
}

template <int FMT>
cudaError_t launch_down(const EngineArgs &p, int rpg, unsigned grid, uint32_t smem, cudaStream_t s) {
  const int ntok = p.a.ntok;
  if (ntok <= 1) return launch_down_nt<FMT, 1>(p, rpg, grid, smem, s);
  if (ntok <= 4) return launch_down_nt<FMT, 4>(p, rpg, grid, smem, s);
  return launch_down_nt<FMT, kMaxTok>(p, rpg, grid, smem, s);
}

epq_status check_moe(const epq_router *r, const epq_experts *x, int ntok, int topk) {
  if (!r || !x) return EPQ_ERR_ARG;
  if (x->down_fmt_set != 0 && x->down_fmt_set != 1) return EPQ_ERR_ARG;
  const epq_fmt gf = x->fmt, df = x->down_fmt_set ? x->down_fmt : x->fmt;
  if (epq_block_weights(gf) < 0 || epq_block_weights(df) < 0) return EPQ_ERR_FORMAT;
  if (!r->weight || !x->gate_up || !x->down) return EPQ_ERR_ARG;
  if (r->n_experts < 1 || r->n_experts > kMaxExperts || x->n_experts != r->n_experts) return EPQ_ERR_ARG;
  if (ntok < 1 || ntok > kMaxTok || topk < 1 || topk > kMaxTopk || topk > r->n_experts) return EPQ_ERR_ARG;
  if (x->hidden < 256 || x->hidden > 16384 || x->hidden % 256) return EPQ_ERR_SHAPE;
  if (x->inter < 256 || x->inter > 16384 || x->inter % 256) return EPQ_ERR_SHAPE;
  if ((x->shared_gate_up == nullptr) != (x->shared_down == nullptr)) return EPQ_ERR_ARG;
  if (x->gate_up_stride < 0 || x->down_stride < 0 || x->gate_up_stride % 16 || x->down_stride % 16)
    return EPQ_ERR_ALIGN;
  const int64_t gu = 2ll * x->inter * epq_row_bytes(gf, x->hidden);
  const int64_t dn = static_cast<int64_t>(x->hidden) * epq_row_bytes(df, x->inter);
  if ((x->gate_up_stride && x->gate_up_stride < gu) || (x->down_stride && x->down_stride < dn)) return EPQ_ERR_ARG;
  if (!aligned16(r->weight) || !aligned16(x->gate_up) || !aligned16(x->down) ||
      (x->shared_gate_up && (!aligned16(x->shared_gate_up) || !aligned16(x->shared_down))) ||
      (x->shared_gate_vec && !aligned16(x->shared_gate_vec)))
    return EPQ_ERR_ALIGN;
  return EPQ_OK;
}

}  // namespace
}  // namespace epq

using namespace epq;

extern "C" size_t epq_moe_workspace_bytes(const epq_router *router, const epq_experts *experts, int ntok, int topk) {
  if (check_moe(router, experts, ntok, topk) != EPQ_OK) return 0;
  return ws_layout(ntok, topk, router->n_experts, experts->inter).total;
}

namespace {

// The routing buffers of a whole call, for the token chunks of its expert
// stages: the router ran once for every token; chunk t0.. reads its tokens'
// rows of the per-token buffers and reuses the per-call scratch (meta,
// active, cnt, list), which each chunk's gate/up kernel rewrites after its
// grid-dependency wait on the previous chunk's down kernel.
struct MoePre {
  float *logits, *xstat, *gshared, *w, *h;
  int32_t *idx, *meta, *active, *cnt, *list;
  uint32_t *hmax;
};

epq_status moe_forward_impl(const epq_router *router, const epq_experts *experts, const float *x, int ntok, int topk,
                            const epq_moe_opts *opts, float *y, int32_t *topk_idx, float *topk_w, void *workspace,
                            size_t workspace_bytes, epq_stream_t stream, const MoePre *pre);

}  // namespace

extern "C" epq_status epq_moe_forward(const epq_router *router, const epq_experts *experts, const float *x, int ntok,
                                      int topk, const epq_moe_opts *opts, float *y, int32_t *topk_idx, float *topk_w,
                                      void *workspace, size_t workspace_bytes, epq_stream_t stream) {
  return moe_forward_impl(router, experts, x, ntok, topk, opts, y, topk_idx, topk_w, workspace, workspace_bytes,
                          stream, nullptr);
}

namespace {

epq_status moe_forward_impl(const epq_router *router, const epq_experts *experts, const float *x, int ntok, int topk,
                            const epq_moe_opts *opts, float *y, int32_t *topk_idx, float *topk_w, void *workspace,
                            size_t workspace_bytes, epq_stream_t stream, const MoePre *pre) {
  epq_status st = check_moe(router, experts, ntok, topk);
  if (st != EPQ_OK) return st;
  if (!x || !y) return EPQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return EPQ_ERR_ALIGN;
  epq_moe_opts o = {};
  if (opts) o = *opts;
  if (o.rms_prenorm && !(o.rms_eps >= 0.0f)) return EPQ_ERR_ARG;
  if (o.h_out && !aligned16(o.h_out)) return EPQ_ERR_ALIGN;
  const int E = router->n_experts, H = experts->hidden, I = experts->inter;
  const WsLayout L = ws_layout(ntok, topk, E, I);
  if (!workspace || workspace_bytes < L.total) return EPQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EPQ_ERR_ALIGN;
  const epq_fmt gf = experts->fmt, df = experts->down_fmt_set ? experts->down_fmt : experts->fmt;
  // the k16 expert kernels: Q2_K / Q6_K stages, and Q4_K ones under engine 3
  // (measured in the chained layer: no faster than the ring kernels, which
  // stay the automatic choice for Q4_K experts)
  const int eng_t = tune_gemv_engine();
  const bool k16g = gf == EPQ_Q2_K || gf == EPQ_Q6_K || (eng_t == 3 && gf == EPQ_Q4_K);
  const bool k16d = df == EPQ_Q2_K || df == EPQ_Q6_K || (eng_t == 3 && df == EPQ_Q4_K);
  const bool whole = (o.stages & 7) == 0 || (o.stages & 7) == 7;
  // Tokens per pass of the Q2_K / Q6_K expert kernels: two when their
  // operands fit shared memory, else one.
  int k16_chunk = 0;
  if (k16g || k16d) {
    DeviceInfo dv;
    if (!current_device(&dv) || dv.major * 10 + dv.minor < 100) return EPQ_ERR_DEVICE;
    MoeArgs q = {};
    q.H = H;
    q.I = I;
    q.topk = topk;
    const int shared = experts->shared_gate_up != nullptr ? 1 : 0;
    for (int c = 2; c >= 1 && !k16_chunk; --c) {
      q.ntok = c;
      if (moe_k16_fits(q, std::min(E, c * topk) + shared, k16g, k16d, dv)) k16_chunk = c;
    }
    if (!k16_chunk) return EPQ_ERR_SHAPE;
    // stage calls with expert stages are not split into token chunks
    if (ntok > k16_chunk && !whole && (o.stages & (EPQ_MOE_GATE_UP | EPQ_MOE_DOWN))) return EPQ_ERR_SHAPE;
  }
  // Q4_K with three or more tokens, all stages in this call: the tensor-core
  // expert kernels take two tokens per pass, so the expert stages run as
  // chunks of two tokens (an expert chosen in two chunks is read once per
  // chunk) after ONE router launch for every token.  Measured faster than
  // the CUDA-core engines, which read every chosen expert once for all
  // tokens.  Calls with a Q2_K / Q6_K stage run as chunks of k16_chunk
  // tokens.
  const int chunk = k16_chunk ? k16_chunk : 2;
  if (!pre && ntok > chunk && whole &&
      (k16_chunk || (gf == EPQ_Q4_K && df == EPQ_Q4_K && tune_gemv_engine() != 1))) {
    epq_moe_opts orr = o;
    orr.stages = EPQ_MOE_ROUTE;
    st = moe_forward_impl(router, experts, x, ntok, topk, &orr, y, nullptr, nullptr, workspace, workspace_bytes,
                          stream, nullptr);
    if (st != EPQ_OK) return st;
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    const MoePre all{o.logits_out ? o.logits_out : reinterpret_cast<float *>(wsb + L.logits),
                     reinterpret_cast<float *>(wsb + L.xstat),
                     reinterpret_cast<float *>(wsb + L.gshared),
                     reinterpret_cast<float *>(wsb + L.w),
                     o.h_out ? o.h_out : reinterpret_cast<float *>(wsb + L.h),
                     reinterpret_cast<int32_t *>(wsb + L.idx),
                     reinterpret_cast<int32_t *>(wsb + L.meta),
                     reinterpret_cast<int32_t *>(wsb + L.active),
                     reinterpret_cast<int32_t *>(wsb + L.cnt),
                     reinterpret_cast<int32_t *>(wsb + L.list),
                     reinterpret_cast<uint32_t *>(wsb + L.hmax)};
    for (int t0 = 0; t0 < ntok; t0 += chunk) {
      const int nt = std::min(chunk, ntok - t0);
      epq_moe_opts oc = o;
      oc.stages = EPQ_MOE_GATE_UP | EPQ_MOE_DOWN;
      oc.logits_out = nullptr;
      oc.h_out = nullptr;
      MoePre pc = all;
      pc.logits += static_cast<int64_t>(t0) * E;
      pc.xstat += 2 * t0;
      pc.gshared += t0;
      pc.w += t0 * topk;
      pc.idx += t0 * topk;
      pc.h += static_cast<int64_t>(t0) * (topk + 1) * I;
      pc.hmax += t0 * (topk + 1);
      st = moe_forward_impl(router, experts, x + static_cast<int64_t>(t0) * H, nt, topk, &oc,
                            y + static_cast<int64_t>(t0) * H, topk_idx ? topk_idx + t0 * topk : nullptr,
                            topk_w ? topk_w + t0 * topk : nullptr, workspace, workspace_bytes, stream, &pc);
      if (st != EPQ_OK) return st;
    }
    return EPQ_OK;
  }
  DeviceInfo dev;
  if (!current_device(&dev) || dev.major * 10 + dev.minor < 100) return EPQ_ERR_DEVICE;
  unsigned *err = device_error_slot();
  if (!err) return EPQ_ERR_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);

  MoeArgs a = {};
  a.R = router->weight;
  a.bias = router->bias;
  a.gvec = experts->shared_gate_up ? experts->shared_gate_vec : nullptr;
  a.E = E;
  a.H = H;
  a.I = I;
  a.ntok = ntok;
  a.topk = topk;
  a.norm_topk = router->norm_topk;
  a.rms = o.rms_prenorm;
  a.eps = o.rms_eps;
  a.has_shared = experts->shared_gate_up != nullptr;
  a.gu_row_bytes = epq_row_bytes(gf, H);
  a.dn_row_bytes = epq_row_bytes(df, I);
  a.gate_up = static_cast<const uint8_t *>(experts->gate_up);
  a.gu_stride = experts->gate_up_stride ? experts->gate_up_stride : 2ll * I * a.gu_row_bytes;
  a.down = static_cast<const uint8_t *>(experts->down);
  a.dn_stride = experts->down_stride ? experts->down_stride : static_cast<int64_t>(H) * a.dn_row_bytes;
  a.sh_gate_up = static_cast<const uint8_t *>(experts->shared_gate_up);
  a.sh_down = static_cast<const uint8_t *>(experts->shared_down);
  a.x = x;
  a.y = y;
  a.out_idx = topk_idx;
  a.out_w = topk_w;
  a.logits = o.logits_out ? o.logits_out : reinterpret_cast<float *>(ws + L.logits);
  a.xstat = reinterpret_cast<float *>(ws + L.xstat);
  a.gshared = reinterpret_cast<float *>(ws + L.gshared);
  a.idx = reinterpret_cast<int32_t *>(ws + L.idx);
  a.w = reinterpret_cast<float *>(ws + L.w);
  a.meta = reinterpret_cast<int32_t *>(ws + L.meta);
  a.active = reinterpret_cast<int32_t *>(ws + L.active);
  a.cnt = reinterpret_cast<int32_t *>(ws + L.cnt);
  a.list = reinterpret_cast<int32_t *>(ws + L.list);
  a.hmax = reinterpret_cast<uint32_t *>(ws + L.hmax);
  a.h = o.h_out ? o.h_out : reinterpret_cast<float *>(ws + L.h);
  if (pre) {  // a token chunk of a routed call: the whole call's buffers
    a.logits = pre->logits;
    a.xstat = pre->xstat;
    a.gshared = pre->gshared;
    a.idx = pre->idx;
    a.w = pre->w;
    a.meta = pre->meta;
    a.active = pre->active;
    a.cnt = pre->cnt;
    a.list = pre->list;
    a.hmax = pre->hmax;
    a.h = pre->h;
  }
  a.err = err;

  const int stages = (o.stages & 7) ? (o.stages & 7) : 7;
  cudaError_t e = cudaSuccess;
  if (stages & EPQ_MOE_ROUTE) {
    const int nrows = E + (a.gvec ? 1 : 0);
    // staged form when every CTA's rows of R fit shared memory (one CTA per SM)
    const int sgrid = std::max(1, std::min(dev.sm_count, nrows));
    const int64_t srows = (nrows + sgrid - 1) / sgrid;
    // dynamic shared memory: the CTA's rows of R, then x of every token
    const int64_t sbytes = (srows + ntok) * H * 4;
    const uint32_t ssmem = static_cast<uint32_t>(sbytes);
    const bool staged = sbytes <= kRouterStageMax && (reinterpret_cast<uintptr_t>(a.R) & 15) == 0;
    if (staged) {
      auto launch = [&](auto k) {
        cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, ssmem);
        return r != cudaSuccess ? r : launch_pdl(k, dim3(sgrid), dim3(kRouterThreads), ssmem, s, a);
      };
      if (ntok <= 1) e = launch(router_kernel<1, true>);
      else if (ntok <= 4) e = launch(router_kernel<4, true>);
      else e = launch(router_kernel<kMaxTok, true>);
    } else {
      const unsigned rgrid = static_cast<unsigned>(
          std::max(1, std::min(2 * dev.sm_count, (nrows + kRouterWarps - 1) / kRouterWarps)));
      if (ntok <= 1) e = launch_pdl(router_kernel<1, false>, dim3(rgrid), dim3(kRouterThreads), 0, s, a);
      else if (ntok <= 4) e = launch_pdl(router_kernel<4, false>, dim3(rgrid), dim3(kRouterThreads), 0, s, a);
      else e = launch_pdl(router_kernel<kMaxTok, false>, dim3(rgrid), dim3(kRouterThreads), 0, s, a);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if (!(stages & EPQ_MOE_GATE_UP) && (topk_idx || topk_w || (stages & EPQ_MOE_DOWN))) {
      // the gate/up kernel routes for itself; without it, route here when
      // this call returns the selection or runs the down stage
      const uint32_t sel_smem = ((4u * meta_words(ntok, topk) + 15u) & ~15u) + 4u * kSelScratchWords;
      e = launch_pdl(select_kernel, dim3(1), dim3(kSelectThreads), sel_smem, s, a);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }

  const int max_slots = std::min(E, ntok * topk) + (a.has_shared ? 1 : 0);
  // Engines per stage: Q2_K / Q6_K matrices run the k16 kernels (moe_k16.cu);
  // Q4_K with one or two tokens the tensor-core kernels (moe_tc.cu) unless
  // the CUDA-core engines are forced; everything else the CUDA-core kernels
  // below.  A CUDA-core down kernel reads the max |h| words, which the
  // tensor-core gate/up kernel does not keep: that pairing runs the
  // CUDA-core gate/up.
  enum { kCC = 0, kTC = 1, kK16 = 2 };
  MoeTcPlan tp;
  const bool tc_ok = tune_gemv_engine() != 1 && (gf == EPQ_Q4_K || df == EPQ_Q4_K) && !(k16g && k16d) &&
                     moe_tc_plan(a, max_slots, dev, &tp);
  const int d_eng = k16d ? kK16 : (df == EPQ_Q4_K && tc_ok ? kTC : kCC);
  int g_eng = k16g ? kK16 : (gf == EPQ_Q4_K && tc_ok ? kTC : kCC);
  if (g_eng == kTC && d_eng == kCC) g_eng = kCC;
  if ((g_eng == kK16 || d_eng == kK16) && ntok > 2 && (stages & (EPQ_MOE_GATE_UP | EPQ_MOE_DOWN)))
    return EPQ_ERR_SHAPE;

  if (stages & EPQ_MOE_GATE_UP) {
    if (g_eng == kK16) {
      e = moe_k16_gateup_launch(gf, a, max_slots, d_eng == kCC, dev, s);
      if (e != cudaSuccess) return cuda_fail(e);
    } else if (g_eng == kTC) {
      e = moe_tc_gateup_launch(tp, a, s);
      if (e != cudaSuccess) return cuda_fail(e);
    } else {
      EnginePlan gp;
      const unsigned ggrid = static_cast<unsigned>(dev.sm_count);
      const int64_t g_hint = (static_cast<int64_t>(max_slots) * I + ggrid - 1) / ggrid;
      const bool gflat = flat_gateup_plan(H, a.gu_row_bytes, I, ggrid, max_slots, ntok, topk, dev, &gp);
      if (!gflat && !engine_plan(H, 2 * a.gu_row_bytes, true, g_hint, ntok, topk, I, false, dev, &gp))
        return EPQ_ERR_SHAPE;
      // the gate/up kernel routes in its stage area before the first copy
      if (static_cast<int64_t>(gp.stages) * gp.stage_bytes < 4ll * kSelScratchWords) return EPQ_ERR_SHAPE;
      EngineArgs ga{a, gp.tpr, gp.groups, gp.tile_rows, gp.stages, gp.stage_h, gp.stage_bytes, gp.bar_off,
                    gp.red_off, gp.meta_off, gp.hs_off, gp.acc_off};
      if (gflat) switch (gf) {
        case EPQ_Q8_0: e = launch_gateup_flat<EPQ_Q8_0>(ga, ggrid, gp.smem, s); break;
        case EPQ_Q4_0: e = launch_gateup_flat<EPQ_Q4_0>(ga, ggrid, gp.smem, s); break;
        case EPQ_Q4_1: e = launch_gateup_flat<EPQ_Q4_1>(ga, ggrid, gp.smem, s); break;
        case EPQ_Q4_K: e = launch_gateup_flat<EPQ_Q4_K>(ga, ggrid, gp.smem, s); break;
        default: return EPQ_ERR_FORMAT;
      }
      else switch (gf) {
        case EPQ_Q8_0: e = launch_gateup<EPQ_Q8_0>(ga, gp.rpg, ggrid, gp.smem, s); break;
        case EPQ_Q4_0: e = launch_gateup<EPQ_Q4_0>(ga, gp.rpg, ggrid, gp.smem, s); break;
        case EPQ_Q4_1: e = launch_gateup<EPQ_Q4_1>(ga, gp.rpg, ggrid, gp.smem, s); break;
        case EPQ_Q4_K: e = launch_gateup<EPQ_Q4_K>(ga, gp.rpg, ggrid, gp.smem, s); break;
        default: return EPQ_ERR_FORMAT;
      }
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }

  if (stages & EPQ_MOE_DOWN) {
    if (d_eng == kK16) {
      e = moe_k16_down_launch(df, a, max_slots, dev, s);
      if (e != cudaSuccess) return cuda_fail(e);
    } else if (d_eng == kTC) {
      e = moe_tc_down_launch(tp, a, s);
      if (e != cudaSuccess) return cuda_fail(e);
    } else {
      EnginePlan dp;
      const unsigned dgrid = static_cast<unsigned>(std::max(1, std::min(dev.sm_count, (H + 7) / 8)));
      const int64_t d_hint = (H + dgrid - 1) / dgrid;
      const bool flat = flat_down_plan(I, a.dn_row_bytes, H, dgrid, max_slots, ntok, topk, dev, &dp);
      if (!flat && !engine_plan(I, a.dn_row_bytes, false, d_hint, ntok, topk, I, true, dev, &dp))
        return EPQ_ERR_SHAPE;
      EngineArgs da{a, dp.tpr, dp.groups, dp.tile_rows, dp.stages, dp.stage_h, dp.stage_bytes, dp.bar_off,
                    dp.red_off, dp.meta_off, dp.hs_off, dp.acc_off};
      if (flat) switch (df) {
        case EPQ_Q8_0: e = launch_down_flat<EPQ_Q8_0>(da, dgrid, dp.smem, s); break;
        case EPQ_Q4_0: e = launch_down_flat<EPQ_Q4_0>(da, dgrid, dp.smem, s); break;
        case EPQ_Q4_1: e = launch_down_flat<EPQ_Q4_1>(da, dgrid, dp.smem, s); break;
        case EPQ_Q4_K: e = launch_down_flat<EPQ_Q4_K>(da, dgrid, dp.smem, s); break;
        default: return EPQ_ERR_FORMAT;
      }
      else switch (df) {
        case EPQ_Q8_0: e = launch_down<EPQ_Q8_0>(da, dp.rpg, dgrid, dp.smem, s); break;
        case EPQ_Q4_0: e = launch_down<EPQ_Q4_0>(da, dp.rpg, dgrid, dp.smem, s); break;
        case EPQ_Q4_1: e = launch_down<EPQ_Q4_1>(da, dp.rpg, dgrid, dp.smem, s); break;
        case EPQ_Q4_K: e = launch_down<EPQ_Q4_K>(da, dp.rpg, dgrid, dp.smem, s); break;
        default: return EPQ_ERR_FORMAT;
      }
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  return EPQ_OK;
}

}  // namespace

// ------------------------------------------------------------------ fixed-scratch variant
// A copy of the MoE workspace that lives in a file-scope device array instead
// of caller memory, for callers that cannot allocate device memory.  Every
// GPU that loads the library holds these bytes until the process exits.
namespace {
constexpr size_t kFixedScratchBytes = size_t(1) << 20;  // 1 MiB
__device__ __align__(256) uint8_t g_moe_fixed_scratch[kFixedScratchBytes];

std::mutex g_fixed_mu;
void *g_fixed_ptr[64] = {};

// Device address of the fixed scratch on the current device.  The host-side
// name of the array is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
epq_status fixed_scratch_ptr(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return EPQ_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_fixed_mu);
  if (!g_fixed_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_fixed_scratch);
    if (e != cudaSuccess || !p) {
      // clear the runtime's sticky last-error slot, so that the next launch
      // of any entry point does not report this failed lookup as its own
      cudaGetLastError();
      return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    }
    g_fixed_ptr[dev] = p;
  }
  *out = g_fixed_ptr[dev];
  return EPQ_OK;
}
}  // namespace

extern "C" epq_status epq_moe_forward_noalloc(const epq_router *router, const epq_experts *experts, const float *x,
                                              int ntok, int topk, const epq_moe_opts *opts, float *y,
                                              int32_t *topk_idx, float *topk_w, epq_stream_t stream) {
  const epq_status st = check_moe(router, experts, ntok, topk);
  if (st != EPQ_OK) return st;
  const size_t need = ws_layout(ntok, topk, router->n_experts, experts->inter).total;
  if (need > kFixedScratchBytes) return EPQ_ERR_WORKSPACE;
  void *ws = nullptr;
  const epq_status sp = fixed_scratch_ptr(&ws);
  if (sp != EPQ_OK) return sp;
  return epq_moe_forward(router, experts, x, ntok, topk, opts, y, topk_idx, topk_w, ws, kFixedScratchBytes, stream);
}

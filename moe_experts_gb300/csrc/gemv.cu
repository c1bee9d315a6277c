// Dense dequant-GEMV (epq_gemv / epq_gemv_ex).
//
// "端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch", section "速度上限：带宽 ÷
// 权重字节数": batch-1 decode reads every weight once per token, so the
// kernel is a pure HBM stream and its bound is bandwidth / packed bytes.
//
// Layout of one launch (persistent, one CTA per SM):
//   * CTA b owns output rows [b*R/G, (b+1)*R/G) and walks them in tiles of
//     TR rows.  A tile is TR whole packed rows, contiguous in HBM, moved into
//     shared memory by ONE cp.async.bulk (the TMA engine) issued by a
//     producer warp; a ring of `stages` tiles keeps ~100+ KB in flight per SM.
//   * NT = groups * tpr consumer threads.  Thread c of a row group owns
//     block column c (see gemv_core.cuh) and holds its 32 activations in
//     registers; group g computes rows g*RPG .. g*RPG+RPG-1 of every tile.
//   * Per tile each thread produces RPG partial sums; a butterfly
//     reduce-scatter over the group's lanes (and, for groups wider than a
//     warp, a shared-memory pass guarded by an mbarrier) yields the rows.
//   * Every wait is bounded (see common.cuh); no __syncthreads after setup.
#include <algorithm>

#include "gemv_core.cuh"
#include "gemv_tc.cuh"

namespace epq {
namespace {

constexpr int kMaxConsumers = 512;
constexpr int kRedRing = 8;              // reduction buffers in flight

struct GemvParams {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows_out;    // output rows
  int64_t up_rows;     // swiglu: row distance gate -> up (= rows_out); 0 otherwise
  int64_t row_bytes;
  int cols;            // weights per row
  int nblk;            // cols / 32
  int tpr;             // threads per row group (>= nblk)
  int groups;          // row groups per CTA
  int teams;           // independent consumer teams (each takes every teams-th tile)
  int gpt;             // row groups per team (1 when tpr >= 32, else 32 / tpr)
  int tile_rows;       // output rows per tile (= gpt * RPG, or gpt * RPG/2 with swiglu)
  int red_rows;        // partial rows per tile (= gpt * RPG)
  int stages;
  uint32_t stage_bytes;
  int nv;              // vectors in this launch (<= NV template)
  int64_t x_stride;    // floats between vectors of x
  int64_t y_stride;    // floats between vectors of y / residual
  int rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early_weights;   // weights are ready: stream them before the PDL wait
  int xstage;          // x is staged once per CTA in shared memory (coalesced)
  unsigned *err;
};

struct SmemLayout {
  uint32_t full_off, empty_off, rfull_off, rempty_off, red_off, scratch_off, xs_off, total;
};

// x staging: 32-float columns padded to 36 floats, so that a thread reading
// its own column with 16-byte loads never shares a bank with its neighbours.
constexpr int kXPad = 36;

__host__ __device__ inline int wpg_of(int tpr) { return tpr > 32 ? tpr / 32 : 1; }

__host__ __device__ inline SmemLayout smem_layout(int stages, uint32_t stage_bytes, int nv, int red_rows, int tpr,
                                                  int nthreads, int xstage_cols = 0) {
  SmemLayout L;
  uint32_t o = static_cast<uint32_t>(stages) * stage_bytes + 16;  // +16: code-word over-read pad
  o = (o + 15u) & ~15u;
  L.full_off = o;
  o += 8u * stages;
  L.empty_off = o;
  o += 8u * stages;
  L.rfull_off = o;
  o += 8u * kRedRing;
  L.rempty_off = o;
  o += 8u * kRedRing;
  L.red_off = o;
  o += 4u * kRedRing * nv * red_rows * wpg_of(tpr);
  o = (o + 15u) & ~15u;
  L.scratch_off = o;
  o += 4u * 2 * nv * (nthreads / 32);
  o = (o + 15u) & ~15u;
  L.xs_off = o;
  o += 4u * nv * (xstage_cols / 32) * kXPad;
  L.total = (o + 15u) & ~15u;
  return L;
}

// Output epilogue for one row of one vector.
__device__ __forceinline__ void store_row(const GemvParams &p, int v, int64_t orow, float val) {
  if (p.residual) val += p.residual[v * p.y_stride + orow];
  p.y[v * p.y_stride + orow] = val;
}

template <int FMT, int NV, int RPG, bool SWIGLU>
__global__ void __launch_bounds__(kMaxConsumers + 64, 1) gemv_kernel(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nthreads = p.groups * p.tpr;
  const int nwarps = nthreads / 32;
  const bool has_fin = p.tpr > 32;   // cross-warp rows go through the finisher warp
  const int wpg = wpg_of(p.tpr);
  const SmemLayout L = smem_layout(p.stages, p.stage_bytes, NV, p.red_rows, p.tpr, nthreads, p.xstage ? p.cols : 0);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full_off);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty_off);
  uint64_t *rfull = reinterpret_cast<uint64_t *>(smem + L.rfull_off);
  uint64_t *rempty = reinterpret_cast<uint64_t *>(smem + L.rempty_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  float *scratch = reinterpret_cast<float *>(smem + L.scratch_off);
  const int tid = threadIdx.x;
  const int lane = tid & 31;

  // rows of this CTA
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * p.rows_out) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * p.rows_out) / gridDim.x;
  const int ntiles = static_cast<int>((re - rb + p.tile_rows - 1) / p.tile_rows);
  const int red_stride = NV * p.red_rows * wpg;   // floats per reduction buffer

  const int team_warps = nwarps / p.teams;
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], team_warps);
    }
    for (int b = 0; b < kRedRing; ++b) {
      mbar_init(&rfull[b], team_warps);
      mbar_init(&rempty[b], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  // ------------------------------------------------------------------ producer
  if (tid >= nthreads && tid < nthreads + 32) {
    if (tid != nthreads) return;
    if (!p.early_weights) pdl_wait();
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % p.stages;
      if (t >= p.stages && !mbar_wait(&empty[s], ((t / p.stages) - 1) & 1, p.err, DEVERR_EMPTY_WAIT, t)) {
        ok = false;
        break;
      }
      const int64_t r0 = rb + static_cast<int64_t>(t) * p.tile_rows;
      const int64_t nr = min(static_cast<int64_t>(p.tile_rows), re - r0);
      const uint32_t bytes = static_cast<uint32_t>(nr * p.row_bytes);
      uint8_t *dst = smem + static_cast<uint32_t>(s) * p.stage_bytes;
      if (SWIGLU) {
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        bulk_g2s(dst, p.W + r0 * p.row_bytes, bytes, &full[s]);
        bulk_g2s(dst + p.tile_rows * p.row_bytes, p.W + (p.up_rows + r0) * p.row_bytes, bytes, &full[s]);
      } else {
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(dst, p.W + r0 * p.row_bytes, bytes, &full[s]);
      }
      ++issued;
    }
    if (!ok) {
      // drain: wait (bounded) for every copy still in flight before leaving
      for (int t = max(0, issued - p.stages); t < issued; ++t)
        mbar_wait(&full[t % p.stages], (t / p.stages) & 1, p.err, DEVERR_DRAIN_WAIT, t);
    }
    return;
  }

  // ------------------------------------------------------------------ prologue
  // consumers load their activation column; everyone (consumers + finisher)
  // learns the per-vector exponent and RMS factor.
  const bool is_fin = tid >= nthreads + 32;
  const int g = tid / p.tpr;
  const int c = tid % p.tpr;
  const bool active = !is_fin && c < p.nblk;
  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  const XGather xg{p.x_group, p.x_head_dim};
  pdl_wait();  // x and the residual are produced upstream

  float xr[NV][32];
  float xsum[NV];
  XCol<NV> xc;
  float *xs = reinterpret_cast<float *>(smem + L.xs_off);
  if (p.xstage) {
    // coalesced, once per CTA: consumer threads copy (gathered) x into the
    // padded staging area and take per-vector max |x| and sum x^2 as they go
    const int c4 = p.cols / 4;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float amax = 0.0f, ssq = 0.0f;
      if (!is_fin && v < p.nv) {
        for (int e4 = tid; e4 < c4; e4 += nthreads) {
          const int j = 4 * e4;
          const float4 q4 = *reinterpret_cast<const float4 *>(p.x + v * p.x_stride + xg.src(j));
          *reinterpret_cast<float4 *>(xs + (v * p.nblk + j / 32) * kXPad + (j & 31)) = q4;
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q4.x), fabsf(q4.y)), fmaxf(fabsf(q4.z), fabsf(q4.w))));
          ssq = fmaf(q4.x, q4.x, fmaf(q4.y, q4.y, fmaf(q4.z, q4.z, fmaf(q4.w, q4.w, ssq))));
        }
      }
      if (!is_fin) {
        amax = warp_max_all(amax);
        ssq = warp_sum_xor<32>(ssq);
        if (lane == 0) {
          scratch[(2 * v) * nwarps + (tid >> 5)] = amax;
          scratch[(2 * v + 1) * nwarps + (tid >> 5)] = ssq;
        }
      }
    }
  } else {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float amax = 0.0f, ssq = 0.0f;
      const bool vv = v < p.nv && active;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (vv) q4 = *reinterpret_cast<const float4 *>(p.x + v * p.x_stride + xg.src(32 * c + j));
        xr[v][j] = q4.x;
        xr[v][j + 1] = q4.y;
        xr[v][j + 2] = q4.z;
        xr[v][j + 3] = q4.w;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        amax = fmaxf(amax, fabsf(xr[v][j]));
        if (g == 0) ssq = fmaf(xr[v][j], xr[v][j], ssq);
      }
      if (!is_fin) {
        amax = warp_max_all(amax);
        ssq = warp_sum_xor<32>(ssq);
        if (lane == 0) {
          scratch[(2 * v) * nwarps + (tid >> 5)] = amax;
          scratch[(2 * v + 1) * nwarps + (tid >> 5)] = ssq;
        }
      }
    }
  }
  named_sync(1, nthreads + (has_fin ? 32 : 0));
  int expo[NV];
  float outscale[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    float a = 0.0f, q = 0.0f;
    for (int w = 0; w < nwarps; ++w) {
      a = fmaxf(a, scratch[(2 * v) * nwarps + w]);
      q += scratch[(2 * v + 1) * nwarps + w];
    }
    // |x| < 2^E; activations are stored as x * 2^(126 - E - shift) so that
    // every product lands at scale 2^(-23 - E).
    const int E = bound_exponent(a);
    expo[v] = E;
    if (p.xstage) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active && v < p.nv) q4 = *reinterpret_cast<const float4 *>(xs + (v * p.nblk + c) * kXPad + j);
        xr[v][j] = q4.x;
        xr[v][j + 1] = q4.y;
        xr[v][j + 2] = q4.z;
        xr[v][j + 3] = q4.w;
      }
    }
    xsum[v] = scale_column<FMT>(xr[v], E, xc.p[v]);
    float r = 1.0f;
    if (p.rms) r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, static_cast<float>(p.cols)), p.rms_eps)));
    outscale[v] = r;
  }
  constexpr int RH = SWIGLU ? RPG / 2 : RPG;  // gate rows per group (swiglu)

  // ------------------------------------------------------------------ finisher
  if (is_fin) {
    for (int t = 0; t < ntiles; ++t) {
      const int b = t % kRedRing;
      if (!warp_wait(&rfull[b], (t / kRedRing) & 1, p.err, DEVERR_RED_WAIT, t)) return;
      const float *rbuf = red + b * red_stride;
      const int64_t r0 = rb + static_cast<int64_t>(t) * p.tile_rows;
      const int nr = static_cast<int>(min(static_cast<int64_t>(p.tile_rows), re - r0));
      for (int o = lane; o < nr; o += 32) {
        const int gg = o / RH, k = o % RH;
        for (int v = 0; v < p.nv && v < NV; ++v) {
          const float *slot = rbuf + (v * p.red_rows + gg * RPG + k) * wpg;
          float acc = 0.0f;
          for (int w = 0; w < wpg; ++w) acc += slot[w];
          float val = unscale(acc, expo[v]) * outscale[v];
          if (SWIGLU) {
            const float *us = slot + RH * wpg;
            float ua = 0.0f;
            for (int w = 0; w < wpg; ++w) ua += us[w];
            val = silu(val) * (unscale(ua, expo[v]) * outscale[v]);
          }
          store_row(p, v, r0 + o, val);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[b]);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int W = p.tpr < 32 ? p.tpr : 32;
  const int wg = c >> 5;
  const int team_size = nthreads / p.teams;
  const int team = tid / team_size;
  const int gt = g % p.gpt;  // group index within the team (row block of the tile)
  // stages % teams == 0 (see make_plan): the stages this team waits on are its own
  for (int t = team; t < ntiles; t += p.teams) {
    const int s = t % p.stages;
    if (!warp_wait(&full[s], (t / p.stages) & 1, p.err, DEVERR_FULL_WAIT, t)) return;
    const uint8_t *base = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    const int64_t r0 = rb + static_cast<int64_t>(t) * p.tile_rows;
    const int nr = static_cast<int>(min(static_cast<int64_t>(p.tile_rows), re - r0));
    float part[NV][RPG];
#pragma unroll
    for (int k = 0; k < RPG; ++k) {
      const int lr = SWIGLU ? (gt * RH + (k % RH)) : (gt * RPG + k);
      float pr[NV];
      if (active && lr < nr) {
        const uint8_t *row = base + static_cast<uint32_t>(lr) * p.row_bytes;
        if (SWIGLU && k >= RH) row += p.tile_rows * p.row_bytes;
        column_dot<FMT, NV>(row, cc, xc, xsum, pr);
      } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) pr[v] = 0.0f;
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) part[v][k] = pr[v];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    const int ri = reduce_scatter<RPG, NV>(part, W, lane % W);
    if (has_fin) {
      // hand the warp's row partials to the finisher through the ring (one
      // buffer per tile, in tile order)
      const int b = t % kRedRing;
      if (t >= kRedRing && !warp_wait(&rempty[b], ((t / kRedRing) - 1) & 1, p.err, DEVERR_RED_WAIT, t)) return;
      float *rbuf = red + b * red_stride;
      if ((lane % (32 / RPG)) == 0) {
#pragma unroll
        for (int v = 0; v < NV; ++v) rbuf[(v * p.red_rows + gt * RPG + ri) * wpg + wg] = part[v][0];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[b]);
    } else {
      // the whole row lives in this warp: the first lane of each run finishes it
      float up[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) up[v] = SWIGLU ? __shfl_xor_sync(0xffffffffu, part[v][0], W / 2) : 0.0f;
      const bool holder = ((lane % W) % (W / RPG)) == 0;
      if (holder && (!SWIGLU || ri < RH)) {
        const int lr = SWIGLU ? gt * RH + ri : gt * RPG + ri;
        if (lr < nr) {
          for (int v = 0; v < p.nv && v < NV; ++v) {
            float val = unscale(part[v][0], expo[v]) * outscale[v];
            if (SWIGLU) val = silu(val) * (unscale(up[v], expo[v]) * outscale[v]);
            store_row(p, v, r0 + lr, val);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ one-shot form
// One vector, and a CTA's whole row range fits shared memory at once
// (decode projections).  The producer stages the rows with one bulk copy
// (two with SwiGLU: the gate rows and the up rows) on a single barrier,
// before the grid-dependency wait when the weights are ready; the consumers
// take max|x| and sum x^2 (RMS pre-norm), stage x in scaled pairs once, and
// then row group g computes rows g, g + groups, ... over its column blocks
// (c, c + tpr, ...; tpr <= 32, so a row is reduced inside its warp).
constexpr int kFlatMaxX4 = 8;  // float4 of x per thread kept in registers between the passes

template <int FMT, bool SWIGLU>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) gemv_flat_kernel(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nthreads = p.groups * p.tpr;
  const int nwarps = nthreads / 32;
  const int tid = threadIdx.x, lane = tid & 31;
  const int nblk = p.nblk;
  // layout: rows (gate, then up) | 16-byte over-read pad | barrier | scratch | x pairs | x column sums
  const uint32_t rows_bytes = static_cast<uint32_t>(p.tile_rows * p.row_bytes);
  uint8_t *gate_s = smem;
  uint8_t *up_s = smem + rows_bytes;
  uint32_t o = (SWIGLU ? 2u : 1u) * rows_bytes + 16u;
  o = (o + 15u) & ~15u;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + o);
  float *scratch = reinterpret_cast<float *>(smem + o + 16);  // [2][nwarps]
  f2_t *xp = reinterpret_cast<f2_t *>(smem + ((o + 16 + 8u * nwarps + 15u) & ~15u));  // [16][nblk]
  float *xsum = reinterpret_cast<float *>(xp + 16 * nblk);                                // [nblk]

  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * p.rows_out) / gridDim.x;
  const int nr = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * p.rows_out) / gridDim.x - rb);

  if (tid == 0) {
    mbar_init(full, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (tid >= nthreads) {
    if (tid == nthreads && nr > 0) {
      if (!p.early_weights) pdl_wait();
      const uint32_t bytes = static_cast<uint32_t>(nr * p.row_bytes);
      mbar_arrive_expect_tx(full, SWIGLU ? 2 * bytes : bytes);
      bulk_g2s(gate_s, p.W + rb * p.row_bytes, bytes, full);
      if (SWIGLU) bulk_g2s(up_s, p.W + (p.up_rows + rb) * p.row_bytes, bytes, full);
    }
    return;
  }

  pdl_wait();  // x and the residual are produced upstream
  // pass 1: max|x| and sum x^2 (x kept in registers for pass 2)
  const XGather xg{p.x_group, p.x_head_dim};
  const int c4 = p.cols / 4;
  float4 xv[kFlatMaxX4];
  float amax = 0.0f, ssq = 0.0f;
#pragma unroll
  for (int k = 0; k < kFlatMaxX4; ++k) {
    const int e4 = (tid - lane) + k * nthreads + lane;
    xv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e4 < c4) {
      xv[k] = *reinterpret_cast<const float4 *>(p.x + xg.src(4 * e4));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(xv[k].x), fabsf(xv[k].y)), fmaxf(fabsf(xv[k].z), fabsf(xv[k].w))));
      ssq = fmaf(xv[k].x, xv[k].x, fmaf(xv[k].y, xv[k].y, fmaf(xv[k].z, xv[k].z, fmaf(xv[k].w, xv[k].w, ssq))));
    }
  }
  amax = warp_max_all(amax);
  ssq = warp_sum_xor<32>(ssq);
  if (lane == 0) {
    scratch[tid >> 5] = amax;
    scratch[nwarps + (tid >> 5)] = ssq;
  }
  named_sync(1, nthreads);
  float am = 0.0f, q = 0.0f;
  for (int w = 0; w < nwarps; ++w) {
    am = fmaxf(am, scratch[w]);
    q += scratch[nwarps + w];
  }
  const int E = bound_exponent(am);
  const float outscale =
      p.rms ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, static_cast<float>(p.cols)), p.rms_eps))) : 1.0f;
  // pass 2: scaled pairs; 8 consecutive threads hold one 32-float column
#pragma unroll
  for (int k = 0; k < kFlatMaxX4; ++k) {
    const int e4 = (tid - lane) + k * nthreads + lane;
    if ((tid - lane) + k * nthreads < c4) {  // warp-uniform
      const float4 v = xv[k];
      const int j = (4 * e4) & 31, col = (4 * e4) >> 5;
      float sum = (v.x + v.y) + (v.z + v.w);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      if (e4 < c4) {
        const int base = (j / 2) * nblk + col;
        xp[base] = f2_pack(scale_pow2(v.x, 126 - E - Fmt<FMT>::shift(j)),
                           scale_pow2(v.y, 126 - E - Fmt<FMT>::shift(j + 1)));
        xp[base + nblk] = f2_pack(scale_pow2(v.z, 126 - E - Fmt<FMT>::shift(j + 2)),
                                  scale_pow2(v.w, 126 - E - Fmt<FMT>::shift(j + 3)));
        if (j == 0) xsum[col] = scale_pow2(sum, -23 - E);
      }
    }
  }
  named_sync(1, nthreads);

  const int g = tid / p.tpr, c = tid % p.tpr;
  const bool active = c < nblk;
  const int cb_bytes = FMT == EPQ_Q4_K ? p.tpr * 144 / 8 : p.tpr * Fmt<FMT>::kBlockBytes;
  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  XCol<1> xc;
  float xs[1] = {0.0f};
  if (nr > 0 && !warp_wait(full, 0, p.err, DEVERR_FULL_WAIT, 0)) return;
  const int iters = (nr + p.groups - 1) / p.groups;  // the same for every warp
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int v = g + it * p.groups;
    const bool have = v < nr && active;
    float pg = 0.0f, pu = 0.0f;
    if (have) {
      const uint8_t *grow = gate_s + static_cast<uint32_t>(v) * p.row_bytes;
      const uint8_t *urow = up_s + static_cast<uint32_t>(v) * p.row_bytes;
#pragma unroll 1
      for (int cb = c, ib = 0; cb < nblk; cb += p.tpr, ++ib) {
#pragma unroll
        for (int i = 0; i < 16; ++i) xc.p[0][i] = xp[i * nblk + cb];
        xs[0] = xsum[cb];
        float pr[1] = {0.0f};
        column_dot<FMT, 1>(grow + ib * cb_bytes, cc, xc, xs, pr);
        pg += pr[0];
        if (SWIGLU) {
          pr[0] = 0.0f;
          column_dot<FMT, 1>(urow + ib * cb_bytes, cc, xc, xs, pr);
          pu += pr[0];
        }
      }
    }
    for (int off = p.tpr / 2; off > 0; off >>= 1) {
      pg += __shfl_xor_sync(0xffffffffu, pg, off);
      if (SWIGLU) pu += __shfl_xor_sync(0xffffffffu, pu, off);
    }
    if (c == 0 && v < nr) {
      float val = unscale(pg, E) * outscale;
      if (SWIGLU) val = silu(val) * (unscale(pu, E) * outscale);
      store_row(p, 0, rb + v, val);
    }
  }
}

// ------------------------------------------------------------------ host
struct Plan {
  int tpr, groups, gpt, teams, rpg, tile_rows, stages, xstage;
  uint32_t stage_bytes, smem;
  unsigned grid;
};

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

bool make_plan(int64_t row_bytes, int cols, int64_t rows_out, bool swiglu, int nv, const DeviceInfo &dev,
               Plan *pl) {
  const int nblk = cols / 32;
  pl->tpr = nblk <= 32 ? std::max(8, next_pow2(nblk)) : ((nblk + 31) / 32) * 32;
  if (pl->tpr > kMaxConsumers) return false;
  pl->groups = std::max(1, kMaxConsumers / pl->tpr);
  int64_t g = std::min<int64_t>(dev.sm_count, (rows_out + 7) / 8);
  pl->grid = static_cast<unsigned>(std::max<int64_t>(1, g));
  const int64_t rows_per_cta = (rows_out + pl->grid - 1) / pl->grid;
  const int rmax = std::min(8, std::min(pl->tpr, 32));
  const int64_t per_row = row_bytes * (swiglu ? 2 : 1);
  const int64_t tile_target = tune_tile_bytes(), ring_target = tune_ring_bytes();
  const int min_gpt = pl->tpr >= 32 ? 1 : 32 / pl->tpr;  // a team is whole warps
  const int nthreads = pl->groups * pl->tpr;
  // Pick (groups per team, rows per group): the bulk copy of one tile must be
  // large (the TMA engine has a per-copy cost: below ~32 KB it cannot keep
  // HBM busy), every team should get >= 2 tiles, and more teams are better
  // (they overlap each other's latency).  Score = copy size capped at the
  // target, then teams.
  int best_gpt = pl->groups, best_rpg = swiglu ? 2 : 1;
  int64_t best_score = -1;
  for (int gpt = min_gpt; gpt <= pl->groups; gpt *= 2) {
    if (pl->groups % gpt) continue;
    const int teams = pl->groups / gpt;
    for (int rpg = swiglu ? 2 : 1; rpg <= rmax; rpg *= 2) {
      const int64_t tile_rows = static_cast<int64_t>(gpt) * (swiglu ? rpg / 2 : rpg);
      const int64_t bytes = tile_rows * per_row;
      if (bytes > 2 * tile_target && rpg > (swiglu ? 2 : 1)) continue;
      const bool two_each = tile_rows * 2 * teams <= rows_per_cta;
      const int64_t eff = std::min(bytes, tile_target);
      const int64_t score = (two_each ? (int64_t(1) << 40) : 0) + eff * 64 + teams;
      if (score > best_score) {
        best_score = score;
        best_gpt = gpt;
        best_rpg = rpg;
      }
    }
  }
  pl->gpt = best_gpt;
  pl->teams = pl->groups / best_gpt;
  pl->rpg = best_rpg;
  pl->tile_rows = static_cast<int>(static_cast<int64_t>(best_gpt) * (swiglu ? best_rpg / 2 : best_rpg));
  pl->stage_bytes = static_cast<uint32_t>(((pl->tile_rows * per_row) + 15) & ~int64_t(15));
  // Every stage must belong to one team: with stages a multiple of teams,
  // tile t and tile t + stages are consumed by the same team, so each team
  // waits on its stages strictly in order and a parity wait can never see a
  // phase that is two uses old.
  const int red_rows = pl->gpt * pl->rpg;
  auto fits = [&](int st) {
    return smem_layout(st, pl->stage_bytes, nv, red_rows, pl->tpr, nthreads).total <=
           static_cast<uint32_t>(dev.max_smem_optin);
  };
  int per_team = static_cast<int>(std::min<int64_t>(16, ring_target / pl->stage_bytes)) / pl->teams;
  per_team = std::max(1, std::min(per_team, 16 / pl->teams));
  while (per_team > 1 && !fits(per_team * pl->teams)) --per_team;
  if (pl->teams == 1 && per_team < 2 && fits(2)) per_team = 2;
  pl->stages = per_team * pl->teams;
  if (!fits(pl->stages)) return false;
  // stage x in shared memory too when it fits beside the ring
  const int min_stages = pl->teams == 1 ? 2 : pl->teams;
  pl->xstage = 0;
  for (int st = pl->stages; st >= min_stages; st -= pl->teams) {
    if (smem_layout(st, pl->stage_bytes, nv, red_rows, pl->tpr, nthreads, cols).total <=
        static_cast<uint32_t>(dev.max_smem_optin)) {
      pl->stages = st;
      pl->xstage = 1;
      break;
    }
  }
  pl->smem = smem_layout(pl->stages, pl->stage_bytes, nv, red_rows, pl->tpr, nthreads, pl->xstage ? cols : 0).total;
  return true;
}

// One-shot form when one vector is computed and a CTA's rows fit shared
// memory with x beside them.
bool flat_plan(int64_t row_bytes, int cols, int64_t rows_out, bool swiglu, int nvec, const DeviceInfo &dev,
               Plan *pl) {
  if (nvec != 1 || cols / 4 > kFlatMaxX4 * kMaxConsumers) return false;
  const int nblk = cols / 32;
  pl->tpr = std::min(32, std::max(8, next_pow2(nblk)));
  pl->groups = kMaxConsumers / pl->tpr;
  const int64_t g = std::min<int64_t>(dev.sm_count, (rows_out + 7) / 8);
  pl->grid = static_cast<unsigned>(std::max<int64_t>(1, g));
  pl->tile_rows = static_cast<int>((rows_out + pl->grid - 1) / pl->grid);
  pl->gpt = pl->teams = pl->rpg = 1;
  pl->stages = 1;
  pl->xstage = 1;
  pl->stage_bytes = static_cast<uint32_t>(pl->tile_rows * row_bytes);
  const int nwarps = kMaxConsumers / 32;
  uint32_t o = (swiglu ? 2u : 1u) * pl->stage_bytes + 16u;
  o = (o + 15u) & ~15u;
  o = ((o + 16 + 8u * nwarps + 15u) & ~15u) + 8u * 16 * nblk + 4u * nblk;
  pl->smem = (o + 15u) & ~15u;
  return pl->smem <= static_cast<uint32_t>(dev.max_smem_optin);
}

template <int FMT, bool SW>
cudaError_t launch_flat(const GemvParams &p, const Plan &pl, cudaStream_t s) {
  auto k = gemv_flat_kernel<FMT, SW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(pl.grid), dim3(pl.groups * pl.tpr + 32), pl.smem, s, p);
}

template <int FMT, int NV, int RPG, bool SW>
cudaError_t launch_one(const GemvParams &p, const Plan &pl, cudaStream_t s, bool pdl) {
  auto k = gemv_kernel<FMT, NV, RPG, SW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(pl.grid), block(pl.groups * pl.tpr + 32 + (pl.tpr > 32 ? 32 : 0));
  if (pdl) return launch_pdl(k, grid, block, pl.smem, s, p);
  k<<<grid, block, pl.smem, s>>>(p);
  return cudaGetLastError();
}

template <int FMT, int NV, bool SW>
cudaError_t dispatch_rpg(const GemvParams &p, const Plan &pl, cudaStream_t s, bool pdl) {
  switch (pl.rpg) {
    case 1:
      if constexpr (SW) return cudaErrorInvalidValue;
      else return launch_one<FMT, NV, 1, SW>(p, pl, s, pdl);
    case 2: return launch_one<FMT, NV, 2, SW>(p, pl, s, pdl);
    case 4: return launch_one<FMT, NV, 4, SW>(p, pl, s, pdl);
    case 8: return launch_one<FMT, NV, 8, SW>(p, pl, s, pdl);
  }
  return cudaErrorInvalidValue;
}

template <int FMT>
cudaError_t dispatch_fmt(const GemvParams &p, const Plan &pl, cudaStream_t s, bool pdl, bool sw) {
  if (p.nv == 1) return sw ? dispatch_rpg<FMT, 1, true>(p, pl, s, pdl) : dispatch_rpg<FMT, 1, false>(p, pl, s, pdl);
  return sw ? dispatch_rpg<FMT, 2, true>(p, pl, s, pdl) : dispatch_rpg<FMT, 2, false>(p, pl, s, pdl);
}

}  // namespace

// Shared with the expert kernels: plain dense launch over one matrix.
epq_status gemv_launch(epq_fmt fmt, const void *blocks, const float *x, float *y, int64_t rows, int64_t cols,
                       int nvec, const epq_gemv_opts *o, cudaStream_t s) {
  epq_gemv_opts opts = {};
  if (o) opts = *o;
  if (epq_block_weights(fmt) < 0) return EPQ_ERR_FORMAT;
  if (!blocks || !x || !y) return EPQ_ERR_ARG;
  if (nvec < 1 || nvec > 8) return EPQ_ERR_ARG;
  if (rows < 1 || cols < 256 || cols > 16384 || cols % 256) return EPQ_ERR_SHAPE;
  if (opts.swiglu && (rows % 2)) return EPQ_ERR_SHAPE;
  const int xg = opts.x_group > 1 ? opts.x_group : 1;
  if (xg > 1 && (opts.x_head_dim <= 0 || opts.x_head_dim % 32 || cols % (opts.x_head_dim * xg)))
    return EPQ_ERR_SHAPE;
  if (!aligned16(blocks) || !aligned16(x) || !aligned16(y) || (opts.residual && !aligned16(opts.residual)))
    return EPQ_ERR_ALIGN;
  if (opts.rms_prenorm && !(opts.rms_eps >= 0.0f)) return EPQ_ERR_ARG;
  if (opts.x_ld < 0 || (opts.x_ld && (opts.x_ld % 4 || opts.x_ld < cols / xg))) return EPQ_ERR_ARG;
  DeviceInfo dev;
  if (!current_device(&dev) || dev.major * 10 + dev.minor < 100) return EPQ_ERR_DEVICE;
  unsigned *err = device_error_slot();
  if (!err) return EPQ_ERR_DEVICE;

  const int64_t row_bytes = epq_row_bytes(fmt, cols);
  const int64_t rows_out = opts.swiglu ? rows / 2 : rows;
  const bool sw = opts.swiglu != 0;
  const int xs = opts.x_ld ? static_cast<int>(opts.x_ld) : static_cast<int>(cols / xg);
  // Q2_K / Q6_K, and Q4_K with one vector (or engine 3): the block-diagonal
  // tensor-core engine (gemv_k16.cu), measured faster than the ring engine
  // below on every matrix of the 8B-class decode step with one vector
  // (1.681 -> 1.459 ms per step) and slower with two (1.748 -> 2.046 ms),
  // where the ring engine's two-vector operands pay.  Two to four Q4_K
  // vectors keep the ring engine (one pass for 3..8 vectors on 4096-column
  // rows, else two vectors per pass).
  const int eng0 = tune_gemv_engine();
  // Q4_K with several vectors: the vector-column engine (gemv_vn.cu, one
  // weight pass for up to 8 vectors on every shape) from 5 vectors on, where
  // it was measured faster than the ring engine on the 8B-class step (8
  // vectors: 3.13 against 4.48 ms per step).  With 3 or 4 vectors it wins
  // only on gate/up and the LM head, and a step that alternates the two
  // engines lost 0.5 ms at the switches (neither overlaps the other's
  // tail: each needs a whole SM), so below 5 vectors every matrix keeps the
  // ring engine.  Engine 4 takes it for every Q4_K launch of 2+ vectors.
  const bool vn_auto = eng0 == 0 && nvec >= 5;
  if (fmt == EPQ_Q4_K && nvec >= 2 && (eng0 == 4 || vn_auto)) {
    const epq_status st = gemv_vn_launch(blocks, x, y, rows, cols, nvec, opts, xs, dev, s);
    if (st != EPQ_ERR_SHAPE) return st;  // rows too many for its chunked partial sums: the ring engine below
  }
  if (fmt == EPQ_Q2_K || fmt == EPQ_Q6_K || (fmt == EPQ_Q4_K && (eng0 == 3 || (eng0 != 1 && eng0 != 2 && nvec == 1))))
    return gemv_k16_launch(fmt, blocks, x, y, rows, cols, nvec, opts, xs, dev, s);

  // Q4_K (three or more vectors, or engine 2): the ring tensor-core engine
  // (two vectors per weight pass, more in the multi-vector form).  Engine 2
  // with one vector takes it for matrices of >= 2 MiB; smaller one-vector
  // launches keep the one-shot CUDA-core form, whose prologue is shorter.
  const int eng = tune_gemv_engine();
  const bool tc_auto = nvec >= 2 || rows * row_bytes >= (int64_t(2) << 20);
  TcPlan tp;
  if (fmt == EPQ_Q4_K && eng != 1 && (eng == 2 || tc_auto) &&
      gemv_tc_plan(row_bytes, static_cast<int>(cols), rows_out, sw, dev, &tp)) {
    TcArgs a;
    a.W = static_cast<const uint8_t *>(blocks);
    a.rows_out = rows_out;
    a.row_bytes = row_bytes;
    a.cols = static_cast<int>(cols);
    a.x_stride = xs;
    a.y_stride = rows_out;
    a.swiglu = sw ? 1 : 0;
    a.rms = opts.rms_prenorm;
    a.rms_eps = opts.rms_eps;
    a.x_group = xg;
    a.x_head_dim = opts.x_head_dim;
    a.early_weights = opts.weights_ready ? 1 : 0;
    a.err = err;
    if (nvec > 2) {  // all vectors in one weight pass where the shape allows
      a.x = x;
      a.y = y;
      a.residual = opts.residual;
      a.nv = nvec;
      cudaError_t e = cudaSuccess;
      if (gemv_tc_multi_launch(a, nvec, dev, s, &e)) return e == cudaSuccess ? EPQ_OK : cuda_fail(e);
    }
    for (int v0 = 0; v0 < nvec; v0 += 2) {
      a.nv = std::min(2, nvec - v0);
      a.x = x + v0 * a.x_stride;
      a.y = y + v0 * a.y_stride;
      a.residual = opts.residual ? opts.residual + v0 * a.y_stride : nullptr;
      const cudaError_t e = gemv_tc_launch(tp, a, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return EPQ_OK;
  }

  Plan pl;
  const bool flat = flat_plan(row_bytes, static_cast<int>(cols), rows_out, sw, nvec, dev, &pl);
  if (!flat && !make_plan(row_bytes, static_cast<int>(cols), rows_out, sw, std::min(nvec, 2), dev, &pl))
    return EPQ_ERR_SHAPE;

  GemvParams p;
  p.W = static_cast<const uint8_t *>(blocks);
  p.residual = opts.residual;
  p.rows_out = rows_out;
  p.up_rows = sw ? rows_out : 0;
  p.row_bytes = row_bytes;
  p.cols = static_cast<int>(cols);
  p.nblk = static_cast<int>(cols / 32);
  p.tpr = pl.tpr;
  p.groups = pl.groups;
  p.tile_rows = pl.tile_rows;
  p.red_rows = pl.gpt * pl.rpg;
  p.teams = pl.teams;
  p.gpt = pl.gpt;
  p.stages = pl.stages;
  p.stage_bytes = pl.stage_bytes;
  p.x_stride = xs;
  p.y_stride = rows_out;
  p.rms = opts.rms_prenorm;
  p.rms_eps = opts.rms_eps;
  p.x_group = xg;
  p.x_head_dim = opts.x_head_dim;
  p.early_weights = opts.weights_ready ? 1 : 0;
  p.xstage = pl.xstage;
  p.err = err;
  for (int v0 = 0; v0 < nvec; v0 += 2) {
    p.nv = std::min(2, nvec - v0);
    p.x = x + v0 * p.x_stride;
    p.y = y + v0 * p.y_stride;
    p.residual = opts.residual ? opts.residual + v0 * p.y_stride : nullptr;
    cudaError_t e = cudaErrorInvalidValue;
    if (flat) {
      switch (fmt) {
        case EPQ_Q8_0: e = sw ? launch_flat<EPQ_Q8_0, true>(p, pl, s) : launch_flat<EPQ_Q8_0, false>(p, pl, s); break;
        case EPQ_Q4_0: e = sw ? launch_flat<EPQ_Q4_0, true>(p, pl, s) : launch_flat<EPQ_Q4_0, false>(p, pl, s); break;
        case EPQ_Q4_1: e = sw ? launch_flat<EPQ_Q4_1, true>(p, pl, s) : launch_flat<EPQ_Q4_1, false>(p, pl, s); break;
        case EPQ_Q4_K: e = sw ? launch_flat<EPQ_Q4_K, true>(p, pl, s) : launch_flat<EPQ_Q4_K, false>(p, pl, s); break;
        default: return EPQ_ERR_FORMAT;  // Q2_K / Q6_K took the block-diagonal engine above
      }
      if (e != cudaSuccess) return cuda_fail(e);
      continue;
    }
    switch (fmt) {
      case EPQ_Q8_0: e = dispatch_fmt<EPQ_Q8_0>(p, pl, s, true, sw); break;
      case EPQ_Q4_0: e = dispatch_fmt<EPQ_Q4_0>(p, pl, s, true, sw); break;
      case EPQ_Q4_1: e = dispatch_fmt<EPQ_Q4_1>(p, pl, s, true, sw); break;
      case EPQ_Q4_K: e = dispatch_fmt<EPQ_Q4_K>(p, pl, s, true, sw); break;
      default: return EPQ_ERR_FORMAT;  // as above
    }
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return EPQ_OK;
}

}  // namespace epq

extern "C" epq_status epq_gemv(epq_fmt fmt, const void *blocks, const float *x, float *y, int64_t rows, int64_t cols,
                               int nvec, epq_stream_t stream) {
  return epq::gemv_launch(fmt, blocks, x, y, rows, cols, nvec, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" epq_status epq_gemv_ex(epq_fmt fmt, const void *blocks, const float *x, float *y, int64_t rows,
                                  int64_t cols, int nvec, const epq_gemv_opts *opts, epq_stream_t stream) {
  return epq::gemv_launch(fmt, blocks, x, y, rows, cols, nvec, opts, reinterpret_cast<cudaStream_t>(stream));
}

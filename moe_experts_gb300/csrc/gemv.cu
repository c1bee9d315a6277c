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

namespace epq {
namespace {

constexpr int kMaxConsumers = 512;
constexpr int kProducerThreads = 32;
constexpr int kTileTarget = 40 * 1024;   // bytes of packed weights per stage
constexpr int kSmemTarget = 160 * 1024;  // ring budget per CTA

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
  int tile_rows;       // output rows per tile (= groups * RPG, or groups * RPG/2 with swiglu)
  int red_rows;        // partial rows per tile (= groups * RPG)
  int stages;
  uint32_t stage_bytes;
  int nv;              // vectors in this launch (<= NV template)
  int64_t x_stride;    // floats between vectors of x
  int64_t y_stride;    // floats between vectors of y / residual
  int rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early_weights;   // weights are ready: stream them before the PDL wait
  unsigned *err;
};

struct SmemLayout {
  uint32_t stage_off, full_off, empty_off, redbar_off, red_off, scratch_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int stages, uint32_t stage_bytes, int nv, int red_rows, int tpr,
                                                  int nthreads) {
  SmemLayout L;
  L.stage_off = 0;
  uint32_t o = static_cast<uint32_t>(stages) * stage_bytes + 16;  // +16: code-word over-read pad
  o = (o + 15u) & ~15u;
  L.full_off = o;
  o += 8u * stages;
  L.empty_off = o;
  o += 8u * stages;
  L.redbar_off = o;
  o += 16;
  L.red_off = o;
  const int wpg = tpr > 32 ? tpr / 32 : 1;
  o += 4u * 2 * nv * red_rows * wpg;
  o = (o + 15u) & ~15u;
  L.scratch_off = o;
  o += 4u * 3 * nv * (nthreads / 32);
  L.total = (o + 15u) & ~15u;
  return L;
}

// Butterfly reduce-scatter of RPG partials over W lanes (W = segment width,
// a power of two >= RPG).  The first log2(RPG) levels (offsets W/2, W/4, ...)
// halve the set of rows a lane carries; the remaining levels are plain
// butterflies.  On return v[.][0] holds the full sum of row `base` (the
// returned index); the W/RPG lanes of each run share a row.
template <int RPG, int NV>
__device__ __forceinline__ int reduce_scatter(float (&v)[NV][RPG], int W, int lane) {
  int base = 0;
  int o = W >> 1;
#pragma unroll
  for (int n = RPG; n > 1; n >>= 1) {
    const int h = n / 2;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        const float send = upper ? v[q][i] : v[q][i + h];
        const float keep = upper ? v[q][i + h] : v[q][i];
        v[q][i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    if (upper) base += h;
    o >>= 1;
  }
  for (; o >= 1; o >>= 1) {
#pragma unroll
    for (int q = 0; q < NV; ++q) v[q][0] += __shfl_xor_sync(0xffffffffu, v[q][0], o);
  }
  return base;
}

__device__ __forceinline__ float silu(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

template <int FMT, int NV, int RPG, bool SWIGLU>
__global__ void __launch_bounds__(kMaxConsumers + kProducerThreads, 1) gemv_kernel(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nthreads = p.groups * p.tpr;
  const SmemLayout L = smem_layout(p.stages, p.stage_bytes, NV, p.red_rows, p.tpr, nthreads);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full_off);
  uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty_off);
  uint64_t *redbar = reinterpret_cast<uint64_t *>(smem + L.redbar_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  float *scratch = reinterpret_cast<float *>(smem + L.scratch_off);
  const int tid = threadIdx.x;
  const int nwarps = nthreads / 32;

  // rows of this CTA
  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * p.rows_out) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * p.rows_out) / gridDim.x;
  const int ntiles = static_cast<int>((re - rb + p.tile_rows - 1) / p.tile_rows);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nwarps);
    }
    mbar_init(&redbar[0], nwarps);
    mbar_init(&redbar[1], nwarps);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (tid >= nthreads) {
    // ------------------------------------------------------------ producer
    if (tid != nthreads) return;
    if (!p.early_weights) pdl_wait();
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % p.stages;
      if (t >= p.stages && !mbar_wait(&empty[s], ((t / p.stages) - 1) & 1, p.err, DEVERR_EMPTY_WAIT)) {
        ok = false;
        break;
      }
      const int64_t r0 = rb + static_cast<int64_t>(t) * p.tile_rows;
      const int64_t nr = min(static_cast<int64_t>(p.tile_rows), re - r0);
      const uint32_t bytes = static_cast<uint32_t>(nr * p.row_bytes);
      uint8_t *dst = smem + L.stage_off + static_cast<uint32_t>(s) * p.stage_bytes;
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
        mbar_wait(&full[t % p.stages], (t / p.stages) & 1, p.err, DEVERR_DRAIN_WAIT);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = tid / p.tpr;
  const int c = tid % p.tpr;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool active = c < p.nblk;
  const int W = p.tpr < 32 ? p.tpr : 32;

  ColConst<FMT> cc;
  cc.init(active ? c : 0);
  const XGather xg{p.x_group, p.x_head_dim};

  pdl_wait();  // x is produced upstream

  // load the column's activations
  float xr[NV][32];
  float amax[NV], ssq[NV], xsum[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    amax[v] = 0.0f;
    ssq[v] = 0.0f;
    xsum[v] = 0.0f;
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
      amax[v] = fmaxf(amax[v], fabsf(xr[v][j]));
      if (g == 0) ssq[v] = fmaf(xr[v][j], xr[v][j], ssq[v]);
      xsum[v] += xr[v][j];
    }
  }
  // CTA-wide max |x| and sum x^2 per vector (consumer threads only)
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    float a = warp_max_all(amax[v]);
    float q = warp_sum_xor<32>(ssq[v]);
    if (lane == 0) {
      scratch[(2 * v) * nwarps + warp] = a;
      scratch[(2 * v + 1) * nwarps + warp] = q;
    }
  }
  named_sync(1, nthreads);
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
    int eb = (__float_as_int(a) >> 23) & 0xFF;
    if (eb == 0) eb = 1;
    const int E = eb - 126;
    expo[v] = E;
#pragma unroll
    for (int j = 0; j < 32; ++j) xr[v][j] = scale_pow2(xr[v][j], 126 - E - Fmt<FMT>::shift(j));
    xsum[v] = scale_pow2(xsum[v], -23 - E);
    float r = 1.0f;
    if (p.rms) r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, static_cast<float>(p.cols)), p.rms_eps)));
    outscale[v] = r;
  }

  // per-tile loop
  constexpr int RH = SWIGLU ? RPG / 2 : RPG;  // gate rows per group (swiglu)
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % p.stages;
    if (!warp_wait(&full[s], (t / p.stages) & 1, p.err, DEVERR_FULL_WAIT)) return;
    const uint8_t *base = smem + L.stage_off + static_cast<uint32_t>(s) * p.stage_bytes;
    const int64_t r0 = rb + static_cast<int64_t>(t) * p.tile_rows;
    const int nr = static_cast<int>(min(static_cast<int64_t>(p.tile_rows), re - r0));
    float part[NV][RPG];
#pragma unroll
    for (int k = 0; k < RPG; ++k) {
      const int lr = SWIGLU ? (g * RH + (k % RH)) : (g * RPG + k);
      float pr[NV];
      if (active && lr < nr) {
        const uint8_t *row = base + static_cast<uint32_t>(lr) * p.row_bytes;
        if (SWIGLU && k >= RH) row += p.tile_rows * p.row_bytes;
        column_dot<FMT, NV>(row, cc, xr, xsum, pr);
      } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) pr[v] = 0.0f;
      }
#pragma unroll
      for (int v = 0; v < NV; ++v) part[v][k] = pr[v];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    // reduce over the group
    int ri = reduce_scatter<RPG, NV>(part, W, lane % W);
    float res[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) res[v] = 0.0f;
    int row_k = -1;  // which of the group's RPG rows this thread finalizes
    if (p.tpr > 32) {
      const int wpg = p.tpr / 32;
      const int wg = c >> 5;
      float *rbuf = red + (t & 1) * NV * p.red_rows * wpg;
      const int per_row = 32 / RPG;
      if ((lane % per_row) == 0) {
#pragma unroll
        for (int v = 0; v < NV; ++v) rbuf[(v * p.red_rows + g * RPG + ri) * wpg + wg] = part[v][0];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&redbar[t & 1]);
      if (wg == 0) {
        if (!warp_wait(&redbar[t & 1], (t >> 1) & 1, p.err, DEVERR_FULL_WAIT)) return;
        if (c < RPG) {
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            float acc = 0.0f;
            for (int w = 0; w < wpg; ++w) acc += rbuf[(v * p.red_rows + g * RPG + c) * wpg + w];
            res[v] = acc;
          }
          row_k = c;
        }
      }
    } else {
#pragma unroll
      for (int v = 0; v < NV; ++v) res[v] = part[v][0];
      if (((lane % W) % (W / RPG)) == 0) row_k = ri;
    }

    // epilogue
    if (SWIGLU) {
      // gate row k (< RH) pairs with up row k + RH
      float up[NV];
      if (p.tpr > 32) {
#pragma unroll
        for (int v = 0; v < NV; ++v) up[v] = __shfl_down_sync(0xffffffffu, res[v], RH);
      } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) up[v] = __shfl_xor_sync(0xffffffffu, res[v], W / 2);
      }
      if (row_k >= 0 && row_k < RH) {
        const int lr = g * RH + row_k;
        if (lr < nr) {
          const int64_t orow = r0 + lr;
          for (int v = 0; v < p.nv && v < NV; ++v) {
            const float gv = scale_pow2(res[v], 23 + expo[v]) * outscale[v];
            const float uv = scale_pow2(up[v], 23 + expo[v]) * outscale[v];
            float o = silu(gv) * uv;
            if (p.residual) o += p.residual[v * p.y_stride + orow];
            p.y[v * p.y_stride + orow] = o;
          }
        }
      }
    } else if (row_k >= 0) {
      const int lr = g * RPG + row_k;
      if (lr < nr) {
        const int64_t orow = r0 + lr;
        for (int v = 0; v < p.nv && v < NV; ++v) {
          float o = scale_pow2(res[v], 23 + expo[v]) * outscale[v];
          if (p.residual) o += p.residual[v * p.y_stride + orow];
          p.y[v * p.y_stride + orow] = o;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ host
struct Plan {
  int tpr, groups, rpg, tile_rows, stages;
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
  const int wcap = std::min(pl->tpr, 32);
  const int rmax = std::min(8, wcap);
  const int64_t per_row = row_bytes * (swiglu ? 2 : 1);
  int rpg = swiglu ? 2 : 1;
  while (rpg * 2 <= rmax && static_cast<int64_t>(pl->groups) * rpg * 2 * per_row <= kTileTarget) rpg *= 2;
  pl->rpg = rpg;
  const int rows_per_tile = pl->groups * (swiglu ? rpg / 2 : rpg);
  pl->tile_rows = rows_per_tile;
  pl->stage_bytes = static_cast<uint32_t>(((rows_per_tile * per_row) + 15) & ~int64_t(15));
  pl->stages = static_cast<int>(std::max<int64_t>(2, std::min<int64_t>(8, kSmemTarget / pl->stage_bytes)));
  const int red_rows = pl->groups * rpg;
  while (pl->stages > 2 &&
         smem_layout(pl->stages, pl->stage_bytes, nv, red_rows, pl->tpr, pl->groups * pl->tpr).total >
             static_cast<uint32_t>(dev.max_smem_optin))
    --pl->stages;
  pl->smem = smem_layout(pl->stages, pl->stage_bytes, nv, red_rows, pl->tpr, pl->groups * pl->tpr).total;
  if (pl->smem > static_cast<uint32_t>(dev.max_smem_optin)) return false;
  int64_t g = std::min<int64_t>(dev.sm_count, (rows_out + 7) / 8);
  pl->grid = static_cast<unsigned>(std::max<int64_t>(1, g));
  return true;
}

template <int FMT, int NV, int RPG, bool SW>
cudaError_t launch_one(const GemvParams &p, const Plan &pl, cudaStream_t s, bool pdl) {
  auto k = gemv_kernel<FMT, NV, RPG, SW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(pl.grid), block(pl.groups * pl.tpr + kProducerThreads);
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
  DeviceInfo dev;
  if (!current_device(&dev) || dev.major * 10 + dev.minor < 100) return EPQ_ERR_DEVICE;
  unsigned *err = device_error_slot();
  if (!err) return EPQ_ERR_DEVICE;

  const int64_t row_bytes = epq_row_bytes(fmt, cols);
  const int64_t rows_out = opts.swiglu ? rows / 2 : rows;
  const bool sw = opts.swiglu != 0;
  Plan pl;
  if (!make_plan(row_bytes, static_cast<int>(cols), rows_out, sw, std::min(nvec, 2), dev, &pl)) return EPQ_ERR_SHAPE;

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
  p.red_rows = pl.groups * pl.rpg;
  p.stages = pl.stages;
  p.stage_bytes = pl.stage_bytes;
  p.x_stride = cols / xg;
  p.y_stride = rows_out;
  p.rms = opts.rms_prenorm;
  p.rms_eps = opts.rms_eps;
  p.x_group = xg;
  p.x_head_dim = opts.x_head_dim;
  p.early_weights = 0;
  p.err = err;
  for (int v0 = 0; v0 < nvec; v0 += 2) {
    p.nv = std::min(2, nvec - v0);
    p.x = x + v0 * p.x_stride;
    p.y = y + v0 * p.y_stride;
    p.residual = opts.residual ? opts.residual + v0 * p.y_stride : nullptr;
    cudaError_t e = cudaErrorInvalidValue;
    switch (fmt) {
      case EPQ_Q8_0: e = dispatch_fmt<EPQ_Q8_0>(p, pl, s, false, sw); break;
      case EPQ_Q4_0: e = dispatch_fmt<EPQ_Q4_0>(p, pl, s, false, sw); break;
      case EPQ_Q4_1: e = dispatch_fmt<EPQ_Q4_1>(p, pl, s, false, sw); break;
      case EPQ_Q4_K: e = dispatch_fmt<EPQ_Q4_K>(p, pl, s, false, sw); break;
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

// Tensor-core dequant-GEMV for Q2_K and Q6_K (epq_gemv / epq_gemv_ex), and
// the block-diagonal engine for Q4_K (EPQ_TUNE_GEMV_ENGINE 3).
//
// [H] "速度上限：带宽 ÷ 权重字节数": batch-1 decode streams every packed
// weight once per token.  The operand decode and the MMA layout are those of
// k16_core.cuh; this file adds the CTA organisation:
//   * a CTA of 8 warps works on RG row groups at a time (16 output rows
//     each; 8 gate + 8 up rows with SwiGLU) and splits the superblocks of
//     every row between KP = 8 / RG warps (warp kq takes superblocks kq,
//     kq + KP, ...); the grid holds at most two CTAs per SM and a CTA loops
//     over blocks of RG groups (k16_split picks RG and the grid);
//   * the CTA first converts all of x into the shared-memory operand records
//     (one warp per (vector, superblock)), together with the per-superblock
//     scales, the sub-block sums of x and the sums of squares (RMS pre-norm);
//   * each warp streams its rows' planes straight into registers (16-byte
//     loads, no L1 allocation) through a ring of 4 (Q2_K) or 2 (Q6_K)
//     superblocks in flight ahead of the MMAs;
//   * row totals: the 4 lanes of a row add their owners' parts with two
//     butterflies, the KP warps' partials are added in k-part order through
//     shared memory (deterministic), then the epilogue applies the RMS
//     scale, SwiGLU and the residual.
// Rows run past the end of the matrix read the last row and store nothing.
#include <algorithm>

#include "k16_core.cuh"

namespace epq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct K16Params {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows_out;
  int64_t up_rows;  // swiglu: row distance gate -> up
  int64_t row_bytes;
  int nsb;
  int rg, kp;  // row groups per CTA, warps per row group
  int nv;      // vectors in this launch (<= NV)
  int64_t x_stride, y_stride;
  int rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early;  // weights may be read before the grid-dependency wait
};

struct K16Layout {
  uint32_t frag, ps, xsum, red, ssq, total;
};

__host__ __device__ inline uint32_t al16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline K16Layout k16_layout(int nv, int nsb) {
  K16Layout L;
  uint32_t o = 0;
  L.frag = o;
  o += static_cast<uint32_t>(nv * nsb) * k16::kSbFragBytes;
  L.ps = o;
  o = al16(o + 4u * nv * nsb);
  L.xsum = o;
  o = al16(o + 4u * nv * nsb * 16);
  L.red = o;  // [warp][16 rows][nv]
  o = al16(o + 4u * kWarps * 16 * nv);
  L.ssq = o;  // [warp][nv]
  o = al16(o + 4u * kWarps * nv);
  L.total = o;
  return L;
}

__device__ __forceinline__ float silu(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

__device__ __forceinline__ int x_src(int j, int group, int head_dim) {
  if (group <= 1) return j;
  const int span = head_dim * group;
  return (j / span) * head_dim + (j % head_dim);
}

template <int FMT, int NV, int ALIGN, bool SW>
__global__ void __launch_bounds__(kThreads, NV <= 2 ? 2 : 1) gemv_k16_kernel(const K16Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const K16Layout L = k16_layout(NV, p.nsb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kq = warp % p.kp, rgl = warp / p.kp;
  constexpr int kOut = SW ? 8 : 16;  // outputs per row group
  // The CTA takes the row-group blocks blockIdx.x, blockIdx.x + gridDim.x,
  // ... (RG groups each); x is staged once for all of them.
  const int64_t ngroups = (p.rows_out + kOut - 1) / kOut;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * p.rg, stride = static_cast<int64_t>(gridDim.x) * p.rg;
  const int iters = first < ngroups ? static_cast<int>((ngroups - first + stride - 1) / stride) : 0;
  const int64_t nsb = p.nsb;
  // rows of A held by this lane in iteration it: g (lo) and g + 8 (hi),
  // clamped to the matrix (rows past the end are read but not stored)
  auto rows_of = [&](int it, const uint8_t *&lo, const uint8_t *&hi) {
    const int64_t rg = first + it * stride + rgl;
    int64_t r_lo, r_hi;
    if (SW) {
      r_lo = min(rg * 8 + g, p.rows_out - 1);
      r_hi = p.up_rows + r_lo;
    } else {
      r_lo = min(rg * 16 + g, p.rows_out - 1);
      r_hi = min(rg * 16 + g + 8, p.rows_out - 1);
    }
    lo = p.W + r_lo * p.row_bytes;
    hi = p.W + r_hi * p.row_bytes;
  };

  // This warp's superblocks kq, kq + KP, ... of each row group: kDepth of
  // them are in flight (a register ring indexed by compile-time slots); the
  // first ones of the next row group are issued before the row totals.
  constexpr int kDepth = FMT == EPQ_Q2_K ? 4 : 2;
  k16::RowOps<FMT> ring_lo[kDepth], ring_hi[kDepth];
  const int cnt = kq < p.nsb ? (p.nsb - kq + p.kp - 1) / p.kp : 0;
  pdl_launch_dependents();  // the next kernel may start its prologue; it waits for this grid before reading y
  const uint8_t *row_lo = nullptr, *row_hi = nullptr;
  auto fill = [&](int it) {
    rows_of(it, row_lo, row_hi);
#pragma unroll
    for (int d = 0; d < kDepth; ++d)
      if (d < cnt) {
        k16::load_ops<FMT, ALIGN>(ring_lo[d], row_lo, nsb, kq + d * p.kp, t);
        k16::load_ops<FMT, ALIGN>(ring_hi[d], row_hi, nsb, kq + d * p.kp, t);
      }
  };
  if (p.early && iters > 0) fill(0);
  pdl_wait();
  if (!p.early && iters > 0) fill(0);

  // ---------------------------------------------------------------- x staging
  float ssq[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) ssq[v] = 0.0f;
  float *ps_s = reinterpret_cast<float *>(smem + L.ps);
  float *xsum_s = reinterpret_cast<float *>(smem + L.xsum);
  // a warp stages units warp, warp + 8, ...; the x loads of kStageBatch
  // units are issued before any of them is converted, and their warp
  // maxima are reduced back to back before the conversions
  constexpr int kStageBatch = 4;
  const int nunits = NV * p.nsb;
  for (int u0 = warp; u0 < nunits; u0 += kWarps * kStageBatch) {
    float xv[kStageBatch][8];
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const int u = u0 + kWarps * k;
      const int v = u / p.nsb, b = u - v * p.nsb;
      const int j0 = b * 256 + 8 * lane;
      if (u < nunits && v < p.nv) {
        // the 8 columns lie in one head (head_dim % 32 == 0), so their
        // sources are consecutive too: one index, two 16-byte loads
        const float *xr = p.x + v * p.x_stride + x_src(j0, p.x_group, p.x_head_dim);
        const float4 a = *reinterpret_cast<const float4 *>(xr);
        const float4 c = *reinterpret_cast<const float4 *>(xr + 4);
        xv[k][0] = a.x, xv[k][1] = a.y, xv[k][2] = a.z, xv[k][3] = a.w;
        xv[k][4] = c.x, xv[k][5] = c.y, xv[k][6] = c.z, xv[k][7] = c.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[k][e] = 0.0f;
      }
    }
    float mx[kStageBatch];
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) mx[k] = warp_absmax(k16::lane_absmax(xv[k]));
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const int u = u0 + kWarps * k;
      if (u >= nunits) break;  // warp-uniform
      const int v = u / p.nsb, b = u - v * p.nsb;
      if (p.rms) {
        float sq = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) sq = fmaf(xv[k][e], xv[k][e], sq);
#pragma unroll
        for (int w = 0; w < NV; ++w)
          if (w == v) ssq[w] += sq;
      }
      uint8_t *frag_sb = smem + L.frag + static_cast<uint32_t>(v * p.nsb + b) * k16::kSbFragBytes;
      const int ex = FMT == EPQ_Q4_K
                         ? k16::stage_superblock_q4k(xv[k], mx[k], frag_sb, lane, xsum_s + (v * p.nsb + b) * 16)
                         : k16::stage_superblock(xv[k], mx[k], frag_sb, lane, xsum_s + (v * p.nsb + b) * 16);
      if (lane == 0) ps_s[v * p.nsb + b] = k16::sum_scale<FMT>(ex);
    }
  }
  float *ssq_s = reinterpret_cast<float *>(smem + L.ssq);
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const float s = warp_sum_xor<32>(ssq[v]);
    if (lane == 0) ssq_s[warp * NV + v] = s;
  }
  __syncthreads();

  // ---------------------------------------------------------------- main loop
  const uint8_t *frag0 = smem + L.frag + k16::lane_slot(lane);
  const uint32_t vstride = static_cast<uint32_t>(p.nsb) * k16::kSbFragBytes;
  float *red = reinterpret_cast<float *>(smem + L.red);
  float rs[NV];  // RMS factors of the vectors
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    rs[v] = 1.0f;
    if (p.rms) {
      float q = 0.0f;
      for (int w = 0; w < kWarps; ++w) q += ssq_s[w * NV + v];
      rs[v] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, static_cast<float>(p.nsb * 256)), p.rms_eps)));
    }
  }
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    float acc[2][NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[0][v] = acc[1][v] = 0.0f;
    for (int j0 = 0; j0 < cnt; j0 += kDepth) {
#pragma unroll
      for (int d = 0; d < kDepth; ++d) {
        const int j = j0 + d;
        if (j >= cnt) break;
        const int b = kq + j * p.kp;
        float ps[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) ps[v] = ps_s[v * p.nsb + b];
        k16::superblock<FMT, NV>(ring_lo[d], ring_hi[d], frag0 + b * k16::kSbFragBytes,
                                 vstride, ps, xsum_s + b * 16, p.nsb * 16, t, acc);
        if (j + kDepth < cnt) {
          k16::load_ops<FMT, ALIGN>(ring_lo[d], row_lo, nsb, b + kDepth * p.kp, t);
          k16::load_ops<FMT, ALIGN>(ring_hi[d], row_hi, nsb, b + kDepth * p.kp, t);
        }
      }
    }
    if (it + 1 < iters) fill(it + 1);

    // ---------------------------------------------------------------- row totals
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float s = acc[r][v];
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (t == 0) red[(warp * 16 + g + 8 * r) * NV + v] = s;
      }
    __syncthreads();
    const int nout = p.rg * kOut * NV;
    for (int idx = threadIdx.x; idx < nout; idx += kThreads) {
      const int v = idx % NV, o = (idx / NV) % kOut, gl = idx / (NV * kOut);
      const int64_t i = (first + it * stride + gl) * kOut + o;
      if (v >= p.nv || i >= p.rows_out) continue;
      float a = 0.0f, b = 0.0f;
      for (int k = 0; k < p.kp; ++k) {
        const float *rr = red + ((gl * p.kp + k) * 16) * NV;
        a += rr[o * NV + v];
        if (SW) b += rr[(o + 8) * NV + v];
      }
      float r = rs[0];
#pragma unroll
      for (int w = 1; w < NV; ++w)
        if (w == v) r = rs[w];  // constant indices keep rs in registers
      float val = a * r;
      if (SW) val = silu(val) * (b * r);
      if (p.residual) val += p.residual[v * p.y_stride + i];
      p.y[v * p.y_stride + i] = val;
    }
    __syncthreads();  // red is rewritten by the next row group
  }
}

template <int FMT, int NV, int ALIGN, bool SW>
cudaError_t launch_k16(const K16Params &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  auto k = gemv_k16_kernel<FMT, NV, ALIGN, SW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(kThreads), smem, s, p);
}

template <int FMT, int NV, int ALIGN>
cudaError_t dispatch_sw(const K16Params &p, bool sw, unsigned grid, uint32_t smem, cudaStream_t s) {
  return sw ? launch_k16<FMT, NV, ALIGN, true>(p, grid, smem, s) : launch_k16<FMT, NV, ALIGN, false>(p, grid, smem, s);
}

template <int FMT, int NV>
cudaError_t dispatch_k16(const K16Params &p, int align, bool sw, unsigned grid, uint32_t smem, cudaStream_t s) {
  if (align == 16) return dispatch_sw<FMT, NV, 16>(p, sw, grid, smem, s);
  if (align == 4) return dispatch_sw<FMT, NV, 4>(p, sw, grid, smem, s);
  if constexpr (FMT == EPQ_Q6_K) return dispatch_sw<FMT, NV, 2>(p, sw, grid, smem, s);
  return cudaErrorInvalidValue;
}

// Row groups per CTA (RG; the 8 warps split the superblocks KP = 8 / RG
// ways) and grid.  Two CTAs per SM hide latency far better than one, so
// among the RGs that still give every SM two CTAs (blocks >= 2 SMs) the one
// with the fewest per-CTA iterations x (superblocks per warp + 1 for the
// per-iteration reduction) wins, ties going to the larger RG; when no RG
// fills the GPU twice, RG = 1 and one CTA per row group.
void k16_split(int64_t ngroups, int nsb, int sms, int per_sm, int *rg_out, unsigned *grid_out) {
  const int64_t cap = static_cast<int64_t>(per_sm) * sms;
  int64_t best = -1;
  *rg_out = 1;
  *grid_out = static_cast<unsigned>(std::max<int64_t>(1, std::min(ngroups, cap)));
  for (int rg = 8; rg >= 1; rg >>= 1) {
    const int64_t units = (ngroups + rg - 1) / rg;
    if (units < cap) continue;
    const int kp = kWarps / rg;
    const int64_t cost = (units + cap - 1) / cap * ((nsb + kp - 1) / kp + 1);
    if (best < 0 || cost < best) {
      best = cost;
      *rg_out = rg;
      *grid_out = static_cast<unsigned>(cap);
    }
  }
}

}  // namespace

// Called by gemv_launch (gemv.cu) after the common argument checks.
epq_status gemv_k16_launch(epq_fmt fmt, const void *blocks, const float *x, float *y, int64_t rows, int64_t cols,
                           int nvec, const epq_gemv_opts &o, int64_t x_stride, const DeviceInfo &dev,
                           cudaStream_t s) {
  const int64_t row_bytes = epq_row_bytes(fmt, cols);
  const bool sw = o.swiglu != 0;
  const int64_t rows_out = sw ? rows / 2 : rows;
  const int nsb = static_cast<int>(cols / 256);
  // vectors per weight pass: Q4_K takes up to 8 in one pass when their x
  // operands fit shared memory (one CTA per SM from 4 vectors on), else
  // passes of two
  int nvl = nvec <= 1 ? 1 : nvec <= 2 ? 2 : nvec <= 4 ? 4 : 8;
  if (fmt != EPQ_Q4_K) nvl = std::min(nvl, 2);
  while (nvl > 2 && k16_layout(nvl, nsb).total > static_cast<uint32_t>(dev.max_smem_optin)) nvl /= 2;
  const K16Layout L = k16_layout(nvl, nsb);
  if (L.total > static_cast<uint32_t>(dev.max_smem_optin)) return EPQ_ERR_SHAPE;
  // resident CTAs per SM: two when the launch bounds and 2 x (smem + the
  // 1 KB the runtime reserves per CTA) fit the SM's 228 KB
  const int per_sm = nvl <= 2 && 2 * (L.total + 1024u) <= 233472u ? 2 : 1;
  const int64_t ngroups = (rows_out + (sw ? 7 : 15)) / (sw ? 8 : 16);
  int rg = 1;
  unsigned grid = 1;
  k16_split(ngroups, nsb, dev.sm_count, per_sm, &rg, &grid);
  K16Params p;
  p.W = static_cast<const uint8_t *>(blocks);
  p.rows_out = rows_out;
  p.up_rows = sw ? rows_out : 0;
  p.row_bytes = row_bytes;
  p.nsb = nsb;
  p.rg = rg;
  p.kp = kWarps / rg;
  p.x_stride = x_stride;
  p.y_stride = rows_out;
  p.rms = o.rms_prenorm;
  p.rms_eps = o.rms_eps;
  p.x_group = o.x_group > 1 ? o.x_group : 1;
  p.x_head_dim = o.x_head_dim;
  p.early = o.weights_ready ? 1 : 0;
  const int align = row_bytes % 16 == 0 ? 16 : (row_bytes % 4 == 0 ? 4 : 2);
  for (int v0 = 0; v0 < nvec; v0 += nvl) {
    p.nv = std::min(nvl, nvec - v0);
    p.x = x + v0 * x_stride;
    p.y = y + v0 * rows_out;
    p.residual = o.residual ? o.residual + v0 * rows_out : nullptr;
    cudaError_t e;
    if (fmt == EPQ_Q4_K)  // 144-byte superblocks: every row starts on a 16-byte boundary
      e = nvl == 1   ? dispatch_sw<EPQ_Q4_K, 1, 16>(p, sw, grid, L.total, s)
          : nvl == 2 ? dispatch_sw<EPQ_Q4_K, 2, 16>(p, sw, grid, L.total, s)
          : nvl == 4 ? dispatch_sw<EPQ_Q4_K, 4, 16>(p, sw, grid, L.total, s)
                     : dispatch_sw<EPQ_Q4_K, 8, 16>(p, sw, grid, L.total, s);
    else if (fmt == EPQ_Q2_K)
      e = nvl == 1 ? dispatch_k16<EPQ_Q2_K, 1>(p, align, sw, grid, L.total, s)
                   : dispatch_k16<EPQ_Q2_K, 2>(p, align, sw, grid, L.total, s);
    else
      e = nvl == 1 ? dispatch_k16<EPQ_Q6_K, 1>(p, align, sw, grid, L.total, s)
                   : dispatch_k16<EPQ_Q6_K, 2>(p, align, sw, grid, L.total, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return EPQ_OK;
}

}  // namespace epq

// Tensor-core Q4_K dequant-GEMV for 3 to 8 vectors in one weight pass
// (epq_gemv / epq_gemv_ex with nvec > 2): the speculative-verify columns.
//
// [H] "速度上限：带宽 ÷ 权重字节数": a decode step is bound by the bytes of the
// weights it streams, so checking several draft tokens costs about one
// weight pass when the columns share it.  The kernel is the one-vector-pair
// engine of gemv_tc.cu with each decoded A fragment (8 rows x 32 weights,
// the nibble -> fp16 decode being the costly part) multiplied by NVP vector
// pairs: NVP MMAs per code word instead of one, and NVP sets of x operands
// in registers.  It covers rows of 16 superblocks (4096 weights), where all
// 16 warps take one superblock each of every 8-row block; wider rows fall
// back to one pass per vector pair.
#include <algorithm>

#include "gemv_tc.cuh"
#include "gemv_tc_core.cuh"

namespace epq {
namespace {

using namespace tc;

constexpr int kMWarps = 16;  // one superblock per warp
constexpr int kMThreads = kMWarps * 32;

struct MultiParams {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows_out, up_rows, row_bytes;
  int cols;
  int stages;
  uint32_t stage_bytes;
  int nv;
  int64_t x_stride, y_stride;
  int rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early_weights;
  unsigned *err;
};

struct MultiLayout {
  uint32_t full, cnt, red, xs, scratch, frag, total;
  int held;
};

__host__ __device__ inline uint32_t al16m(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline MultiLayout multi_layout(int stages, uint32_t stage_bytes, int nvp, bool swiglu) {
  MultiLayout L;
  const int V = 2 * nvp;
  uint32_t o = al16m(static_cast<uint32_t>(stages) * stage_bytes);
  L.full = o;
  o += 8u * stages;
  L.cnt = o;
  o = al16m(o + 4u * stages);
  L.red = o;  // [slot][warp 16][row 8][vector V][gate/up]
  o = al16m(o + 4u * stages * kMWarps * 8 * V * (swiglu ? 2 : 1));
  L.xs = o;  // [superblock 16][t 4][vector V][sub-block pair 2]
  o = al16m(o + 4u * 16 * 4 * V * 2);
  L.scratch = o;  // [warp][vector V]: sums of squares
  o = al16m(o + 4u * kMWarps * V);
  const uint32_t fb = 16u * kFragWarpBytes;  // per-warp staging of one superblock's operands
  const int held = static_cast<int>((fb + stage_bytes - 1) / stage_bytes);
  if (held < stages) {
    L.held = held;
    L.frag = static_cast<uint32_t>(stages - held) * stage_bytes;
  } else {
    L.held = 0;
    L.frag = o;
    o += fb;
  }
  L.total = al16m(o);
  return L;
}

template <int NVP, bool SWIGLU>
__global__ void __launch_bounds__(kMThreads, 1) gemv_q4k_tc_multi_kernel(const MultiParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int M = SWIGLU ? 2 : 1;
  constexpr int V = 2 * NVP;
  const MultiLayout L = multi_layout(p.stages, p.stage_bytes, NVP, SWIGLU);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
  unsigned *cnt = reinterpret_cast<unsigned *>(smem + L.cnt);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *xsum = reinterpret_cast<float *>(smem + L.xs);
  float *scratch = reinterpret_cast<float *>(smem + L.scratch);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int64_t rb = (static_cast<int64_t>(blockIdx.x) * p.rows_out) / gridDim.x;
  const int64_t re = (static_cast<int64_t>(blockIdx.x + 1) * p.rows_out) / gridDim.x;
  const int nst = static_cast<int>((re - rb + 7) / 8);  // one 8-row block per stage

  auto issue = [&](int i) {
    const int s = i % p.stages;
    const int64_t r0 = rb + static_cast<int64_t>(i) * 8;
    const int64_t nr = min(static_cast<int64_t>(8), re - r0);
    const uint32_t bytes = static_cast<uint32_t>(nr * p.row_bytes);
    uint8_t *dst = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    mbar_arrive_expect_tx(&full[s], SWIGLU ? 2 * bytes : bytes);
    bulk_g2s(dst, p.W + r0 * p.row_bytes, bytes, &full[s]);
    if (SWIGLU)
      bulk_g2s(dst + static_cast<uint32_t>(8 * p.row_bytes), p.W + (p.up_rows + r0) * p.row_bytes, bytes,
               &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      cnt[s] = 0u;
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (tid == 0) {
    if (!p.early_weights) pdl_wait();
    for (int i = 0; i < min(p.stages - L.held, nst); ++i) issue(i);
  }

  // ------------------------------------------------------------------ prologue
  // warp w converts superblock w of every vector pair (see gemv_tc.cu)
  pdl_wait();
  const XGather xg{p.x_group, p.x_head_dim};
  const int g = lane >> 2, t = lane & 3;
  const int sb = warp;
  const int cv = t & 1;
  uint32_t bq[NVP][8][2];
  float fsc[NVP];
  {
    uint2 *frag = reinterpret_cast<uint2 *>(smem + L.frag) + warp * (kFragWarpBytes / 8);
    const int sub = lane >> 2, wi = lane & 3;
    const int tp = sub >> 1, jj = 4 * (sub & 1) + wi;
    float4 xr[V][2];
#pragma unroll
    for (int v = 0; v < V; ++v) {  // loads of absent vectors read vector 0 (zeroed below)
      const float *src = p.x + (v < p.nv ? v : 0) * p.x_stride + xg.src(256 * sb + 8 * lane);
      xr[v][0] = ldg4(src);
      xr[v][1] = ldg4(src + 4);
    }
#pragma unroll
    for (int v = 0; v < V; ++v)
      if (v >= p.nv) xr[v][0] = xr[v][1] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int pp = 0; pp < NVP; ++pp) {
      float fs[2];
#pragma unroll
      for (int w2 = 0; w2 < 2; ++w2) {
        const int v = 2 * pp + w2;
        const float q0[8] = {xr[v][0].x, xr[v][0].y, xr[v][0].z, xr[v][0].w,
                             xr[v][1].x, xr[v][1].y, xr[v][1].z, xr[v][1].w};
        float amax = 0.0f, s8 = 0.0f, ssq = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          amax = fmaxf(amax, fabsf(q0[e]));
          ssq = fmaf(q0[e], q0[e], ssq);
          s8 += q0[e];
        }
        amax = warp_max_all(amax);
        ssq = warp_sum_xor<32>(ssq);
        if (lane == 0) scratch[warp * V + v] = ssq;
        s8 += __shfl_xor_sync(0xffffffffu, s8, 1);
        s8 += __shfl_xor_sync(0xffffffffu, s8, 2);
        if (wi == 0) xsum[((sb * 4 + tp) * V + v) * 2 + (sub & 1)] = s8;
        const int sig = min(126, max(-112, 15 - bound_exponent(amax)));
        fs[w2] = exp2i(14 - sig);
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
          const int l0 = 4 * (4 * h + 2 * w2) + tp;
          frag[jj * kFragRow + l0] = hi;
          frag[jj * kFragRow + l0 + 4] = lo;
        }
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint2 r = frag[j * kFragRow + lane];
        bq[pp][j][0] = r.x;
        bq[pp][j][1] = r.y;
      }
      fsc[pp] = cv ? fs[1] : fs[0];
      __syncwarp();
    }
  }
  named_sync(1, kMThreads);  // all staging areas consumed (prologue only: no warp has left yet)
  if (tid == 0 && L.held > 0 && p.stages - L.held < nst) {
    fence_proxy_async();
    for (int i = p.stages - L.held; i < min(p.stages, nst); ++i) issue(i);
  }
  const uint32_t csel = t == 0 ? 0x10u : (t == 1 ? 0x21u : (t == 2 ? 0x43u : 0x54u));
  const uint32_t ksel = t == 0 ? 0x32u : (t == 1 ? 0x43u : (t == 2 ? 0x65u : 0x76u));
  const int nsh = (t & 1) * 4;
  uint32_t magic = kH1024;
  asm volatile("" : "+r"(magic));
  const uint32_t rbytes = static_cast<uint32_t>(p.row_bytes);

  // ------------------------------------------------------------------ main loop
  for (int i = 0; i < nst; ++i) {
    const int s = i % p.stages;
    if (!warp_wait(&full[s], (i / p.stages) & 1, p.err, DEVERR_FULL_WAIT, i)) {
      if (lane == 0)
        for (int j = i; j < min(nst, i + p.stages); ++j)
          mbar_wait(&full[j % p.stages], (j / p.stages) & 1, p.err, DEVERR_DRAIN_WAIT, j);
      return;
    }
    const uint8_t *sbase = smem + static_cast<uint32_t>(s) * p.stage_bytes;
    float *rs = red + static_cast<uint32_t>(s * kMWarps * 8 * V * M);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const uint8_t *sp = sbase + static_cast<uint32_t>(m * 8 + g) * rbytes + sb * 144;
      const uint4 hd = *reinterpret_cast<const uint4 *>(sp);
      const uint4 qa = *reinterpret_cast<const uint4 *>(sp + 16 + 32 * t);
      const uint4 qb = *reinterpret_cast<const uint4 *>(sp + 32 + 32 * t);
      const uint32_t cc = __byte_perm(hd.y, hd.z, csel) >> nsh;
      const uint32_t kk = __byte_perm(hd.z, hd.w, ksel) >> nsh;
      const SubMul ma = sub_mul(cc & 63u, magic), mb = sub_mul((cc >> 6) & 63u, magic);
      float C[NVP][4];
#pragma unroll
      for (int pp = 0; pp < NVP; ++pp) C[pp][0] = C[pp][1] = C[pp][2] = C[pp][3] = 0.0f;
      const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const SubMul &mm = j < 4 ? ma : mb;
        const uint32_t w = words[j], w8 = w >> 8;
        const uint32_t a0 = hmul2(w & 0x000F000Fu, mm.lo);
        const uint32_t a1 = hmul2(w & 0x00F000F0u, mm.hi);
        const uint32_t a2 = hmul2(w8 & 0x000F000Fu, mm.lo);
        const uint32_t a3 = hmul2(w8 & 0x00F000F0u, mm.hi);
#pragma unroll
        for (int pp = 0; pp < NVP; ++pp) mma16816(C[pp], a0, a1, a2, a3, bq[pp][j][0], bq[pp][j][1]);
      }
      const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hd.x));  // d, dmin
      const float ka = u6_to_float(kk & 63u), kb = u6_to_float((kk >> 6) & 63u);
      const float *X = xsum + (sb * 4 + t) * V * 2;
#pragma unroll
      for (int pp = 0; pp < NVP; ++pp) {
        const float sc = t < 2 ? C[pp][0] + C[pp][1] : C[pp][2] + C[pp][3];
        const float code = dd.x * (sc * fsc[pp]);
        float p0 = (cv == 0 ? code : 0.0f) - dd.y * fmaf(ka, X[(2 * pp) * 2], kb * X[(2 * pp) * 2 + 1]);
        float p1 = (cv == 1 ? code : 0.0f) - dd.y * fmaf(ka, X[(2 * pp + 1) * 2], kb * X[(2 * pp + 1) * 2 + 1]);
        p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
        p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
        if (t < 2) rs[((warp * 8 + g) * V + 2 * pp + t) * M + m] = t == 0 ? p0 : p1;
      }
    }
    __syncwarp();
    unsigned old = 0u;
    if (lane == 0) old = atom_add_acq_rel(&cnt[s], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    __syncwarp();
    if (((old + 1u) & (kMWarps - 1)) == 0u) {
      // last warp on this stage: outputs (k-parts added in warp order), refill
      for (int o = lane; o < 8 * V; o += 32) {
        const int gg = o / V, v = o % V;
        const int64_t row = rb + 8 * i + gg;
        if (row < re && v < p.nv) {
          float sg = 0.0f, su = 0.0f;
#pragma unroll
          for (int q = 0; q < kMWarps; ++q) {
            sg += rs[((q * 8 + gg) * V + v) * M];
            if (SWIGLU) su += rs[((q * 8 + gg) * V + v) * M + 1];
          }
          float os = 1.0f;
          if (p.rms) {
            float qq = 0.0f;
            for (int w = 0; w < kMWarps; ++w) qq += scratch[w * V + v];
            os = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(qq, static_cast<float>(p.cols)), p.rms_eps)));
          }
          float val = sg * os;
          if (SWIGLU) val = silu(val) * (su * os);
          if (p.residual) val += p.residual[v * p.y_stride + row];
          p.y[v * p.y_stride + row] = val;
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

template <int NVP, bool SW>
cudaError_t launch_multi(const MultiParams &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  auto k = gemv_q4k_tc_multi_kernel<NVP, SW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(kMThreads), smem, s, p);
}

}  // namespace

bool gemv_tc_multi_launch(const TcArgs &a, int nvec, const DeviceInfo &dev, cudaStream_t s, cudaError_t *err) {
  if (a.cols != 4096 || nvec < 3 || nvec > 8) return false;
  const int nvp = nvec <= 4 ? 2 : 4;
  MultiParams p;
  p.W = a.W;
  p.x = a.x;
  p.y = a.y;
  p.residual = a.residual;
  p.rows_out = a.rows_out;
  p.up_rows = a.swiglu ? a.rows_out : 0;
  p.row_bytes = a.row_bytes;
  p.cols = a.cols;
  p.nv = nvec;
  p.x_stride = a.x_stride;
  p.y_stride = a.y_stride;
  p.rms = a.rms;
  p.rms_eps = a.rms_eps;
  p.x_group = a.x_group;
  p.x_head_dim = a.x_head_dim;
  p.early_weights = a.early_weights;
  p.err = a.err;
  const bool sw = a.swiglu != 0;
  p.stage_bytes = static_cast<uint32_t>(8 * a.row_bytes * (sw ? 2 : 1));
  const int64_t g = std::min<int64_t>(dev.sm_count, (a.rows_out + 7) / 8);
  const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, g));
  const int64_t nst = ((a.rows_out + grid - 1) / grid + 7) / 8;
  int st = static_cast<int>(std::min<int64_t>(8, std::max<int64_t>(2, nst)));
  for (; st >= 2; --st)
    if (multi_layout(st, p.stage_bytes, nvp, sw).total <= static_cast<uint32_t>(dev.max_smem_optin)) break;
  if (st < 2) return false;
  p.stages = st;
  const uint32_t smem = multi_layout(st, p.stage_bytes, nvp, sw).total;
  cudaError_t e;
  if (nvp == 2) e = sw ? launch_multi<2, true>(p, grid, smem, s) : launch_multi<2, false>(p, grid, smem, s);
  else e = sw ? launch_multi<4, true>(p, grid, smem, s) : launch_multi<4, false>(p, grid, smem, s);
  *err = e;
  return true;
}

}  // namespace epq

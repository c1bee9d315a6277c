// Tensor-core expert kernels of the MoE layer for experts stored as Q2_K or
// Q6_K (one or two tokens per launch), for the Q2_K / Q6_K half of a mixed
// recipe (gate/up in one format, down in another), and for Q4_K experts
// under EPQ_TUNE_GEMV_ENGINE 3.
//
// "Flash-MoE：在笔记本上运行 397B 参数大模型", section "每层流水线": the selected
// experts' gate/up projections with SwiGLU, then the down projections and
// the weighted combine with the residual; the 2-bit experts of "smolmaxxing"
// and the Q6_K down projections of "EPM ... 記憶體怎麼配置的".  The products
// use the operand decode and block-diagonal MMA layout of k16_core.cuh (one
// warp per 16 rows, the two MMA vectors being the two tokens).  What differs
// from the dense kernel (gemv_k16.cu) is where rows and x come from:
//   * gate/up (moe_k16_gateup_kernel): every CTA first routes all tokens
//     from the router's logits (route_tokens; CTA 0 publishes the routing),
//     then converts x of the tokens into operand records.  The virtual row
//     groups (slot, 8 outputs) -- slots are the selected experts in
//     ascending order, then the shared expert -- are dealt round-robin over
//     the grid; a group is 8 gate rows and the matching 8 up rows of the
//     slot's matrix.  Each output writes h = silu(g r_t) * (u r_t) for every
//     entry (token t, choice k) of the slot and raises the max |h| word that
//     the CUDA-core down kernels read.
//   * down (moe_k16_down_kernel): the x operand of token t is the
//     concatenation over the slots of coef * h (coef = routing weight, or the
//     shared gate), zero where t does not use the slot, so one dot per row
//     and token is the whole combine: y = x + dot.  A row's superblocks are
//     walked across the slots' down matrices.
// Partial sums of the KP warps of a row group are added in k-part order
// through shared memory (deterministic).
#include <algorithm>

#include "k16_core.cuh"
#include "moe_common.cuh"
#include "moe_k16.cuh"

namespace epq {
namespace {

constexpr int kKWarps = 8;
constexpr int kKThreads = kKWarps * 32;

struct MkParams {
  MoeArgs a;
  int rg, kp;     // row groups per CTA, warps per row group
  int nsbx;       // superblocks of the x operand (gate/up H/256; down max slots * I/256)
  int want_hmax;  // gate/up: keep the max |h| words for a CUDA-core down kernel
  uint32_t meta_off, frag_off, ps_off, xsum_off, red_off, total;
};

__host__ __device__ inline uint32_t mk_al16(uint32_t v) { return (v + 15u) & ~15u; }

// meta | operand records (gate/up: shared with the routing scratch) | scales
// | sub-block sums of x | partial sums
inline void mk_layout(MkParams &p, int nv, bool gateup) {
  uint32_t o = 0;
  p.meta_off = o;
  o = mk_al16(o + 4u * meta_words(p.a.ntok, p.a.topk));
  p.frag_off = o;
  uint32_t fb = static_cast<uint32_t>(nv * p.nsbx) * k16::kSbFragBytes;
  if (gateup) fb = std::max<uint32_t>(fb, 4u * kSelScratchWords);
  o = mk_al16(o + fb);
  p.ps_off = o;
  o = mk_al16(o + 4u * nv * p.nsbx);
  p.xsum_off = o;
  o = mk_al16(o + 4u * nv * p.nsbx * 16);
  p.red_off = o;
  o = mk_al16(o + 4u * kKWarps * 16 * nv);
  p.total = o;
}

__device__ __forceinline__ float silu_k(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

// Choice k of token t in slot s, or -1 (a slot lists each token at most once).
__device__ __forceinline__ int entry_of(const Meta &m, int ntok, int s, int t) {
  const int c = m.cnt[s];
  for (int j = 0; j < c; ++j) {
    const int ent = m.list[s * ntok + j];
    if ((ent >> 5) == t) return ent & 31;
  }
  return -1;
}

// Row totals of a row group: butterflies over the 4 lanes of a row, then the
// warp's partials into red[warp][16 rows][NV].
template <int NV>
__device__ __forceinline__ void rows_to_smem(const float (&acc)[2][NV], float *red, int warp, int g, int t) {
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float s = acc[r][v];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (t == 0) red[(warp * 16 + g + 8 * r) * NV + v] = s;
    }
}

// ------------------------------------------------------------------ gate/up
template <int FMT, int NV, int ALIGN>
__global__ void __launch_bounds__(kKThreads, 1) moe_k16_gateup_kernel(const MkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const MoeArgs &a = p.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kq = warp % p.kp, rgl = warp / p.kp;
  const int I = a.I, nsb = a.H / 256;
  Meta m(smem + p.meta_off, a.ntok, a.topk);

  pdl_launch_dependents();
  pdl_wait();  // logits, x statistics and cleared max |h| words come from the router kernel
  m.clear(tid, kKThreads);
  __syncthreads();
  route_tokens(a, m, reinterpret_cast<uint32_t *>(smem + p.frag_off), blockIdx.x == 0);
  __syncthreads();  // the routing scratch becomes the operand records

  const int nact = *m.nact, nslots = *m.nslots;
  const int gps = I / 8;  // row groups (8 outputs) per slot
  const int total = nslots * gps;
  // a row group's rows and its first superblock's loads (issued for the
  // first group before x is converted, so that they overlap)
  k16::RowOps<FMT> cl, ch, nl, nh;
  const uint8_t *row_lo = nullptr, *row_hi = nullptr;
  bool work = false;
  auto start = [&](int b0) {
    const int vg = b0 + rgl;
    work = vg < total && kq < nsb;
    if (!work) return;
    const int s = vg / gps, i = (vg - s * gps) * 8 + g;
    const int e = s < nact ? m.active[s] : -1;
    const uint8_t *Wm = e >= 0 ? a.gate_up + static_cast<int64_t>(e) * a.gu_stride : a.sh_gate_up;
    row_lo = Wm + static_cast<int64_t>(i) * a.gu_row_bytes;
    row_hi = Wm + static_cast<int64_t>(I + i) * a.gu_row_bytes;
    k16::load_ops<FMT, ALIGN>(cl, row_lo, nsb, kq, t);
    k16::load_ops<FMT, ALIGN>(ch, row_hi, nsb, kq, t);
  };
  start(blockIdx.x * p.rg);

  // x of the tokens (vector v = token v) into operand records
  float *ps_s = reinterpret_cast<float *>(smem + p.ps_off);
  float *xsum_s = reinterpret_cast<float *>(smem + p.xsum_off);
  for (int u = warp; u < NV * nsb; u += kKWarps) {
    const int v = u / nsb, b = u - v * nsb;
    float xv[8];
    if (v < a.ntok) {
      const float *xr = a.x + static_cast<int64_t>(v) * a.H + b * 256 + 8 * lane;
      const float4 x0 = *reinterpret_cast<const float4 *>(xr), x1 = *reinterpret_cast<const float4 *>(xr + 4);
      xv[0] = x0.x, xv[1] = x0.y, xv[2] = x0.z, xv[3] = x0.w, xv[4] = x1.x, xv[5] = x1.y, xv[6] = x1.z, xv[7] = x1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[e] = 0.0f;
    }
    uint8_t *fr = smem + p.frag_off + static_cast<uint32_t>(v * nsb + b) * k16::kSbFragBytes;
    const float mx = warp_absmax(k16::lane_absmax(xv));
    const int ex = FMT == EPQ_Q4_K ? k16::stage_superblock_q4k(xv, mx, fr, lane, xsum_s + (v * nsb + b) * 16)
                                   : k16::stage_superblock(xv, mx, fr, lane, xsum_s + (v * nsb + b) * 16);
    if (lane == 0) ps_s[v * nsb + b] = k16::sum_scale<FMT>(ex);
  }
  __syncthreads();

  const uint8_t *frag0 = smem + p.frag_off + k16::lane_slot(lane);
  const uint32_t vstride = static_cast<uint32_t>(nsb) * k16::kSbFragBytes;
  float *red = reinterpret_cast<float *>(smem + p.red_off);
#pragma unroll 1
  for (int base = blockIdx.x * p.rg; base < total; base += gridDim.x * p.rg) {
    if (base != static_cast<int>(blockIdx.x) * p.rg) start(base);
    float acc[2][NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[0][v] = acc[1][v] = 0.0f;
    if (work) {
      int sb = kq;
      for (;;) {
        const int nx = sb + p.kp;
        if (nx < nsb) {
          k16::load_ops<FMT, ALIGN>(nl, row_lo, nsb, nx, t);
          k16::load_ops<FMT, ALIGN>(nh, row_hi, nsb, nx, t);
        }
        float ps[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) ps[v] = ps_s[v * nsb + sb];
        k16::superblock<FMT, NV>(cl, ch, frag0 + sb * k16::kSbFragBytes, vstride, ps,
                                 xsum_s + sb * 16, nsb * 16, t, acc);
        if (nx >= nsb) break;
        sb = nx;
        cl = nl;
        ch = nh;
      }
    }
    rows_to_smem<NV>(acc, red, warp, g, t);
    __syncthreads();
    for (int idx = tid; idx < p.rg * 8 * NV; idx += kKThreads) {
      const int v = idx % NV, o = (idx / NV) % 8, gl = idx / (8 * NV);
      const int vg2 = base + gl;
      if (v >= a.ntok || vg2 >= total) continue;
      const int s = vg2 / gps, i = (vg2 - s * gps) * 8 + o;
      const int k = entry_of(m, a.ntok, s, v);
      if (k < 0) continue;
      float gs = 0.0f, us = 0.0f;
      for (int w = 0; w < p.kp; ++w) {
        const float *rr = red + ((gl * p.kp + w) * 16) * NV;
        gs += rr[o * NV + v];
        us += rr[(o + 8) * NV + v];
      }
      const float r = m.rms[v];
      const float hv = silu_k(gs * r) * (us * r);
      const int hs = v * (a.topk + 1) + k;
      a.h[static_cast<int64_t>(hs) * I + i] = hv;
      if (p.want_hmax) atomicMax(a.hmax + hs, __float_as_uint(fabsf(hv)));
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ down + combine
template <int FMT, int NV, int ALIGN>
__global__ void __launch_bounds__(kKThreads, 1) moe_k16_down_kernel(const MkParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const MoeArgs &a = p.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kq = warp % p.kp, rgl = warp / p.kp;
  const int I = a.I, H = a.H, nsbI = I / 256;
  Meta m(smem + p.meta_off, a.ntok, a.topk);

  pdl_launch_dependents();
  pdl_wait();  // h and the routing come from the gate/up kernel
  load_meta(a, m, tid, kKThreads);
  __syncthreads();
  const int nact = *m.nact, nslots = *m.nslots;
  const int nvsb = nslots * nsbI;  // <= p.nsbx
  const int total = (H + 15) / 16;
  auto row_base = [&](int s) -> const uint8_t * {
    const int e = s < nact ? m.active[s] : -1;
    return e >= 0 ? a.down + static_cast<int64_t>(e) * a.dn_stride : a.sh_down;
  };
  // a row group's rows and its first superblock's loads (issued for the
  // first group before h is staged, so that they overlap)
  k16::RowOps<FMT> cl, ch, nl, nh;
  int64_t r_lo = 0, r_hi = 0;
  bool work = false;
  auto start = [&](int b0) {
    const int vg = b0 + rgl;
    work = vg < total && kq < nvsb;
    if (!work) return;
    r_lo = min(vg * 16 + g, H - 1);
    r_hi = min(vg * 16 + g + 8, H - 1);
    const int s0 = kq / nsbI;
    const uint8_t *Wm = row_base(s0);
    k16::load_ops<FMT, ALIGN>(cl, Wm + r_lo * a.dn_row_bytes, nsbI, kq - s0 * nsbI, t);
    k16::load_ops<FMT, ALIGN>(ch, Wm + r_hi * a.dn_row_bytes, nsbI, kq - s0 * nsbI, t);
  };
  start(blockIdx.x * p.rg);

  // x operand of token v: coef * h over the slots, zero where v is absent;
  // the h loads of kBatch units are issued before any is converted
  float *ps_s = reinterpret_cast<float *>(smem + p.ps_off);
  float *xsum_s = reinterpret_cast<float *>(smem + p.xsum_off);
  constexpr int kBatch = 3;
  const int nunits = NV * nvsb;
  for (int u0 = warp; u0 < nunits; u0 += kKWarps * kBatch) {
    float xv[kBatch][8];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int u = u0 + kKWarps * j;
      const int v = u / nvsb, b = u - v * nvsb;
      const int s = b / nsbI, lsb = b - s * nsbI;
      const int k = u < nunits && v < a.ntok ? entry_of(m, a.ntok, s, v) : -1;
      if (k >= 0) {
        const float coef = k == a.topk ? m.gs[v] : m.w[v * a.topk + k];
        const float *hr = a.h + static_cast<int64_t>(v * (a.topk + 1) + k) * I + lsb * 256 + 8 * lane;
        const float4 h0 = __ldcg(reinterpret_cast<const float4 *>(hr));
        const float4 h1 = __ldcg(reinterpret_cast<const float4 *>(hr + 4));
        xv[j][0] = coef * h0.x, xv[j][1] = coef * h0.y, xv[j][2] = coef * h0.z, xv[j][3] = coef * h0.w;
        xv[j][4] = coef * h1.x, xv[j][5] = coef * h1.y, xv[j][6] = coef * h1.z, xv[j][7] = coef * h1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[j][e] = 0.0f;
      }
    }
    float mx[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) mx[j] = warp_absmax(k16::lane_absmax(xv[j]));
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int u = u0 + kKWarps * j;
      if (u >= nunits) break;  // warp-uniform
      const int v = u / nvsb, b = u - v * nvsb;
      uint8_t *fr = smem + p.frag_off + static_cast<uint32_t>(v * p.nsbx + b) * k16::kSbFragBytes;
      const int ex = FMT == EPQ_Q4_K
                         ? k16::stage_superblock_q4k(xv[j], mx[j], fr, lane, xsum_s + (v * p.nsbx + b) * 16)
                         : k16::stage_superblock(xv[j], mx[j], fr, lane, xsum_s + (v * p.nsbx + b) * 16);
      if (lane == 0) ps_s[v * p.nsbx + b] = k16::sum_scale<FMT>(ex);
    }
  }
  __syncthreads();

  const uint8_t *frag0 = smem + p.frag_off + k16::lane_slot(lane);
  const uint32_t vstride = static_cast<uint32_t>(p.nsbx) * k16::kSbFragBytes;
  float *red = reinterpret_cast<float *>(smem + p.red_off);
#pragma unroll 1
  for (int base = blockIdx.x * p.rg; base < total; base += gridDim.x * p.rg) {
    if (base != static_cast<int>(blockIdx.x) * p.rg) start(base);
    float acc[2][NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[0][v] = acc[1][v] = 0.0f;
    if (work) {
      int sb = kq;
      int s = sb / nsbI, lsb = sb - s * nsbI;
      for (;;) {
        const int nx = sb + p.kp;
        int ns = s, nlsb = lsb + p.kp;
        while (nlsb >= nsbI) {
          nlsb -= nsbI;
          ++ns;
        }
        if (nx < nvsb) {
          const uint8_t *Wn = row_base(ns);
          k16::load_ops<FMT, ALIGN>(nl, Wn + r_lo * a.dn_row_bytes, nsbI, nlsb, t);
          k16::load_ops<FMT, ALIGN>(nh, Wn + r_hi * a.dn_row_bytes, nsbI, nlsb, t);
        }
        float ps[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) ps[v] = ps_s[v * p.nsbx + sb];
        k16::superblock<FMT, NV>(cl, ch, frag0 + sb * k16::kSbFragBytes, vstride, ps,
                                 xsum_s + sb * 16, p.nsbx * 16, t, acc);
        if (nx >= nvsb) break;
        sb = nx;
        s = ns;
        lsb = nlsb;
        cl = nl;
        ch = nh;
      }
    }
    rows_to_smem<NV>(acc, red, warp, g, t);
    __syncthreads();
    for (int idx = tid; idx < p.rg * 16 * NV; idx += kKThreads) {
      const int v = idx % NV, o = (idx / NV) % 16, gl = idx / (16 * NV);
      const int r = (base + gl) * 16 + o;
      if (v >= a.ntok || r >= H) continue;
      float d = 0.0f;
      for (int w = 0; w < p.kp; ++w) d += red[((gl * p.kp + w) * 16 + o) * NV + v];
      const int64_t off = static_cast<int64_t>(v) * H + r;
      a.y[off] = a.x[off] + d;
    }
    __syncthreads();
  }
}

template <typename K>
cudaError_t mk_launch(K kernel, const MkParams &p, unsigned grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(p.total));
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(grid), dim3(kKThreads), p.total, s, p);
}

// Rows of `row_bytes` bytes: 16-, 4- or 2-byte aligned starts.
inline int row_align(int64_t row_bytes, int64_t stride) {
  const int64_t v = row_bytes | stride;
  return v % 16 == 0 ? 16 : (v % 4 == 0 ? 4 : 2);
}

template <int FMT, int NV>
cudaError_t gateup_by_align(const MkParams &p, int align, unsigned grid, cudaStream_t s) {
  if (align == 16) return mk_launch(moe_k16_gateup_kernel<FMT, NV, 16>, p, grid, s);
  if (align == 4) return mk_launch(moe_k16_gateup_kernel<FMT, NV, 4>, p, grid, s);
  if constexpr (FMT == EPQ_Q6_K) return mk_launch(moe_k16_gateup_kernel<FMT, NV, 2>, p, grid, s);
  return cudaErrorInvalidValue;
}

template <int FMT, int NV>
cudaError_t down_by_align(const MkParams &p, int align, unsigned grid, cudaStream_t s) {
  if (align == 16) return mk_launch(moe_k16_down_kernel<FMT, NV, 16>, p, grid, s);
  if (align == 4) return mk_launch(moe_k16_down_kernel<FMT, NV, 4>, p, grid, s);
  if constexpr (FMT == EPQ_Q6_K) return mk_launch(moe_k16_down_kernel<FMT, NV, 2>, p, grid, s);
  return cudaErrorInvalidValue;
}

// RG row groups per CTA: the largest power of two <= 8 that still gives
// every SM two CTAs' worth of groups.
int pick_rg(int64_t groups, int sm_count) {
  int rg = 8;
  while (rg > 1 && (groups + rg - 1) / rg < 2ll * sm_count) rg >>= 1;
  return rg;
}

}  // namespace

bool moe_k16_fits(const MoeArgs &a, int max_slots, bool gateup, bool down, const DeviceInfo &dev) {
  if (a.ntok < 1 || a.ntok > 2) return false;
  MkParams p;
  p.a = a;
  if (gateup) {
    p.nsbx = a.H / 256;
    mk_layout(p, a.ntok, true);
    if (p.total > static_cast<uint32_t>(dev.max_smem_optin)) return false;
  }
  if (down) {
    p.nsbx = max_slots * (a.I / 256);
    mk_layout(p, a.ntok, false);
    if (p.total > static_cast<uint32_t>(dev.max_smem_optin)) return false;
  }
  return true;
}

cudaError_t moe_k16_gateup_launch(epq_fmt fmt, const MoeArgs &a, int max_slots, bool want_hmax,
                                  const DeviceInfo &dev, cudaStream_t s) {
  MkParams p;
  p.a = a;
  p.nsbx = a.H / 256;
  p.want_hmax = want_hmax ? 1 : 0;
  mk_layout(p, a.ntok, true);
  const int64_t groups = static_cast<int64_t>(max_slots) * (a.I / 8);
  p.rg = pick_rg(groups, dev.sm_count);
  p.kp = kKWarps / p.rg;
  const unsigned grid = static_cast<unsigned>(
      std::max<int64_t>(1, std::min<int64_t>((groups + p.rg - 1) / p.rg, 2ll * dev.sm_count)));
  const int align = row_align(a.gu_row_bytes, a.gu_stride);
  if (fmt == EPQ_Q4_K)  // 144-byte superblocks: rows and (16-byte) strides keep 16-byte alignment
    return a.ntok == 1 ? mk_launch(moe_k16_gateup_kernel<EPQ_Q4_K, 1, 16>, p, grid, s)
                       : mk_launch(moe_k16_gateup_kernel<EPQ_Q4_K, 2, 16>, p, grid, s);
  if (fmt == EPQ_Q2_K)
    return a.ntok == 1 ? gateup_by_align<EPQ_Q2_K, 1>(p, align, grid, s) : gateup_by_align<EPQ_Q2_K, 2>(p, align, grid, s);
  return a.ntok == 1 ? gateup_by_align<EPQ_Q6_K, 1>(p, align, grid, s) : gateup_by_align<EPQ_Q6_K, 2>(p, align, grid, s);
}

cudaError_t moe_k16_down_launch(epq_fmt fmt, const MoeArgs &a, int max_slots, const DeviceInfo &dev,
                                cudaStream_t s) {
  MkParams p;
  p.a = a;
  p.nsbx = max_slots * (a.I / 256);
  p.want_hmax = 0;
  mk_layout(p, a.ntok, false);
  const int64_t groups = (a.H + 15) / 16;
  p.rg = pick_rg(groups, dev.sm_count);
  p.kp = kKWarps / p.rg;
  const unsigned grid = static_cast<unsigned>(
      std::max<int64_t>(1, std::min<int64_t>((groups + p.rg - 1) / p.rg, 2ll * dev.sm_count)));
  const int align = row_align(a.dn_row_bytes, a.dn_stride);
  if (fmt == EPQ_Q4_K)
    return a.ntok == 1 ? mk_launch(moe_k16_down_kernel<EPQ_Q4_K, 1, 16>, p, grid, s)
                       : mk_launch(moe_k16_down_kernel<EPQ_Q4_K, 2, 16>, p, grid, s);
  if (fmt == EPQ_Q2_K)
    return a.ntok == 1 ? down_by_align<EPQ_Q2_K, 1>(p, align, grid, s) : down_by_align<EPQ_Q2_K, 2>(p, align, grid, s);
  return a.ntok == 1 ? down_by_align<EPQ_Q6_K, 1>(p, align, grid, s) : down_by_align<EPQ_Q6_K, 2>(p, align, grid, s);
}

}  // namespace epq

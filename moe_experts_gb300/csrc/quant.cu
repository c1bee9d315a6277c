// Block packer (epq_quantize) and unpacker (epq_dequantize).
//
// Formats of "端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch", section
// "GGUF 的量化格式".  Every decision is taken in IEEE float32 with the
// explicit round-to-nearest intrinsics (no contraction, no fast-math), so
// codes and factors are bit-exact with the CPU oracle:
//   * Q8_0  d = f16(amax / 127), q = clamp(rint(x / d), -127, 127)
//   * Q4_0  d = f16(v* / -8) with v* the first value of largest magnitude,
//           n = clamp(rint(x / d), -8, 7) + 8
//   * Q4_1  d = f16((max - min) / 15), m = f16(min),
//           n = clamp(rint((x - m) / d), 0, 15)
//   * Q4_K  per sub-block lo = min(min x, 0), sc = (max x - lo) / 15,
//           mn = 0 - lo; d = f16(max sc / 63), dmin = f16(max mn / 63);
//           c = clamp(rint(sc / d), 1, 63) (1 when d = 0),
//           k = clamp(rint(mn / dmin), 0, 63) (0 when dmin = 0);
//           S = d*c, M = dmin*k, n = clamp(rint((x + M) / S), 0, 15)
//   * Q2_K  per 16-weight sub-block lo = min(min x, 0), st = (max x - lo) / 3,
//           lift = 0 - lo; d = f16(max st / 15), dmin = f16(max lift / 15);
//           c = clamp(rint(st / d), 1, 15) (1 when d = 0),
//           k = clamp(rint(lift / dmin), 0, 15); n = clamp(rint((x + M) / S), 0, 3)
//   * Q6_K  per sub-block scale = v* / -32 (v* its first value of largest
//           magnitude); d = f16(max |scale| / 127), c = clamp(rint(scale / d),
//           -127, 127); m = clamp(rint(x / S), -32, 31), stored as u = m + 32
// Zero factors give zero codes; inputs pass through x + 0 so that -0 is +0.
//
// One warp handles one block (32 weights: one weight per lane) or one
// superblock (256 weights: eight consecutive weights per lane; lanes 4s..4s+3
// form Q4_K sub-block s, lanes 2s, 2s+1 form Q2_K / Q6_K sub-block s).  The
// Q2_K / Q6_K rows are stored plane by plane; a 2-bit field of sub-block
// position i sits at bit kField2[i] of the sub-block's 32-bit word.
#include "common.cuh"

namespace epq {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float clampf(float v, float lo, float hi) { return fminf(fmaxf(v, lo), hi); }

// rint(num / den) clamped to [lo, hi]; 0 when den == 0.
__device__ __forceinline__ float code_of(float num, float den, float lo, float hi) {
  if (den == 0.0f) return 0.0f;
  return clampf(rintf(__fdiv_rn(num, den)), lo, hi);
}

__device__ __forceinline__ unsigned short f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }

// ---------------------------------------------------------------- 32-weight formats
template <int FMT>
__global__ void __launch_bounds__(kThreads) quantize32_kernel(const float *__restrict__ W, uint8_t *__restrict__ out,
                                                              int64_t nblocks) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t b = warp; b < nblocks; b += nwarps) {
    const float x = __fadd_rn(W[b * 32 + lane], 0.0f);
    if (FMT == EPQ_Q8_0) {
      uint8_t *o = out + b * 34;
      const float amax = warp_max_all(fabsf(x));
      const unsigned short dh = f16_bits(__fdiv_rn(amax, 127.0f));
      const float dF = half_bits_to_float(dh);
      const int q = static_cast<int>(code_of(x, dF, -127.0f, 127.0f));
      o[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
      if (lane == 0) *reinterpret_cast<unsigned short *>(o) = dh;
    } else if (FMT == EPQ_Q4_0) {
      uint8_t *o = out + b * 18;
      // first index of the largest magnitude
      float a = fabsf(x);
      int idx = lane;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float a2 = __shfl_xor_sync(kFull, a, off);
        const int i2 = __shfl_xor_sync(kFull, idx, off);
        if (a2 > a || (a2 == a && i2 < idx)) {
          a = a2;
          idx = i2;
        }
      }
      const float vmax = __shfl_sync(kFull, x, idx);
      const unsigned short dh = f16_bits(__fdiv_rn(vmax, -8.0f));
      const float dF = half_bits_to_float(dh);
      const int n = static_cast<int>(code_of(x, dF, -8.0f, 7.0f)) + 8;
      const int n_hi = __shfl_down_sync(kFull, n, 1);
      if ((lane & 1) == 0) o[2 + (lane >> 1)] = static_cast<uint8_t>(n | (n_hi << 4));
      if (lane == 0) *reinterpret_cast<unsigned short *>(o) = dh;
    } else {  // Q4_1
      uint8_t *o = out + b * 20;
      const float lo = warp_min_all(x);
      const float hi = warp_max_all(x);
      const unsigned short dh = f16_bits(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
      const unsigned short mh = f16_bits(lo);
      const float dF = half_bits_to_float(dh), mF = half_bits_to_float(mh);
      const int n = static_cast<int>(code_of(__fsub_rn(x, mF), dF, 0.0f, 15.0f));
      const int n_hi = __shfl_down_sync(kFull, n, 1);
      if ((lane & 1) == 0) o[4 + (lane >> 1)] = static_cast<uint8_t>(n | (n_hi << 4));
      if (lane == 0) *reinterpret_cast<uint32_t *>(o) = static_cast<uint32_t>(dh) | (static_cast<uint32_t>(mh) << 16);
    }
  }
}

// ---------------------------------------------------------------- Q4_K
__global__ void __launch_bounds__(kThreads) quantize_q4k_kernel(const float *__restrict__ W, uint8_t *__restrict__ out,
                                                                int64_t nsuper) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t b = warp; b < nsuper; b += nwarps) {
    const float4 *src = reinterpret_cast<const float4 *>(W + b * 256 + lane * 8);
    const float4 p0 = src[0], p1 = src[1];
    float x[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    float mn8 = 0.0f, mx8 = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      x[t] = __fadd_rn(x[t], 0.0f);
      mn8 = t == 0 ? x[t] : fminf(mn8, x[t]);
      mx8 = t == 0 ? x[t] : fmaxf(mx8, x[t]);
    }
    // sub-block (4 lanes) min / max
    mn8 = fminf(mn8, __shfl_xor_sync(kFull, mn8, 1));
    mn8 = fminf(mn8, __shfl_xor_sync(kFull, mn8, 2));
    mx8 = fmaxf(mx8, __shfl_xor_sync(kFull, mx8, 1));
    mx8 = fmaxf(mx8, __shfl_xor_sync(kFull, mx8, 2));
    const float lo = fminf(mn8, 0.0f);
    const float sc = __fdiv_rn(__fsub_rn(mx8, lo), 15.0f);
    const float mn = __fsub_rn(0.0f, lo);
    float maxsc = sc, maxmn = mn;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      maxsc = fmaxf(maxsc, __shfl_xor_sync(kFull, maxsc, off));
      maxmn = fmaxf(maxmn, __shfl_xor_sync(kFull, maxmn, off));
    }
    const unsigned short dh = f16_bits(__fdiv_rn(maxsc, 63.0f));
    const unsigned short dminh = f16_bits(__fdiv_rn(maxmn, 63.0f));
    const float dF = half_bits_to_float(dh), dminF = half_bits_to_float(dminh);
    const int c = dF == 0.0f ? 1 : static_cast<int>(code_of(sc, dF, 1.0f, 63.0f));
    const int k = static_cast<int>(code_of(mn, dminF, 0.0f, 63.0f));
    const float S = __fmul_rn(dF, static_cast<float>(c));
    const float M = __fmul_rn(dminF, static_cast<float>(k));
    uint32_t packed = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int n = static_cast<int>(code_of(__fadd_rn(x[t], M), S, 0.0f, 15.0f));
      packed |= static_cast<uint32_t>(n) << (4 * t);
    }
    uint8_t *o = out + b * 144;
    reinterpret_cast<uint32_t *>(o + 16)[lane] = packed;
    // gather the 16 six-bit codes (lanes 0, 4, ..., 28 hold sub-blocks 0..7)
    uint64_t lo64 = 0;
    uint32_t hi32 = 0;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint64_t cs = static_cast<uint64_t>(__shfl_sync(kFull, c, 4 * s));
      const uint64_t ks = static_cast<uint64_t>(__shfl_sync(kFull, k, 4 * s));
      lo64 |= cs << (6 * s);  // c codes occupy bits 0..47
      const int kb = 48 + 6 * s;  // k codes occupy bits 48..95
      if (kb + 6 <= 64) {
        lo64 |= ks << kb;
      } else if (kb >= 64) {
        hi32 |= static_cast<uint32_t>(ks) << (kb - 64);
      } else {
        lo64 |= ks << kb;
        hi32 |= static_cast<uint32_t>(ks >> (64 - kb));
      }
    }
    if (lane == 0) {
      uint32_t *h = reinterpret_cast<uint32_t *>(o);
      h[0] = static_cast<uint32_t>(dh) | (static_cast<uint32_t>(dminh) << 16);
      h[1] = static_cast<uint32_t>(lo64);
      h[2] = static_cast<uint32_t>(lo64 >> 32);
      h[3] = hi32;
    }
  }
}

// ---------------------------------------------------------------- Q2_K / Q6_K
__constant__ int kField2[16] = {4, 8, 6, 10, 20, 24, 22, 26, 28, 0, 30, 2, 12, 16, 14, 18};

// Byte offsets of superblock sb's plane entries in a row of nsb superblocks.
struct KPlanes {
  int64_t a, b, c, d;
};
__device__ __forceinline__ KPlanes k_planes(int fmt, int64_t nsb, int64_t sb) {
  if (fmt == EPQ_Q2_K) return {64 * sb, 64 * nsb + 16 * sb, 80 * nsb + 4 * sb, 0};
  return {128 * sb, 128 * nsb + 64 * sb, 192 * nsb + 16 * sb, 208 * nsb + 2 * sb};
}

// A Q6_K row of an odd number of superblocks is only 2-byte aligned, so the
// plane entries are moved byte by byte.
__device__ __forceinline__ void put_u32(uint8_t *p, uint32_t v) {
#pragma unroll
  for (int b = 0; b < 4; ++b) p[b] = static_cast<uint8_t>(v >> (8 * b));
}
__device__ __forceinline__ uint32_t get_u32(const uint8_t *p) {
  return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) | (static_cast<uint32_t>(p[2]) << 16) |
         (static_cast<uint32_t>(p[3]) << 24);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) quantize_k16_kernel(const float *__restrict__ W, uint8_t *__restrict__ out,
                                                                int64_t nsuper, int64_t nsb, int64_t row_bytes) {
  const int lane = threadIdx.x & 31;
  const int h = lane & 1;  // half of the sub-block: positions 8h..8h+7
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t b = warp; b < nsuper; b += nwarps) {
    const float4 *src = reinterpret_cast<const float4 *>(W + b * 256 + lane * 8);
    const float4 p0 = src[0], p1 = src[1];
    float x[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) x[t] = __fadd_rn(x[t], 0.0f);
    uint8_t *row = out + (b / nsb) * row_bytes;
    const KPlanes pl = k_planes(FMT, nsb, b % nsb);
    uint32_t word = 0;
    if (FMT == EPQ_Q2_K) {
      float mn = x[0], mx = x[0];
#pragma unroll
      for (int t = 1; t < 8; ++t) {
        mn = fminf(mn, x[t]);
        mx = fmaxf(mx, x[t]);
      }
      mn = fminf(mn, __shfl_xor_sync(kFull, mn, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      const float lo = fminf(mn, 0.0f);
      const float st = __fdiv_rn(__fsub_rn(mx, lo), 3.0f);
      const float lift = __fsub_rn(0.0f, lo);
      float top_st = st, top_lift = lift;
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) {
        top_st = fmaxf(top_st, __shfl_xor_sync(kFull, top_st, off));
        top_lift = fmaxf(top_lift, __shfl_xor_sync(kFull, top_lift, off));
      }
      const unsigned short dh = f16_bits(__fdiv_rn(top_st, 15.0f));
      const unsigned short mh = f16_bits(__fdiv_rn(top_lift, 15.0f));
      const float dF = half_bits_to_float(dh), mF = half_bits_to_float(mh);
      const int c = dF == 0.0f ? 1 : static_cast<int>(code_of(st, dF, 1.0f, 15.0f));
      const int k = static_cast<int>(code_of(lift, mF, 0.0f, 15.0f));
      const float S = __fmul_rn(dF, static_cast<float>(c));
      const float M = __fmul_rn(mF, static_cast<float>(k));
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t n = static_cast<uint32_t>(code_of(__fadd_rn(x[t], M), S, 0.0f, 3.0f));
        word |= n << kField2[8 * h + t];
      }
      word |= __shfl_xor_sync(kFull, word, 1);
      if (h == 0) {
        put_u32(row + pl.a + 4 * (lane >> 1), word);
        row[pl.b + (lane >> 1)] = static_cast<uint8_t>(c | (k << 4));
      }
      if (lane == 0) put_u32(row + pl.c, static_cast<uint32_t>(dh) | (static_cast<uint32_t>(mh) << 16));
    } else {  // Q6_K
      // first index of the largest magnitude in the sub-block
      float a = fabsf(x[0]);
      int idx = 0;
#pragma unroll
      for (int t = 1; t < 8; ++t)
        if (fabsf(x[t]) > a) {
          a = fabsf(x[t]);
          idx = t;
        }
      float peak = x[idx];
      const float a2 = __shfl_xor_sync(kFull, a, 1);
      const float peak2 = __shfl_xor_sync(kFull, peak, 1);
      // the even lane holds the lower positions: it wins ties
      if (h == 0 ? a2 > a : a2 >= a) peak = peak2;
      const float scale = __fdiv_rn(peak, -32.0f);
      float top = fabsf(scale);
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) top = fmaxf(top, __shfl_xor_sync(kFull, top, off));
      const unsigned short dh = f16_bits(__fdiv_rn(top, 127.0f));
      const float dF = half_bits_to_float(dh);
      const int c = static_cast<int>(code_of(scale, dF, -127.0f, 127.0f));
      const float S = __fmul_rn(dF, static_cast<float>(c));
      uint32_t nib = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t u = static_cast<uint32_t>(static_cast<int>(code_of(x[t], S, -32.0f, 31.0f)) + 32);
        nib |= (u & 15u) << (4 * t);
        word |= (u >> 4) << kField2[8 * h + t];
      }
      word |= __shfl_xor_sync(kFull, word, 1);
      put_u32(row + pl.a + 4 * lane, nib);
      if (h == 0) {
        put_u32(row + pl.b + 4 * (lane >> 1), word);
        row[pl.c + (lane >> 1)] = static_cast<uint8_t>(static_cast<int8_t>(c));
      }
      if (lane == 0) {
        row[pl.d] = static_cast<uint8_t>(dh);
        row[pl.d + 1] = static_cast<uint8_t>(dh >> 8);
      }
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) dequantize_k16_kernel(const uint8_t *__restrict__ in,
                                                                  float *__restrict__ W, int64_t nsuper, int64_t nsb,
                                                                  int64_t row_bytes) {
  const int lane = threadIdx.x & 31;
  const int h = lane & 1, s = lane >> 1;
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t b = warp; b < nsuper; b += nwarps) {
    const uint8_t *row = in + (b / nsb) * row_bytes;
    const KPlanes pl = k_planes(FMT, nsb, b % nsb);
    float v[8];
    if (FMT == EPQ_Q2_K) {
      const uint32_t word = get_u32(row + pl.a + 4 * s);
      const uint32_t cb = row[pl.b + s];
      const uint32_t f = get_u32(row + pl.c);
      const float S = __fmul_rn(half_bits_to_float(f), static_cast<float>(cb & 15u));
      const float M = __fmul_rn(half_bits_to_float(f >> 16), static_cast<float>(cb >> 4));
#pragma unroll
      for (int t = 0; t < 8; ++t)
        v[t] = __fsub_rn(__fmul_rn(static_cast<float>((word >> kField2[8 * h + t]) & 3u), S), M);
    } else {
      const uint32_t nib = get_u32(row + pl.a + 4 * lane);
      const uint32_t word = get_u32(row + pl.b + 4 * s);
      const int c = static_cast<int8_t>(row[pl.c + s]);
      const uint32_t dh = static_cast<uint32_t>(row[pl.d]) | (static_cast<uint32_t>(row[pl.d + 1]) << 8);
      const float S = __fmul_rn(half_bits_to_float(dh), static_cast<float>(c));
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int u = static_cast<int>(((nib >> (4 * t)) & 15u) | (((word >> kField2[8 * h + t]) & 3u) << 4));
        v[t] = __fmul_rn(static_cast<float>(u - 32), S);
      }
    }
    float4 *dst = reinterpret_cast<float4 *>(W + b * 256 + lane * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// ---------------------------------------------------------------- dequantize
template <int FMT>
__global__ void __launch_bounds__(kThreads) dequantize32_kernel(const uint8_t *__restrict__ in, float *__restrict__ W,
                                                                int64_t nblocks) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t b = warp; b < nblocks; b += nwarps) {
    float v;
    if (FMT == EPQ_Q8_0) {
      const uint8_t *blk = in + b * 34;
      const float dF = half_bits_to_float(*reinterpret_cast<const unsigned short *>(blk));
      v = __fmul_rn(dF, static_cast<float>(static_cast<int8_t>(blk[2 + lane])));
    } else if (FMT == EPQ_Q4_0) {
      const uint8_t *blk = in + b * 18;
      const float dF = half_bits_to_float(*reinterpret_cast<const unsigned short *>(blk));
      const int byte = blk[2 + (lane >> 1)];
      const int n = (lane & 1) ? (byte >> 4) : (byte & 15);
      v = __fmul_rn(dF, static_cast<float>(n - 8));
    } else {
      const uint8_t *blk = in + b * 20;
      const uint32_t dm = *reinterpret_cast<const uint32_t *>(blk);
      const float dF = half_bits_to_float(dm), mF = half_bits_to_float(dm >> 16);
      const int byte = blk[4 + (lane >> 1)];
      const int n = (lane & 1) ? (byte >> 4) : (byte & 15);
      v = __fadd_rn(__fmul_rn(static_cast<float>(n), dF), mF);
    }
    W[b * 32 + lane] = v;
  }
}

__global__ void __launch_bounds__(kThreads) dequantize_q4k_kernel(const uint8_t *__restrict__ in,
                                                                  float *__restrict__ W, int64_t nsuper) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int s = lane >> 2;
  for (int64_t b = warp; b < nsuper; b += nwarps) {
    const uint32_t *h = reinterpret_cast<const uint32_t *>(in + b * 144);
    const uint32_t w0 = h[0], w1 = h[1], w2 = h[2], w3 = h[3];
    const uint64_t lo64 = static_cast<uint64_t>(w1) | (static_cast<uint64_t>(w2) << 32);
    const int c = static_cast<int>((lo64 >> (6 * s)) & 63u);
    const int kb = 48 + 6 * s;
    int k;
    if (kb + 6 <= 64) {
      k = static_cast<int>((lo64 >> kb) & 63u);
    } else if (kb >= 64) {
      k = static_cast<int>((w3 >> (kb - 64)) & 63u);
    } else {
      k = static_cast<int>(((lo64 >> kb) | (static_cast<uint64_t>(w3) << (64 - kb))) & 63u);
    }
    const float S = __fmul_rn(half_bits_to_float(w0), static_cast<float>(c));
    const float M = __fmul_rn(half_bits_to_float(w0 >> 16), static_cast<float>(k));
    const uint32_t q = h[4 + lane];
    float v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) v[t] = __fsub_rn(__fmul_rn(static_cast<float>((q >> (4 * t)) & 15u), S), M);
    float4 *dst = reinterpret_cast<float4 *>(W + b * 256 + lane * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

epq_status check_pack_args(epq_fmt fmt, const void *a, const void *b, int64_t rows, int64_t cols, DeviceInfo *dev) {
  if (epq_block_weights(fmt) < 0) return EPQ_ERR_FORMAT;
  if (!a || !b) return EPQ_ERR_ARG;
  if (rows < 1 || cols < 256 || cols % 256) return EPQ_ERR_SHAPE;
  if (!aligned16(a) || !aligned16(b)) return EPQ_ERR_ALIGN;
  if (!current_device(dev) || dev->major * 10 + dev->minor < 100) return EPQ_ERR_DEVICE;
  return EPQ_OK;
}

unsigned grid_for(int64_t units_per_warp_items, const DeviceInfo &dev) {
  const int64_t warps = units_per_warp_items;
  int64_t blocks = (warps + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace
}  // namespace epq

using namespace epq;

extern "C" epq_status epq_quantize(epq_fmt fmt, const float *W, int64_t rows, int64_t cols, void *blocks,
                                   epq_stream_t stream) {
  DeviceInfo dev;
  const epq_status st = check_pack_args(fmt, W, blocks, rows, cols, &dev);
  if (st != EPQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *out = static_cast<uint8_t *>(blocks);
  const int64_t nw = rows * cols;
  switch (fmt) {
    case EPQ_Q8_0: quantize32_kernel<EPQ_Q8_0><<<grid_for(nw / 32, dev), kThreads, 0, s>>>(W, out, nw / 32); break;
    case EPQ_Q4_0: quantize32_kernel<EPQ_Q4_0><<<grid_for(nw / 32, dev), kThreads, 0, s>>>(W, out, nw / 32); break;
    case EPQ_Q4_1: quantize32_kernel<EPQ_Q4_1><<<grid_for(nw / 32, dev), kThreads, 0, s>>>(W, out, nw / 32); break;
    case EPQ_Q4_K: quantize_q4k_kernel<<<grid_for(nw / 256, dev), kThreads, 0, s>>>(W, out, nw / 256); break;
    case EPQ_Q2_K:
      quantize_k16_kernel<EPQ_Q2_K><<<grid_for(nw / 256, dev), kThreads, 0, s>>>(W, out, nw / 256, cols / 256,
                                                                                 epq_row_bytes(fmt, cols));
      break;
    case EPQ_Q6_K:
      quantize_k16_kernel<EPQ_Q6_K><<<grid_for(nw / 256, dev), kThreads, 0, s>>>(W, out, nw / 256, cols / 256,
                                                                                 epq_row_bytes(fmt, cols));
      break;
  }
  return check_launch();
}

extern "C" epq_status epq_dequantize(epq_fmt fmt, const void *blocks, int64_t rows, int64_t cols, float *W_out,
                                     epq_stream_t stream) {
  DeviceInfo dev;
  const epq_status st = check_pack_args(fmt, blocks, W_out, rows, cols, &dev);
  if (st != EPQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t *in = static_cast<const uint8_t *>(blocks);
  const int64_t nw = rows * cols;
  switch (fmt) {
    case EPQ_Q8_0: dequantize32_kernel<EPQ_Q8_0><<<grid_for(nw / 32, dev), kThreads, 0, s>>>(in, W_out, nw / 32); break;
    case EPQ_Q4_0: dequantize32_kernel<EPQ_Q4_0><<<grid_for(nw / 32, dev), kThreads, 0, s>>>(in, W_out, nw / 32); break;
    case EPQ_Q4_1: dequantize32_kernel<EPQ_Q4_1><<<grid_for(nw / 32, dev), kThreads, 0, s>>>(in, W_out, nw / 32); break;
    case EPQ_Q4_K: dequantize_q4k_kernel<<<grid_for(nw / 256, dev), kThreads, 0, s>>>(in, W_out, nw / 256); break;
    case EPQ_Q2_K:
      dequantize_k16_kernel<EPQ_Q2_K><<<grid_for(nw / 256, dev), kThreads, 0, s>>>(in, W_out, nw / 256, cols / 256,
                                                                                   epq_row_bytes(fmt, cols));
      break;
    case EPQ_Q6_K:
      dequantize_k16_kernel<EPQ_Q6_K><<<grid_for(nw / 256, dev), kThreads, 0, s>>>(in, W_out, nw / 256, cols / 256,
                                                                                   epq_row_bytes(fmt, cols));
      break;
  }
  return check_launch();
}

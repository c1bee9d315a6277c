// Dequant-GEMV engine: per-thread block-column arithmetic shared by the dense
// GEMV and the expert kernels.
//
// Work split.  A row of `cols` weights is a run of nblk = cols/32 "columns"
// of 32 weights (a Q8_0/Q4_0/Q4_1 block, or one Q4_K sub-block).  Thread c of
// a row group owns column c for the whole kernel: it keeps the 32 activations
// of that column in registers, pre-scaled, and only ever reads the packed
// bytes of column c of each row from shared memory.
//
// Nibble -> float in one instruction.  The 32-bit pattern (n << 4p) read as
// an IEEE float is the exact value n * 2^(4p - 149) (a subnormal or the
// smallest normals, where the encoding is linear) for any bit position up to
// 23.  So masking the packed word with 0xF << 4p yields the weight code as a
// float that carries a known power of two; the activation it multiplies is
// stored pre-multiplied by the inverse power, chosen so that every product
// n * x * 2^(A - 149) is a normal float.  The two nibbles above bit 23 are
// first shifted down by 16.  Codes of Q8_0 use the same trick on bytes after
// an XOR with 0x80 (q + 128).  Products are accumulated with the packed
// fma.rn.f32x2 (two IEEE fp32 FMAs per instruction, subnormals kept).
//
// Per-block scales and minima enter once per column:
//   Q4_K  part = d*c * sum(n x) - dmin*k * sum(x)
//   Q4_0  part = d * (sum(n x) - 8 sum(x))
//   Q4_1  part = d * sum(n x) + m * sum(x)
//   Q8_0  part = d * (sum((q+128) x) - 128 sum(x))
// with sum(x) of the column precomputed once (in the same scaled units).
#pragma once

#include "common.cuh"

namespace epq {

template <int FMT>
struct Fmt;

// Shift (in bits) that each weight position of a 32-weight column carries
// in its float pattern; x is stored as x * 2^(A - shift).
template <>
struct Fmt<EPQ_Q4_K> {
  static constexpr int kBlockBytes = 144;
  __device__ static constexpr int shift(int j) { return (j & 7) < 6 ? 4 * (j & 7) : 4 * ((j & 7) - 4); }
};
template <>
struct Fmt<EPQ_Q4_0> {
  static constexpr int kBlockBytes = 18;
  __device__ static constexpr int shift(int j) { return (j & 7) < 6 ? 4 * (j & 7) : 4 * ((j & 7) - 4); }
};
template <>
struct Fmt<EPQ_Q4_1> {
  static constexpr int kBlockBytes = 20;
  __device__ static constexpr int shift(int j) { return (j & 7) < 6 ? 4 * (j & 7) : 4 * ((j & 7) - 4); }
};
template <>
struct Fmt<EPQ_Q8_0> {
  static constexpr int kBlockBytes = 34;
  __device__ static constexpr int shift(int j) { return (j & 3) == 3 ? 8 : 8 * (j & 3); }
};

__device__ __forceinline__ float fbits(uint32_t u) { return __uint_as_float(u); }

// A pair of floats held in one 64-bit register pair, the operand form of
// fma.rn.f32x2.  Keeping activations and accumulators in this form avoids
// re-pairing registers around every packed FMA.
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f2_t f2_bits(uint32_t lo, uint32_t hi) {
  f2_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ float f2_sum(f2_t v) {
  float lo, hi;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
__device__ __forceinline__ void f2_fma(f2_t &acc, f2_t a, f2_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// acc += acc2, lane-wise (the two halves of a split accumulation)
template <int NV>
__device__ __forceinline__ void f2_join(f2_t (&acc)[NV], const f2_t (&acc2)[NV]) {
#pragma unroll
  for (int v = 0; v < NV; ++v) asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc[v]) : "l"(acc2[v]));
}

// Activations of one 32-weight column for NV vectors, as 16 pairs each.
template <int NV>
struct XCol {
  f2_t p[NV][16];
};

// sum over one 32-bit word of 8 nibbles (weights 8i..8i+7) for NV vectors.
// Callers alternate two accumulators between words (two independent FMA
// chains per column).
template <int NV>
__device__ __forceinline__ void nib_word(uint32_t w, const XCol<NV> &x, int i, f2_t (&acc)[NV]) {
  const f2_t p01 = f2_bits(w & 0x0000000Fu, w & 0x000000F0u);
  const f2_t p23 = f2_bits(w & 0x00000F00u, w & 0x0000F000u);
  const f2_t p45 = f2_bits(w & 0x000F0000u, w & 0x00F00000u);
  const uint32_t h = w >> 16;
  const f2_t p67 = f2_bits(h & 0x00000F00u, h & 0x0000F000u);
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    f2_fma(acc[v], p01, x.p[v][4 * i + 0]);
    f2_fma(acc[v], p23, x.p[v][4 * i + 1]);
    f2_fma(acc[v], p45, x.p[v][4 * i + 2]);
    f2_fma(acc[v], p67, x.p[v][4 * i + 3]);
  }
}

// sum over one 32-bit word of 4 int8 codes (weights 4i..4i+3), biased by 128.
template <int NV>
__device__ __forceinline__ void byte_word(uint32_t w, const XCol<NV> &x, int i, f2_t (&acc)[NV]) {
  const uint32_t u = w ^ 0x80808080u;
  const f2_t p01 = f2_bits(u & 0x000000FFu, u & 0x0000FF00u);
  const f2_t p23 = f2_bits(u & 0x00FF0000u, (u >> 16) & 0x0000FF00u);
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    f2_fma(acc[v], p01, x.p[v][2 * i + 0]);
    f2_fma(acc[v], p23, x.p[v][2 * i + 1]);
  }
}

// Per-thread constants of one block column (independent of the row).
template <int FMT>
struct ColConst {
  int off;        // byte offset of the column's block (or superblock header) in a row
  int qoff;       // byte offset of the aligned word run holding the codes
  int qsh;        // funnel shift (0 or 16) that realigns the code words
  int csel, csh;  // Q4_K: scale-code word pair selector and shift
  int ksel, ksh;  // Q4_K: min-code word pair selector and shift
  __device__ void init(int c) {
    if (FMT == EPQ_Q4_K) {
      const int sb = c >> 3, s = c & 7;
      off = sb * 144;
      qoff = off + 16 + 16 * s;
      qsh = 0;
      const int pc = 6 * s;        // scale code bits in the 96-bit stream
      csel = pc >= 32;
      csh = pc & 31;
      const int pk = 48 + 6 * s;   // min code bits
      ksel = pk >= 64;
      ksh = pk & 31;
    } else {
      const int bb = Fmt<FMT>::kBlockBytes;
      off = c * bb;
      const int q0 = off + (FMT == EPQ_Q4_1 ? 4 : 2);
      qoff = q0 & ~3;
      qsh = (q0 & 3) * 8;
      csel = csh = ksel = ksh = 0;
    }
  }
};

// Partial dot product of one row's column for NV vectors, in scaled units.
// `row` points at the row's packed bytes in shared memory; xs[v] is the
// column's scaled activation sum sum(x) * 2^(A_v - 149).
template <int FMT, int NV>
__device__ __forceinline__ void column_dot(const uint8_t *row, const ColConst<FMT> &cc, const XCol<NV> &x,
                                           const float (&xs)[NV], float (&part)[NV]) {
  f2_t acc[NV], acc2[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) acc[v] = acc2[v] = 0ull;
  if (FMT == EPQ_Q4_K) {
    const uint4 h = *reinterpret_cast<const uint4 *>(row + cc.off);
    const uint4 q = *reinterpret_cast<const uint4 *>(row + cc.qoff);
    nib_word<NV>(q.x, x, 0, acc);
    nib_word<NV>(q.y, x, 1, acc2);
    nib_word<NV>(q.z, x, 2, acc);
    nib_word<NV>(q.w, x, 3, acc2);
    f2_join(acc, acc2);
    const float d = half_bits_to_float(h.x), dmin = half_bits_to_float(h.x >> 16);
    const uint32_t c6 = __funnelshift_r(cc.csel ? h.z : h.y, cc.csel ? h.w : h.z, cc.csh) & 63u;
    const uint32_t k6 = __funnelshift_r(cc.ksel ? h.w : h.z, cc.ksel ? 0u : h.w, cc.ksh) & 63u;
    const float S = d * static_cast<float>(c6);
    const float M = dmin * static_cast<float>(k6);
#pragma unroll
    for (int v = 0; v < NV; ++v) part[v] = fmaf(S, f2_sum(acc[v]), -M * xs[v]);
  } else if (FMT == EPQ_Q4_1) {
    const uint32_t *wq = reinterpret_cast<const uint32_t *>(row + cc.qoff);
    const uint32_t dm = *reinterpret_cast<const uint32_t *>(row + cc.off);
    nib_word<NV>(wq[0], x, 0, acc);
    nib_word<NV>(wq[1], x, 1, acc2);
    nib_word<NV>(wq[2], x, 2, acc);
    nib_word<NV>(wq[3], x, 3, acc2);
    f2_join(acc, acc2);
    const float d = half_bits_to_float(dm), m = half_bits_to_float(dm >> 16);
#pragma unroll
    for (int v = 0; v < NV; ++v) part[v] = fmaf(d, f2_sum(acc[v]), m * xs[v]);
  } else if (FMT == EPQ_Q4_0) {
    const uint32_t *wq = reinterpret_cast<const uint32_t *>(row + cc.qoff);
    const uint32_t w0 = wq[0], w1 = wq[1], w2 = wq[2], w3 = wq[3], w4 = wq[4];
    const float d = half_bits_to_float(*reinterpret_cast<const unsigned short *>(row + cc.off));
    nib_word<NV>(__funnelshift_r(w0, w1, cc.qsh), x, 0, acc);
    nib_word<NV>(__funnelshift_r(w1, w2, cc.qsh), x, 1, acc2);
    nib_word<NV>(__funnelshift_r(w2, w3, cc.qsh), x, 2, acc);
    nib_word<NV>(__funnelshift_r(w3, w4, cc.qsh), x, 3, acc2);
    f2_join(acc, acc2);
#pragma unroll
    for (int v = 0; v < NV; ++v) part[v] = d * (f2_sum(acc[v]) - 8.0f * xs[v]);
  } else {  // Q8_0
    const uint32_t *wq = reinterpret_cast<const uint32_t *>(row + cc.qoff);
    const float d = half_bits_to_float(*reinterpret_cast<const unsigned short *>(row + cc.off));
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = wq[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) byte_word<NV>(__funnelshift_r(w[i], w[i + 1], cc.qsh), x, i, (i & 1) ? acc2 : acc);
    f2_join(acc, acc2);
#pragma unroll
    for (int v = 0; v < NV; ++v) part[v] = d * (f2_sum(acc[v]) - 128.0f * xs[v]);
  }
}

// Load and pre-scale one column of activations for NV vectors.
// Returns per-vector local max |x|, sum x^2 and sum x (unscaled) through
// the output arrays; the scaled registers are filled by scale_column().
struct XGather {
  int group;     // > 1: heads of x are repeated `group` times
  int head_dim;  // floats per head
  __device__ __forceinline__ int src(int j) const {
    if (group <= 1) return j;
    const int span = head_dim * group;
    return (j / span) * head_dim + (j % head_dim);
  }
};

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


// Activation column loader: 32 consecutive floats of x (16-byte aligned).
__device__ __forceinline__ void load_column(const float *src, float (&xr)[32]) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 q = *reinterpret_cast<const float4 *>(src + j);
    xr[j] = q.x;
    xr[j + 1] = q.y;
    xr[j + 2] = q.z;
    xr[j + 3] = q.w;
  }
}

// Exponent E with |v| < 2^E for every |v| <= amax (amax >= 0, finite).
__device__ __forceinline__ int bound_exponent(float amax) {
  int eb = (__float_as_int(amax) >> 23) & 0xFF;
  if (eb == 0) eb = 1;
  return eb - 126;
}

// Turn a loaded column into the scaled form column_dot() expects:
// x_j * 2^(126 - E - shift_j) packed in pairs, and return sum(x) * 2^(-23 - E).
template <int FMT>
__device__ __forceinline__ float scale_column(const float (&xr)[32], int E, f2_t (&out)[16]) {
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) s += xr[j];
#pragma unroll
  for (int j = 0; j < 32; j += 2)
    out[j / 2] = f2_pack(scale_pow2(xr[j], 126 - E - Fmt<FMT>::shift(j)),
                         scale_pow2(xr[j + 1], 126 - E - Fmt<FMT>::shift(j + 1)));
  return scale_pow2(s, -23 - E);
}

// Undo the scaling of a finished row sum.
__device__ __forceinline__ float unscale(float v, int E) { return scale_pow2(v, 23 + E); }

// silu(g) = g / (1 + exp(-g))
__device__ __forceinline__ float silu(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

}  // namespace epq

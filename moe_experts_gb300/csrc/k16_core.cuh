// Device building blocks of the tensor-core dequant-GEMV for the K-quants
// with 16-weight sub-blocks, Q2_K and Q6_K (gemv_k16.cu and the expert
// kernels).
//
// The formats (two-level K-quants, "EPM ... 記憶體怎麼配置的" fixes Q6_K at
// 210 B per 256 weights; the 2-bit experts of "smolmaxxing"):
//   Q2_K  w = d*c_s*n - dmin*k_s,  n 0..3, c_s 1..15, k_s 0..15
//   Q6_K  w = d*c_s*(u - 32),       u 0..63, c_s int8
// A row of nsb superblocks is stored plane by plane; lane t of a warp reads
// the entries of sub-blocks 4t..4t+3 of each plane, which are contiguous:
//   Q2_K  code words[16 nsb] (one 32-bit word per sub-block) | c | k<<4 [16 nsb]
//         | f16 d, dmin [nsb]
//   Q6_K  low nibbles[128 nsb] (8 bytes per sub-block) | high parts[16 nsb words]
//         | int8 c[16 nsb] | f16 d[nsb]
// A 2-bit field (Q2_K code, Q6_K high part) of sub-block position i sits at
// bit kField[i] of the sub-block's word, kField = {4, 8, 6, 10, 20, 24, 22,
// 26, 28, 0, 30, 2, 12, 16, 14, 18}: masking the word W with 0x00300030
// isolates positions (0, 4) at fp16 mantissa bits 4-5 of its two halves,
// 0x03000300 positions (1, 5) at bits 8-9; W >> 2 gives (2, 6) and (3, 7)
// the same way, rotr(W, 24) gives (8, 12), (9, 13) and rotr(W, 24) >> 2 gives
// (10, 14), (11, 15).  The low nibbles of positions (0, 4) are at bits 0-3
// of the sub-block's first nibble word, (1, 5) at bits 4-7, and (2, 6),
// (3, 7) the same after a shift by 8 (second word: positions 8..15).  So a
// pair of codes becomes an fp16 MMA operand pair with one or two logic
// ops, exact (fp16 subnormals, which the tensor cores take as they are):
//   Q2_K  (W & m) read as fp16 = n * 2^-20 (mask A) or n * 2^-16 (mask B)
//   Q6_K  (N & nibble mask) | (W & field mask) read as fp16 = u * 2^-24
//         (A) or u * 2^-20 (B), u = m + 32 (the offset is taken off with
//         32 * sum(x) per sub-block)
// and the x operands of class-B slots carry 2^4 less than those of class A.
//
// MMA layout (m16n8k16, A row-major, B column-major), one warp per 16 rows:
//   * A rows are the 16 weight rows; lane (g, t) holds rows g and g + 8;
//   * the warp walks a superblock in 4 groups q; in group q lane t owns
//     sub-block 4t + q of both its rows, and the group's 4 MMAs take
//     positions (0,4)(1,5) | (2,6)(3,7) | (8,12)(9,13) | (10,14)(11,15) of it
//     in the k-slots {2t, 2t+1} and {2t+8, 2t+9};
//   * the 8 columns of B are (owner t' = n >> 1, part = n & 1): x at the
//     positions of owner t''s sub-block, split into fp16 hi and lo parts,
//     zero in the k-slots of the other owners (block-diagonal B);
//   * so after a group's 4 MMAs, C[row][(t, part)] is the dot product of
//     the row's sub-block 4t + q with that part of x, and lane (g, t) holds
//     exactly the two parts of its own sub-block for rows g and g + 8: the
//     sub-block scale c (and for Q2_K the lift k * sum(x)) is applied in
//     float32 right there, no data leaves the lane until the row reduction.
// x is split per (vector, superblock) into fp16 hi + lo parts after a
// power-of-two scale that maps its largest |x| into [2^14, 2^15) for the
// class-A slots; the superblock factor d is multiplied by the inverse
// scale (sum_scale) to undo it.
#pragma once

#include "common.cuh"

namespace epq {
namespace k16 {

// x operands of one (vector, superblock): [group 4][mma 4][slot 9][8 B];
// slots 0..7 = (owner t, part), slot 8 = zeros for the lanes whose column
// belongs to another owner.
constexpr int kSlotBytes = 8;
constexpr int kMmaBytes = 9 * kSlotBytes;
constexpr int kSbFragBytes = 16 * kMmaBytes;  // 1152

// operand masks
constexpr uint32_t kMaskA = 0x00300030u;    // 2-bit fields at bits 4-5 of each half
constexpr uint32_t kMaskB = 0x03000300u;    // 2-bit fields at bits 8-9
constexpr uint32_t kNibA = 0x000F000Fu;     // nibbles at bits 0-3
constexpr uint32_t kNibB = 0x00F000F0u;     // nibbles at bits 4-7

__device__ __forceinline__ uint32_t rotr(uint32_t w, int s) { return __funnelshift_r(w, w, s); }

__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

// B operands are read with plain loads from the __shared__ array (not
// volatile asm): the compiler may then issue them ahead of the preceding
// MMAs, and the CTA barriers still order them after the staging stores.
__device__ __forceinline__ uint2 lds64(const uint8_t *p) { return *reinterpret_cast<const uint2 *>(p); }

// Streaming loads of packed weights (read once, not kept in L1).
__device__ __forceinline__ uint4 ldg_stream16(const uint8_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream4(const uint8_t *p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const uint8_t *p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// A 32-bit word at a 2-byte boundary.
__device__ __forceinline__ uint32_t ldg_w2(const uint8_t *p) { return ldg_u16(p) | (ldg_u16(p + 2) << 16); }

// A word of a plane: ALIGN is the row alignment (16, 4 or 2 bytes).
template <int ALIGN>
__device__ __forceinline__ uint32_t ldg_word(const uint8_t *p) {
  if constexpr (ALIGN >= 4) return ldg_stream4(p);
  else return ldg_w2(p);
}

// Exact float of a byte / of an int8 byte (magic-number conversion).
__device__ __forceinline__ float u8_to_float(uint32_t b) { return __uint_as_float(0x4B000000u | b) - 8388608.0f; }
__device__ __forceinline__ float s8_to_float(uint32_t b) {
  return __uint_as_float(0x4B000000u | ((b ^ 0x80u) & 0xFFu)) - 8388736.0f;
}

// ------------------------------------------------------------------ packed operands
// What lane t reads of one row for one superblock.
template <int FMT>
struct RowOps;

template <>
struct RowOps<EPQ_Q2_K> {
  uint32_t q[4];  // code words of sub-blocks 4t..4t+3
  uint32_t sub;   // their c | k << 4 bytes
  uint32_t fac;   // d | dmin << 16
};

template <>
struct RowOps<EPQ_Q6_K> {
  uint32_t ql[8];  // low nibbles of sub-blocks 4t..4t+3 (two words each)
  uint32_t qh[4];  // their high-part words
  uint32_t sc;     // their int8 scale codes
  uint32_t d;      // f16 d
};

template <>
struct RowOps<EPQ_Q4_K> {
  uint32_t qs[8];  // nibbles of sub-blocks 2t, 2t+1 (four words each; word i = weights 8i..8i+7)
  uint4 hdr;       // f16 d | f16 dmin, then the 96-bit stream of scale and min codes
};

// ALIGN: the rows start on 16-byte boundaries (row bytes % 16 == 0: wide
// planes read 16 bytes at a time), on 4-byte boundaries (word loads) or, for
// Q6_K rows of an odd number of superblocks, on 2-byte boundaries.
template <int FMT, int ALIGN>
__device__ __forceinline__ void load_ops(RowOps<FMT> &o, const uint8_t *row, int64_t nsb, int sb, int t) {
  if constexpr (FMT == EPQ_Q2_K) {
    const uint8_t *qp = row + 64 * static_cast<int64_t>(sb) + 16 * t;
    if constexpr (ALIGN == 16) {
      const uint4 v = ldg_stream16(qp);
      o.q[0] = v.x, o.q[1] = v.y, o.q[2] = v.z, o.q[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) o.q[i] = ldg_word<ALIGN>(qp + 4 * i);
    }
    o.sub = ldg_word<ALIGN>(row + 64 * nsb + 16 * static_cast<int64_t>(sb) + 4 * t);
    o.fac = ldg_word<ALIGN>(row + 80 * nsb + 4 * static_cast<int64_t>(sb));
  } else if constexpr (FMT == EPQ_Q4_K) {  // 144-byte superblocks: rows are always 16-byte multiples
    const uint8_t *b = row + 144 * static_cast<int64_t>(sb);
    const uint4 h = ldg_stream16(b), a = ldg_stream16(b + 16 + 32 * t), c = ldg_stream16(b + 32 + 32 * t);
    o.hdr = h;
    o.qs[0] = a.x, o.qs[1] = a.y, o.qs[2] = a.z, o.qs[3] = a.w;
    o.qs[4] = c.x, o.qs[5] = c.y, o.qs[6] = c.z, o.qs[7] = c.w;
  } else {
    const uint8_t *lp = row + 128 * static_cast<int64_t>(sb) + 32 * t;
    const uint8_t *hp = row + 128 * nsb + 64 * static_cast<int64_t>(sb) + 16 * t;
    if constexpr (ALIGN == 16) {
      const uint4 a = ldg_stream16(lp), b = ldg_stream16(lp + 16), h = ldg_stream16(hp);
      o.ql[0] = a.x, o.ql[1] = a.y, o.ql[2] = a.z, o.ql[3] = a.w;
      o.ql[4] = b.x, o.ql[5] = b.y, o.ql[6] = b.z, o.ql[7] = b.w;
      o.qh[0] = h.x, o.qh[1] = h.y, o.qh[2] = h.z, o.qh[3] = h.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) o.ql[i] = ldg_word<ALIGN>(lp + 4 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i) o.qh[i] = ldg_word<ALIGN>(hp + 4 * i);
    }
    o.sc = ldg_word<ALIGN>(row + 192 * nsb + 16 * static_cast<int64_t>(sb) + 4 * t);
    o.d = ldg_u16(row + 208 * nsb + 2 * static_cast<int64_t>(sb));
  }
}

// The 8 fp16 operand pairs of one sub-block of one row, in MMA order:
// p[2i] and p[2i+1] feed MMA i (k-slots {2t, 2t+1} and {2t+8, 2t+9}).  The
// pairs are the masked code bits read as fp16 subnormals (the tensor cores
// take subnormal fp16 operands exactly): even pairs ("class A") carry
// code * 2^-20 (Q2_K) / u * 2^-24 (Q6_K), odd pairs ("class B") 16 times
// that; the x operands of the two classes carry the compensating powers of
// two (stage_superblock).
__device__ __forceinline__ void pairs_q2k(uint32_t w, uint32_t (&p)[8]) {
  const uint32_t w2 = w >> 2, r = rotr(w, 24), r2 = r >> 2;
  p[0] = w & kMaskA;
  p[1] = w & kMaskB;
  p[2] = w2 & kMaskA;
  p[3] = w2 & kMaskB;
  p[4] = r & kMaskA;
  p[5] = r & kMaskB;
  p[6] = r2 & kMaskA;
  p[7] = r2 & kMaskB;
}

__device__ __forceinline__ void pairs_q6k(uint32_t n0, uint32_t n1, uint32_t w, uint32_t (&p)[8]) {
  const uint32_t w2 = w >> 2, r = rotr(w, 24), r2 = r >> 2;
  const uint32_t m0 = n0 >> 8, m1 = n1 >> 8;
  p[0] = (n0 & kNibA) | (w & kMaskA);
  p[1] = (n0 & kNibB) | (w & kMaskB);
  p[2] = (m0 & kNibA) | (w2 & kMaskA);
  p[3] = (m0 & kNibB) | (w2 & kMaskB);
  p[4] = (n1 & kNibA) | (r & kMaskA);
  p[5] = (n1 & kNibB) | (r & kMaskB);
  p[6] = (m1 & kNibA) | (r2 & kMaskA);
  p[7] = (m1 & kNibB) | (r2 & kMaskB);
}

// Power of two that brings a superblock's code sums back to code * x units:
// the class-A product is code * 2^-20 * x * 2^(14 - e) (Q2_K) or
// u * 2^-24 * x * 2^(14 - e) (Q6_K), e the exponent of the superblock's
// largest |x| (stage_superblock).
template <int FMT>
__device__ __forceinline__ float sum_scale(int e) {
  return exp2i((FMT == EPQ_Q2_K ? 6 : 10) + e);  // Q4_K nibbles carry 2^-24 like the Q6_K codes
}

// Q4_K: the 6-bit scale / min codes of sub-blocks 2t, 2t+1 from a
// superblock header (the 96-bit stream: c_0..c_7 at bits 0..47, k_0..k_7 at
// bits 48..95, code j at bits 6j).
__device__ __forceinline__ void q4k_codes(const uint4 &h, int t, float (&c)[2], float (&k)[2]) {
  const uint64_t cf = static_cast<uint64_t>(h.y) | (static_cast<uint64_t>(h.z) << 32);
  const uint64_t kf = static_cast<uint64_t>(h.z) | (static_cast<uint64_t>(h.w) << 32);
  const uint32_t cc = static_cast<uint32_t>(cf >> (12 * t)), kk = static_cast<uint32_t>(kf >> (16 + 12 * t));
  c[0] = u8_to_float(cc & 63u);
  c[1] = u8_to_float((cc >> 6) & 63u);
  k[0] = u8_to_float(kk & 63u);
  k[1] = u8_to_float((kk >> 6) & 63u);
}

// Q4_K superblock: lane t owns sub-blocks 2t (group 0) and 2t+1 (group 1)
// of 32 weights; MMA m of a group takes nibble word m/2, positions
// (0,4)(1,5) for even m and (2,6)(3,7) for odd m (the word shifted by 8),
// as fp16 subnormals n 2^-24 (class A) and 16 n 2^-24 (class B).
template <int NV>
__device__ __forceinline__ void superblock_q4k(const RowOps<EPQ_Q4_K> &lo, const RowOps<EPQ_Q4_K> &hi, const uint8_t *frag,
                                               uint32_t vstride, const float (&ps)[NV], const float *xsum, int xstride,
                                               int t, float (&acc)[2][NV]) {
  float cl[2], kl[2], ch[2], kh[2];
  q4k_codes(lo.hdr, t, cl, kl);
  q4k_codes(hi.hdr, t, ch, kh);
  float cs[2][NV], ms[2][NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) cs[0][v] = cs[1][v] = ms[0][v] = ms[1][v] = 0.0f;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    float c[NV][4];
#pragma unroll
    for (int v = 0; v < NV; ++v) c[v][0] = c[v][1] = c[v][2] = c[v][3] = 0.0f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint32_t wl = m & 1 ? lo.qs[4 * q + m / 2] >> 8 : lo.qs[4 * q + m / 2];
      const uint32_t wh = m & 1 ? hi.qs[4 * q + m / 2] >> 8 : hi.qs[4 * q + m / 2];
      const uint32_t a[4] = {wl & kNibA, wh & kNibA, wl & kNibB, wh & kNibB};
#pragma unroll
      for (int v = 0; v < NV; ++v)
        mma(c[v], a, lds64(frag + v * vstride + (q * 8 + m) * kMmaBytes));
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float X = xsum[v * xstride + 2 * t + q];
      cs[0][v] = fmaf(cl[q], c[v][0] + c[v][1], cs[0][v]);
      cs[1][v] = fmaf(ch[q], c[v][2] + c[v][3], cs[1][v]);
      ms[0][v] = fmaf(kl[q], X, ms[0][v]);
      ms[1][v] = fmaf(kh[q], X, ms[1][v]);
    }
  }
  const float dl = half_bits_to_float(lo.hdr.x), ml = half_bits_to_float(lo.hdr.x >> 16);
  const float dh = half_bits_to_float(hi.hdr.x), mh = half_bits_to_float(hi.hdr.x >> 16);
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    acc[0][v] = fmaf(dl * ps[v], cs[0][v], fmaf(-ml, ms[0][v], acc[0][v]));
    acc[1][v] = fmaf(dh * ps[v], cs[1][v], fmaf(-mh, ms[1][v], acc[1][v]));
  }
}

// ------------------------------------------------------------------ one superblock
// Adds one superblock's contribution to acc[row 0 = g, 1 = g + 8][vector]
// (partial: only lane t's owner sub-blocks; the 4 lanes of a row sum later).
//   frag   this superblock's x operands for vector 0 (in the __shared__
//          array) plus the lane's slot offset; vector v adds v * vstride
//   ps     2^(10 - sigma) of this superblock per vector
//   xsum   shared float sums of x over the superblock's 16 sub-blocks for
//          vector 0 (the Q2_K lift term, the Q6_K code offset); vector v adds
//          v * xstride floats
template <int FMT, int NV>
__device__ __forceinline__ void superblock(const RowOps<FMT> &lo, const RowOps<FMT> &hi, const uint8_t *frag,
                                           uint32_t vstride, const float (&ps)[NV], const float *xsum, int xstride,
                                           int t, float (&acc)[2][NV]) {
  if constexpr (FMT == EPQ_Q4_K) {
    superblock_q4k<NV>(lo, hi, frag, vstride, ps, xsum, xstride, t, acc);
    return;
  } else {
  float cs[2][NV], ms[2][NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) cs[0][v] = cs[1][v] = ms[0][v] = ms[1][v] = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pl[8], ph[8];
    if constexpr (FMT == EPQ_Q2_K) {
      pairs_q2k(lo.q[q], pl);
      pairs_q2k(hi.q[q], ph);
    } else {
      pairs_q6k(lo.ql[2 * q], lo.ql[2 * q + 1], lo.qh[q], pl);
      pairs_q6k(hi.ql[2 * q], hi.ql[2 * q + 1], hi.qh[q], ph);
    }
    float c[NV][4];
#pragma unroll
    for (int v = 0; v < NV; ++v) c[v][0] = c[v][1] = c[v][2] = c[v][3] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a[4] = {pl[2 * i], ph[2 * i], pl[2 * i + 1], ph[2 * i + 1]};
#pragma unroll
      for (int v = 0; v < NV; ++v)
        mma(c[v], a, lds64(frag + v * vstride + (q * 4 + i) * kMmaBytes));
    }
    if constexpr (FMT == EPQ_Q2_K) {
      const uint32_t bl = (lo.sub >> (8 * q)) & 0xFFu, bh = (hi.sub >> (8 * q)) & 0xFFu;
      const float cl = u8_to_float(bl & 15u), kl = u8_to_float(bl >> 4);
      const float ch = u8_to_float(bh & 15u), kh = u8_to_float(bh >> 4);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float X = xsum[v * xstride + 4 * t + q];
        cs[0][v] = fmaf(cl, c[v][0] + c[v][1], cs[0][v]);
        cs[1][v] = fmaf(ch, c[v][2] + c[v][3], cs[1][v]);
        ms[0][v] = fmaf(kl, X, ms[0][v]);
        ms[1][v] = fmaf(kh, X, ms[1][v]);
      }
    } else {  // codes carry u = m + 32: the sub-block term is c (sum u x - 32 sum x)
      const float cl = s8_to_float((lo.sc >> (8 * q)) & 0xFFu), ch = s8_to_float((hi.sc >> (8 * q)) & 0xFFu);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float X = xsum[v * xstride + 4 * t + q];
        cs[0][v] = fmaf(cl, c[v][0] + c[v][1], cs[0][v]);
        cs[1][v] = fmaf(ch, c[v][2] + c[v][3], cs[1][v]);
        ms[0][v] = fmaf(cl, X, ms[0][v]);
        ms[1][v] = fmaf(ch, X, ms[1][v]);
      }
    }
  }
  if constexpr (FMT == EPQ_Q2_K) {
    const float dl = half_bits_to_float(lo.fac), ml = half_bits_to_float(lo.fac >> 16);
    const float dh = half_bits_to_float(hi.fac), mh = half_bits_to_float(hi.fac >> 16);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      acc[0][v] = fmaf(dl * ps[v], cs[0][v], fmaf(-ml, ms[0][v], acc[0][v]));
      acc[1][v] = fmaf(dh * ps[v], cs[1][v], fmaf(-mh, ms[1][v], acc[1][v]));
    }
  } else {
    const float dl = half_bits_to_float(lo.d), dh = half_bits_to_float(hi.d);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      acc[0][v] = fmaf(dl * ps[v], cs[0][v], fmaf(-32.0f * dl, ms[0][v], acc[0][v]));
      acc[1][v] = fmaf(dh * ps[v], cs[1][v], fmaf(-32.0f * dh, ms[1][v], acc[1][v]));
    }
  }
  }
}

// ------------------------------------------------------------------ x staging
// Largest |x| of a lane's 8 values, and of the warp's 256 (one redux.sync;
// callers reduce several units' maxima back to back so that their latencies
// overlap).
__device__ __forceinline__ float lane_absmax(const float (&xv)[8]) {
  float m = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(xv[e]));
  return m;
}

// One warp converts one (vector, superblock) of x (m: the warp's largest
// |x| of it, the same on every lane): lane l holds positions
// 8h..8h+7 (h = l & 1) of sub-block s = l >> 1, already gathered into xv.
// With e the exponent of the superblock's largest |x| (clamped to
// [-100, 100]), the class-A slots get x * 2^(14 - e) and the class-B slots
// x * 2^(10 - e), each split into fp16 hi + lo parts (the largest class-A
// value lands in [2^14, 2^15)).  Writes the operand slots of sub-block s,
// the zero slots (lanes of owner 0) and the sub-block's sum of x into
// sum16[s]; returns e (same on every lane).
__device__ __forceinline__ int stage_superblock(const float (&xv)[8], float m, uint8_t *frag_sb, int lane,
                                                float *sum16) {
  int ex = 0;
  if (m > 0.0f) ex = min(100, max(-100, static_cast<int>((__float_as_uint(m) >> 23) & 255u) - 127));
  const int s = lane >> 1, h = lane & 1, q = s & 3, o = s >> 2;
  uint32_t hi[4], lo[4];  // fp16 pairs (k, k + 4) for k = 0..3; even k class A, odd k class B
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int sh = (k & 1 ? 10 : 14) - ex;
    const float f = exp2i(sh);  // sh in [-90, 114]: a normal power of two
    const float xa = xv[k] * f, xb = xv[k + 4] * f;
    const __half2 hh = __floats2half2_rn(xa, xb);
    const float2 hf = __half22float2(hh);
    const __half2 ll = __floats2half2_rn(xa - hf.x, xb - hf.y);
    hi[k] = *reinterpret_cast<const uint32_t *>(&hh);
    lo[k] = *reinterpret_cast<const uint32_t *>(&ll);
  }
#pragma unroll
  for (int ip = 0; ip < 2; ++ip) {
    const int i = 2 * h + ip;
    uint8_t *m0 = frag_sb + (q * 4 + i) * kMmaBytes;
    *reinterpret_cast<uint2 *>(m0 + (2 * o) * kSlotBytes) = make_uint2(hi[2 * ip], hi[2 * ip + 1]);
    *reinterpret_cast<uint2 *>(m0 + (2 * o + 1) * kSlotBytes) = make_uint2(lo[2 * ip], lo[2 * ip + 1]);
    if (o == 0) *reinterpret_cast<uint2 *>(m0 + 8 * kSlotBytes) = make_uint2(0u, 0u);
  }
  float sx = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) sx += xv[e];
  const float other = __shfl_xor_sync(0xffffffffu, sx, 1);
  if (h == 0) sum16[s] = sx + other;
  return ex;
}

// Q4_K staging: lane l holds positions 8l..8l+7 of the superblock = word
// i = l & 3 of sub-block s = l >> 2 (owner s >> 1, group s & 1), which feed
// MMAs 2i (pairs (0,4), (1,5)) and 2i+1 (pairs (2,6), (3,7)) of the group.
// Same scales as stage_superblock; sum8[s] receives the sub-block's sum of x.
__device__ __forceinline__ int stage_superblock_q4k(const float (&xv)[8], float m, uint8_t *frag_sb, int lane,
                                                    float *sum8) {
  int ex = 0;
  if (m > 0.0f) ex = min(100, max(-100, static_cast<int>((__float_as_uint(m) >> 23) & 255u) - 127));
  const int s = lane >> 2, i = lane & 3, q = s & 1, o = s >> 1;
  uint32_t hi[4], lo[4];  // fp16 pairs (k, k + 4); even k class A, odd k class B
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int sh = (k & 1 ? 10 : 14) - ex;
    const float f = exp2i(sh);  // sh in [-90, 114]: a normal power of two
    const float xa = xv[k] * f, xb = xv[k + 4] * f;
    const __half2 hh = __floats2half2_rn(xa, xb);
    const float2 hf = __half22float2(hh);
    const __half2 ll = __floats2half2_rn(xa - hf.x, xb - hf.y);
    hi[k] = *reinterpret_cast<const uint32_t *>(&hh);
    lo[k] = *reinterpret_cast<const uint32_t *>(&ll);
  }
#pragma unroll
  for (int mm = 0; mm < 2; ++mm) {
    uint8_t *m0 = frag_sb + (q * 8 + 2 * i + mm) * kMmaBytes;
    *reinterpret_cast<uint2 *>(m0 + (2 * o) * kSlotBytes) = make_uint2(hi[2 * mm], hi[2 * mm + 1]);
    *reinterpret_cast<uint2 *>(m0 + (2 * o + 1) * kSlotBytes) = make_uint2(lo[2 * mm], lo[2 * mm + 1]);
    if (o == 0) *reinterpret_cast<uint2 *>(m0 + 8 * kSlotBytes) = make_uint2(0u, 0u);
  }
  float sx = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) sx += xv[e];
  sx += __shfl_xor_sync(0xffffffffu, sx, 1);
  sx += __shfl_xor_sync(0xffffffffu, sx, 2);
  if (i == 0) sum8[s] = sx;
  return ex;
}

// Lane's byte offset into a (group, mma) record: its own column's slot when
// the column belongs to its owner, else the zero slot.
__device__ __forceinline__ uint32_t lane_slot(int lane) {
  const int g = lane >> 2, t = lane & 3;
  return (g >> 1) == t ? static_cast<uint32_t>((2 * t + (g & 1)) * kSlotBytes) : 8u * kSlotBytes;
}

}  // namespace k16
}  // namespace epq

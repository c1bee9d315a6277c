// Device building blocks of the tensor-core Q4_K dequant-GEMV (gemv_tc.cu,
// gemv_chain.cu): fp16 pair arithmetic, the m16n8k16 MMA, shared-memory
// synchronisation helpers, the nibble -> fp16 operand decode and the dot
// products of one 8-row block over a warp's superblocks.  The operand
// layout is described at the top of gemv_tc.cu.
#pragma once

#include "gemv_core.cuh"

namespace epq {
namespace tc {

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ unsigned ld_acquire_shared(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(unsigned *p, unsigned v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

// fp16 pair constants
constexpr uint32_t kH1024 = 0x64006400u;  // {1024, 1024}
constexpr uint32_t kH2p10 = 0x64006400u;  // {2^10, 2^10}
constexpr uint32_t kH2p6 = 0x54005400u;   // {2^6, 2^6}

// Sub-block multipliers {c 2^10} for low nibbles (n 2^-24) and {c 2^6} for
// high nibbles (16 n 2^-24): both products are c*n*2^-14, exact.
struct SubMul {
  uint32_t lo, hi;
};

__device__ __forceinline__ SubMul sub_mul(uint32_t c, uint32_t magic) {
  const uint32_t mc = hsub2((c * 0x00010001u) | magic, magic);  // {c, c}, exact
  return SubMul{hmul2(mc, kH2p10), hmul2(mc, kH2p6)};
}

// One MMA over the eight nibbles of code word w (weights 8i..8i+7 of a
// sub-block): A registers hold c*n*2^-14 at positions {0,4} {1,5} {2,6} {3,7}.
__device__ __forceinline__ void mma_word(uint32_t w, const SubMul &m, uint32_t b0, uint32_t b1, float (&c)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t a0 = hmul2(w & 0x000F000Fu, m.lo);
  const uint32_t a1 = hmul2(w & 0x00F000F0u, m.hi);
  const uint32_t a2 = hmul2(w8 & 0x000F000Fu, m.lo);
  const uint32_t a3 = hmul2(w8 & 0x00F000F0u, m.hi);
  mma16816(c, a0, a1, a2, a3, b0, b1);
}

// Per-warp staging of one superblock's x operands: 8 rows (one per MMA) of
// 32 lane records, padded to 34: a half-warp of converting lanes stores to
// 8 rows x 2 lane groups at once, and a row stride of 2 mod 16 records puts
// those 16 eight-byte stores in distinct bank pairs.
constexpr int kFragRow = 34;
constexpr uint32_t kFragWarpBytes = 8u * kFragRow * 8u;

// 16-byte load of x through the read-only path (x is not written by the
// kernel that reads it).
__device__ __forceinline__ float4 ldg4(const float *p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

// x pair (already scaled) -> fp16 pair of the hi parts, or of the remainders.
__device__ __forceinline__ uint32_t split_pair(float xa, float xb, bool lo) {
  const __half2 h = __floats2half2_rn(xa, xb);
  const float2 f = __half22float2(h);
  const __half2 r = __floats2half2_rn(xa - f.x, xb - f.y);
  const __half2 o = lo ? r : h;
  return *reinterpret_cast<const uint32_t *>(&o);
}

__device__ __forceinline__ float u6_to_float(uint32_t k) { return __uint2float_rn(k); }

// Dot products of one 8-row block (row g of this lane) over the superblocks
// of this warp's k-part, for one matrix (gate or up).  acc: code sums of the
// lane's vector; am0/am1: min terms of vectors 0 and 1 (all unscaled).
// The scale codes 2t, 2t+1 of the lane are header bytes 4 + 1.5t .. (12 bits,
// at bit 4t mod 8), the min codes bytes 10 + 1.5t ..; `csel`/`ksel` pick the
// two bytes with one byte permute and `nsh` is the residual shift.
template <int KP, int NSB, bool FULL>
__device__ __forceinline__ void block_dot(const uint8_t *row, int kq, int nsb, int t, uint32_t magic,
                                          uint32_t csel, uint32_t ksel, int nsh,
                                          const uint32_t (&bq)[NSB][8][2], const float (&fsc)[NSB],
                                          const float *xsum, float &acc, float &am0, float &am1) {
#pragma unroll
  for (int i = 0; i < NSB; ++i) {
    const int sb = kq + i * KP;
    if (!FULL && sb >= nsb) break;  // warp-uniform
    const uint8_t *sp = row + sb * 144;
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
    // useful entries: half 0 (c0, c1) for t < 2, half 1 (c2, c3) for t >= 2
    const float s = t < 2 ? (Ca[0] + Cb[0]) + (Ca[1] + Cb[1]) : (Ca[2] + Cb[2]) + (Ca[3] + Cb[3]);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hd.x));  // d, dmin
    acc = fmaf(dd.x, s * fsc[i], acc);
    const float ka = u6_to_float(kk & 63u), kb = u6_to_float((kk >> 6) & 63u);
    am0 = fmaf(dd.y, fmaf(ka, X.x, kb * X.y), am0);
    am1 = fmaf(dd.y, fmaf(ka, X.z, kb * X.w), am1);
  }
}


}  // namespace tc
}  // namespace epq

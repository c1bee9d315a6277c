// Q4_K dequant-GEMV for 2 to 8 vectors in one weight pass, the vectors in
// the MMA's n dimension (epq_gemv / epq_gemv_ex with nvec >= 2: the
// speculative-verify columns).
//
// [H] "速度上限：带宽 ÷ 权重字节数": a decode step is bound by the bytes of the
// weights it streams, so checking several draft tokens should cost one
// weight pass.  Here one m16n8k16 MMA multiplies 16 weight rows x 16 weights
// by 8 vector columns, so the MMAs per weight do not grow with the number of
// vectors (up to 8).
//
// Operands (Q4_K, w = d c_s n - dmin m_s, n 0..15, c_s, m_s 0..63):
//   * lane (g, t) holds rows g and g + 8 of a 16-row group and, of each
//     superblock, sub-blocks 2t and 2t + 1 (the same 32 bytes of nibbles per
//     row the block-diagonal engine reads: word j = weights 8j..8j+7 of the
//     lane's 64);
//   * MMA 2j + h takes word j: (w >> 8h) & 0x000F000F read as an fp16 pair
//     is the nibbles of positions (2h, 2h + 4) as subnormals n 2^-24, and
//     (w >> 8h) & 0x00F000F0 those of (2h + 1, 2h + 5) as 16 n 2^-24; one
//     HMUL2 by c 2^10 (resp. c 2^6), c the sub-block's scale code, makes
//     both c n 2^-14 exactly (c n <= 945): the scale rides in the operand,
//     so C sums whole superblocks;
//   * B (k16 x n8) holds x of the same positions for the 8 vectors, split
//     per (vector, superblock) into fp16 hi + lo parts after the factor
//     2^(14 - e), e the exponent of the superblock's largest |x|;
//   * the min term dmin sum_s m_s X_s (X_s the sub-block sums of x) is one
//     more MMA pair per superblock: A = the lane's m_{2t}, m_{2t+1} in
//     k-slots 2t, 2t+1 of its rows, B = X hi / lo scaled by 2^(9 - e);
//   * per superblock and vector: result = 2^(e - 9) (512 d C - dmin C_min).
// x operands of a chunk of KC superblocks (all of them when they fit) sit in
// shared memory; longer rows run chunk by chunk with the partial sums of
// every row group of the CTA kept in shared memory between chunks.
//
// CTA: 16 warps = RG row groups x KP k-parts (warp kq takes superblocks
// kq, kq + KP, ... of the chunk); the CTA takes row-group blocks blockIdx.x,
// blockIdx.x + gridDim.x, ...  Each warp streams its rows' superblocks into
// a register ring of 2; the k-parts' partials are added in k-part order
// (then chunk order) through shared memory: bitwise reproducible.
#include <algorithm>
#include <map>
#include <mutex>

#include "gemv_tc.cuh"
#include "k16_core.cuh"

namespace epq {
namespace {

using k16::RowOps;

constexpr int kVnWarps = 16;
constexpr int kVnThreads = kVnWarps * 32;
constexpr uint32_t kVnMma = 512;                // one MMA's B operands: 32 lanes x (hi 8 B, lo 8 B)
constexpr uint32_t kVnPair = 2 * kVnMma + 16;   // MMAs 2j, 2j + 1, then 16 B: an odd number of 16-B units
constexpr uint32_t kVnSbMain = 8 * kVnPair;     // per superblock
constexpr uint32_t kVnSbMin = 32 * 8;           // min-term B operands: 32 lanes x (hi, lo)
constexpr uint32_t kVnSbPs = 8 * 4;             // 2^(e - 9) per vector

struct VnParams {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows_out, up_rows, row_bytes;
  int nsb, kc, nchunks;  // superblocks per row / per chunk, chunks
  int rg, kp, iters_max;
  int nv;
  int64_t x_stride, y_stride;
  int rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early;
};

struct VnLayout {
  uint32_t main, minb, ps, red, part, ssq, total;
};

__host__ __device__ inline uint32_t vn_al16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline VnLayout vn_layout(int kc, int nchunks, int rg, int iters_max, int cl) {
  VnLayout L;
  uint32_t o = 0;
  L.main = o;  // [sb of chunk][word j 8][half h 2][lane 32][hi 8 B | lo 8 B] + 16 B per j (bank offset)
  o += static_cast<uint32_t>(kc) * kVnSbMain;
  L.minb = o;  // [sb][lane 32][hi 4 B | lo 4 B]
  o += static_cast<uint32_t>(kc) * kVnSbMin;
  L.ps = o;  // [sb][vector 8]
  o = vn_al16(o + static_cast<uint32_t>(kc) * kVnSbPs);
  L.red = o;  // [warp][row 16][vector 8]
  o = vn_al16(o + 4u * kVnWarps * 16 * 8);
  L.part = o;  // [iteration][row group][row 16][vector 8], only with several chunks
  if (nchunks > 1) o = vn_al16(o + 4u * static_cast<uint32_t>(iters_max) * rg * 16 * 8);
  L.ssq = o;  // [cluster rank][warp][vector 8] sums of squares, then [vector 8] RMS factors
  o = vn_al16(o + 4u * cl * kVnWarps * 8 + 4u * 8);
  L.total = o;
  return L;
}

__device__ __forceinline__ float vn_silu(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

__device__ __forceinline__ int vn_x_src(int j, int group, int head_dim) {
  if (group <= 1) return j;
  const int span = head_dim * group;
  return (j / span) * head_dim + (j % head_dim);
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t s) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&s));
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t half2_bits(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Split (a, b) into fp16 hi and lo pairs.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ uint32_t cluster_rank_vn() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_vn(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Shared-memory stores into the CTA itself (CL = 1) or into every CTA of
// the cluster at the same offset (base[r] = this CTA's shared window in
// cluster rank r's view).
template <int CL>
struct VnStore {
  uint32_t base[CL];
  __device__ __forceinline__ void v4(uint32_t off, uint4 a) const {
#pragma unroll
    for (int r = 0; r < CL; ++r) {
      if constexpr (CL == 1)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(base[r] + off), "r"(a.x), "r"(a.y), "r"(a.z),
                     "r"(a.w)
                     : "memory");
      else
        asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(base[r] + off), "r"(a.x), "r"(a.y),
                     "r"(a.z), "r"(a.w)
                     : "memory");
    }
  }
  __device__ __forceinline__ void v2(uint32_t off, uint2 a) const {
#pragma unroll
    for (int r = 0; r < CL; ++r) {
      if constexpr (CL == 1)
        asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(base[r] + off), "r"(a.x), "r"(a.y) : "memory");
      else
        asm volatile("st.shared::cluster.v2.u32 [%0], {%1,%2};" ::"r"(base[r] + off), "r"(a.x), "r"(a.y)
                     : "memory");
    }
  }
  __device__ __forceinline__ void f32(uint32_t off, float a) const {
#pragma unroll
    for (int r = 0; r < CL; ++r) {
      if constexpr (CL == 1)
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(base[r] + off), "f"(a) : "memory");
      else
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(base[r] + off), "f"(a) : "memory");
    }
  }
};

template <int CL>
__device__ __forceinline__ void cl_sync() {
  if constexpr (CL == 1)
    __syncthreads();
  else
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One (vector column v, superblock) of x by one warp (m: the warp's largest
// |x| of it): lane l holds positions 8l..8l+7 (word j = l % 8 of owner
// t' = l / 8).  Writes the B
// operands of MMAs 2j and 2j+1 for column v, the min-term operands and
// 2^(e - 9) (offsets into the shared window, to every target of st);
// returns the lane's sum of squares.
template <int CL>
__device__ __forceinline__ float vn_stage(const float (&xv)[8], float m, const VnStore<CL> &st, uint32_t main_sb,
                                          uint32_t min_sb, uint32_t ps_sb, int v, int lane) {
  int ex = 0;
  if (m > 0.0f) ex = min(100, max(-100, static_cast<int>((__float_as_uint(m) >> 23) & 255u) - 127));
  const float f = exp2i(14 - ex);
  const int tp = lane >> 3, j = lane & 7;
  const int L = 4 * v + tp;  // the B-operand lane of column v, k-slot owner tp
  uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
  split_pair(xv[0] * f, xv[4] * f, h0, l0);
  split_pair(xv[1] * f, xv[5] * f, h1, l1);
  split_pair(xv[2] * f, xv[6] * f, h2, l2);
  split_pair(xv[3] * f, xv[7] * f, h3, l3);
  // j-records 1040 B (65 x 16 B) apart: the 8 lanes of a quarter-warp (one tp, j = 0..7) store to 8
  // different bank groups
  st.v4(main_sb + j * kVnPair + L * 16, make_uint4(h0, h1, l0, l1));
  st.v4(main_sb + j * kVnPair + kVnMma + L * 16, make_uint4(h2, h3, l2, l3));
  // sub-block sums: sub-block s = l / 4 (4 lanes); owner tp holds s = 2tp (lane 8tp) and 2tp + 1 (lane 8tp + 4)
  float sx = 0.0f, sq = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sx += xv[e];
    sq = fmaf(xv[e], xv[e], sq);
  }
  sx += __shfl_xor_sync(0xffffffffu, sx, 1);
  sx += __shfl_xor_sync(0xffffffffu, sx, 2);
  const float sx_next = __shfl_down_sync(0xffffffffu, sx, 4);
  if (j == 0) {
    const float g = exp2i(9 - ex);
    uint32_t xh, xl;
    split_pair(sx * g, sx_next * g, xh, xl);
    st.v2(min_sb + L * 8, make_uint2(xh, xl));
  }
  if (lane == 0) st.f32(ps_sb + 4 * v, exp2i(ex - 9));
  return sq;
}

template <bool SW, int CL>
__global__ void __launch_bounds__(kVnThreads, 1) gemv_vn_kernel(const VnParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const VnLayout L = vn_layout(p.kc, p.nchunks, p.rg, p.iters_max, CL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kq = warp % p.kp, rgl = warp / p.kp;
  constexpr int kOut = SW ? 8 : 16;  // outputs per row group
  const int64_t ngroups = (p.rows_out + kOut - 1) / kOut;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * p.rg, stride = static_cast<int64_t>(gridDim.x) * p.rg;
  const int iters = first < ngroups ? static_cast<int>((ngroups - first + stride - 1) / stride) : 0;
  const int64_t nsb = p.nsb;
  const int npass = iters * p.nchunks;  // chunk-major: pass = chunk * iters + iteration

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
  // superblocks of this warp in chunk c: b0 = c KC + kq, + KP, ... < end
  auto count_of = [&](int c) {
    const int b0 = c * p.kc + kq, end = min(p.nsb, (c + 1) * p.kc);
    return b0 < end ? (end - b0 + p.kp - 1) / p.kp : 0;
  };

  constexpr int kDepth = 2;
  RowOps<EPQ_Q4_K> ring_lo[kDepth], ring_hi[kDepth];
  const uint8_t *row_lo = nullptr, *row_hi = nullptr;
  int cnt = 0, bbase = 0;  // of the current pass
  auto fill = [&](int pass) {
    const int c = pass / iters, it = pass - c * iters;
    rows_of(it, row_lo, row_hi);
    cnt = count_of(c);
    bbase = c * p.kc + kq;
#pragma unroll
    for (int d = 0; d < kDepth; ++d)
      if (d < cnt) {
        k16::load_ops<EPQ_Q4_K, 16>(ring_lo[d], row_lo, nsb, bbase + d * p.kp, t);
        k16::load_ops<EPQ_Q4_K, 16>(ring_hi[d], row_hi, nsb, bbase + d * p.kp, t);
      }
  };
  pdl_launch_dependents();  // the next kernel may start its prologue; it waits for this grid before reading y
  if (p.early && npass > 0) fill(0);
  pdl_wait();
  if (!p.early && npass > 0) fill(0);

  float *ps_s = reinterpret_cast<float *>(smem + L.ps);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *part = reinterpret_cast<float *>(smem + L.part);
  float *ssq_s = reinterpret_cast<float *>(smem + L.ssq);  // [rank][warp][vector]: sums of squares
  float *rs_s = ssq_s + CL * kVnWarps * 8;                    // [vector]: RMS factors (1 without the pre-norm)
  const uint32_t rank = CL > 1 ? cluster_rank_vn() : 0u;
  for (int i = threadIdx.x; i < CL * kVnWarps * 8 + 8; i += kVnThreads) ssq_s[i] = i < CL * kVnWarps * 8 ? 0.0f : 1.0f;
  VnStore<CL> st;
#pragma unroll
  for (int r = 0; r < CL; ++r) st.base[r] = CL == 1 ? smem_addr(smem) : mapa_vn(smem_addr(smem), static_cast<uint32_t>(r));
  // every CTA of the cluster has initialised its shared memory before any
  // other CTA stores into it (the first wait follows below)
  if constexpr (CL > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  else __syncthreads();

  // x operands of chunk c: units (vector column v, superblock); this CTA
  // converts units rank, rank + CL, ... (warp w: the w-th, (w+16)-th, ... of
  // those) and stores them into every CTA of the cluster; the loads of 2
  // units are issued before either is converted
  auto stage_chunk = [&](int c) {
    const int b0 = c * p.kc, nb = min(p.kc, p.nsb - b0);
    const int nunits = p.nv * nb;  // columns past nv stay unset: they only reach C columns nobody stores
    constexpr int kBatch = 2;
    for (int l0 = warp; static_cast<int>(rank) + CL * l0 < nunits; l0 += kVnWarps * kBatch) {
      float xv[kBatch][8];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int u = static_cast<int>(rank) + CL * (l0 + kVnWarps * k);
        const int v = u / nb, bl = u - v * nb;
        if (u < nunits) {
          const int j0 = (b0 + bl) * 256 + 8 * lane;  // the 8 columns lie in one head (head_dim % 32 == 0)
          const float *xr = p.x + v * p.x_stride + vn_x_src(j0, p.x_group, p.x_head_dim);
          const float4 a = *reinterpret_cast<const float4 *>(xr);
          const float4 b = *reinterpret_cast<const float4 *>(xr + 4);
          xv[k][0] = a.x, xv[k][1] = a.y, xv[k][2] = a.z, xv[k][3] = a.w;
          xv[k][4] = b.x, xv[k][5] = b.y, xv[k][6] = b.z, xv[k][7] = b.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) xv[k][e] = 0.0f;
        }
      }
      float mx[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) mx[k] = warp_absmax(k16::lane_absmax(xv[k]));
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int u = static_cast<int>(rank) + CL * (l0 + kVnWarps * k);
        if (u >= nunits) break;  // warp-uniform
        const int v = u / nb, bl = u - v * nb;
        const float sq = vn_stage<CL>(xv[k], mx[k], st, L.main + bl * kVnSbMain, L.minb + bl * kVnSbMin,
                                      L.ps + bl * 32, v, lane);
        if (p.rms) {
          const float s = warp_sum_xor<32>(sq);
          if (lane == 0) ssq_s[(rank * kVnWarps + warp) * 8 + v] += s;  // the warp's own slot
        }
      }
    }
  };

  // B operands: plain loads from the __shared__ array, which the compiler may
  // issue ahead of the preceding MMAs
  const uint8_t *main0 = smem + L.main + lane * 16;
  const uint8_t *min0 = smem + L.minb + lane * 8;
  if constexpr (CL > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  // Every CTA of a cluster runs the same barrier sequence, whatever its rows:
  // per chunk one barrier before the staging (c > 0: every CTA has finished
  // reading the previous chunk's operands) and one after it.
#pragma unroll 1
  for (int c = 0; c < p.nchunks; ++c) {
    if (c > 0) cl_sync<CL>();
    stage_chunk(c);
    __syncwarp();  // lane 0's sums of squares are visible to the warp's other lanes
    if (c == p.nchunks - 1 && p.rms && lane < 8) {  // this warp's sums of squares -> the other CTAs
      const uint32_t off = L.ssq + 4u * ((rank * kVnWarps + warp) * 8 + lane);
      const float vq = ssq_s[(rank * kVnWarps + warp) * 8 + lane];
#pragma unroll
      for (int r = 0; r < CL; ++r)
        if (r != static_cast<int>(rank)) {
          if constexpr (CL > 1) asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(st.base[r] + off), "f"(vq) : "memory");
        }
    }
    cl_sync<CL>();
    if (c == p.nchunks - 1 && p.rms && threadIdx.x < 8) {
      float q = 0.0f;
      for (int w = 0; w < CL * kVnWarps; ++w) q += ssq_s[w * 8 + threadIdx.x];
      rs_s[threadIdx.x] =
          __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q, static_cast<float>(p.nsb * 256)), p.rms_eps)));
    }  // read in the epilogue, after at least one more barrier
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    const int pass = c * iters + it;
    // ------------------------------------------------------------ this pass's superblocks
    float acc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};  // rows g, g + 8 x vectors 2t, 2t + 1
    const int pcnt = cnt, pbase = bbase;
    const uint8_t *plo = row_lo, *phi = row_hi;
    for (int j0 = 0; j0 < pcnt; j0 += kDepth) {
#pragma unroll
      for (int d = 0; d < kDepth; ++d) {
        const int jj = j0 + d;
        if (jj >= pcnt) break;
        const int b = pbase + jj * p.kp;
        const int bl = b - c * p.kc;
        const RowOps<EPQ_Q4_K> &lo = ring_lo[d], &hi = ring_hi[d];
        float cl[2], kl[2], ch[2], kh[2];
        k16::q4k_codes(lo.hdr, t, cl, kl);
        k16::q4k_codes(hi.hdr, t, ch, kh);
        // scale multipliers: class A c 2^10, class B c 2^6 (sub-blocks 2t, 2t + 1)
        const uint32_t sAl0 = half2_bits(cl[0] * 1024.0f, cl[0] * 1024.0f), sBl0 = half2_bits(cl[0] * 64.0f, cl[0] * 64.0f);
        const uint32_t sAl1 = half2_bits(cl[1] * 1024.0f, cl[1] * 1024.0f), sBl1 = half2_bits(cl[1] * 64.0f, cl[1] * 64.0f);
        const uint32_t sAh0 = half2_bits(ch[0] * 1024.0f, ch[0] * 1024.0f), sBh0 = half2_bits(ch[0] * 64.0f, ch[0] * 64.0f);
        const uint32_t sAh1 = half2_bits(ch[1] * 1024.0f, ch[1] * 1024.0f), sBh1 = half2_bits(ch[1] * 64.0f, ch[1] * 64.0f);
        // four independent accumulators (word half h x hi / lo) keep the MMA chains short
        float cm[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cm[q][0] = cm[q][1] = cm[q][2] = cm[q][3] = 0.0f;
        const uint8_t *mb = main0 + bl * kVnSbMain;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t sAl = j < 4 ? sAl0 : sAl1, sBl = j < 4 ? sBl0 : sBl1;
          const uint32_t sAh = j < 4 ? sAh0 : sAh1, sBh = j < 4 ? sBh0 : sBh1;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wl = h ? lo.qs[j] >> 8 : lo.qs[j];
            const uint32_t wh = h ? hi.qs[j] >> 8 : hi.qs[j];
            const uint32_t a[4] = {hmul2u(wl & k16::kNibA, sAl), hmul2u(wh & k16::kNibA, sAh),
                                   hmul2u(wl & k16::kNibB, sBl), hmul2u(wh & k16::kNibB, sBh)};
            const uint4 bb = *reinterpret_cast<const uint4 *>(mb + j * kVnPair + h * kVnMma);
            k16::mma(cm[2 * h], a, make_uint2(bb.x, bb.y));
            k16::mma(cm[2 * h + 1], a, make_uint2(bb.z, bb.w));
          }
        }
        // min term: k-slots 2t, 2t + 1 = the lane's sub-blocks
        float cn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        {
          const uint32_t am[4] = {half2_bits(kl[0], kl[1]), half2_bits(kh[0], kh[1]), 0u, 0u};
          const uint2 xb = *reinterpret_cast<const uint2 *>(min0 + bl * kVnSbMin);
          k16::mma(cn, am, make_uint2(xb.x, 0u));
          k16::mma(cn, am, make_uint2(xb.y, 0u));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) cm[0][e] = (cm[0][e] + cm[1][e]) + (cm[2][e] + cm[3][e]);
        const float2 ps = *reinterpret_cast<const float2 *>(ps_s + bl * 8 + 2 * t);
        const float dl = half_bits_to_float(lo.hdr.x) * 512.0f, ml = half_bits_to_float(lo.hdr.x >> 16);
        const float dh = half_bits_to_float(hi.hdr.x) * 512.0f, mh = half_bits_to_float(hi.hdr.x >> 16);
        acc[0][0] = fmaf(ps.x, fmaf(dl, cm[0][0], -ml * cn[0]), acc[0][0]);
        acc[0][1] = fmaf(ps.y, fmaf(dl, cm[0][1], -ml * cn[1]), acc[0][1]);
        acc[1][0] = fmaf(ps.x, fmaf(dh, cm[0][2], -mh * cn[2]), acc[1][0]);
        acc[1][1] = fmaf(ps.y, fmaf(dh, cm[0][3], -mh * cn[3]), acc[1][1]);
        if (jj + kDepth < pcnt) {
          k16::load_ops<EPQ_Q4_K, 16>(ring_lo[d], plo, nsb, b + kDepth * p.kp, t);
          k16::load_ops<EPQ_Q4_K, 16>(ring_hi[d], phi, nsb, b + kDepth * p.kp, t);
        }
      }
    }
    if (pass + 1 < npass) fill(pass + 1);  // the next pass's first superblocks fly over the reduction

    // ------------------------------------------------------------ row totals
    red[(warp * 16 + g) * 8 + 2 * t] = acc[0][0];
    red[(warp * 16 + g) * 8 + 2 * t + 1] = acc[0][1];
    red[(warp * 16 + g + 8) * 8 + 2 * t] = acc[1][0];
    red[(warp * 16 + g + 8) * 8 + 2 * t + 1] = acc[1][1];
    __syncthreads();
    const bool last = c == p.nchunks - 1;
    const int nsum = p.rg * 16 * 8;
    for (int idx = threadIdx.x; idx < nsum; idx += kVnThreads) {
      const int gl = idx / 128, r = idx - gl * 128;  // r = row 16 x vector 8
      float s = 0.0f;
      for (int k = 0; k < p.kp; ++k) s += red[(gl * p.kp + k) * 128 + r];
      if (p.nchunks > 1) {
        float *pp = part + (it * p.rg + gl) * 128 + r;
        s = c == 0 ? s : *pp + s;
        if (!last) *pp = s;
      }
      if (last) red[(gl * p.kp) * 128 + r] = s;  // the k-part 0 slot of the group now holds its total
    }
    if (last) {
      __syncthreads();
      const int nout = p.rg * kOut * 8;
      for (int idx = threadIdx.x; idx < nout; idx += kVnThreads) {
        const int v = idx & 7, o = (idx >> 3) % kOut, gl = idx / (8 * kOut);
        const int64_t i = (first + it * stride + gl) * kOut + o;
        if (v >= p.nv || i >= p.rows_out) continue;
        const float r = rs_s[v];
        const float *tot = red + (gl * p.kp) * 128;
        float val = tot[o * 8 + v] * r;
        if (SW) val = vn_silu(val) * (tot[(o + 8) * 8 + v] * r);
        if (p.residual) val += p.residual[v * p.y_stride + i];
        p.y[v * p.y_stride + i] = val;
      }
    }
    __syncthreads();  // red (and the chunk's x operands) are rewritten next
  }
  }
}

template <bool SW, int CL>
void vn_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[2], unsigned grid, uint32_t smem,
               cudaStream_t s) {
  cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kVnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  int n = 0;
  if (CL > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = CL;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
}

template <bool SW, int CL>
cudaError_t launch_vn(const VnParams &p, unsigned grid, uint32_t smem, cudaStream_t s) {
  auto k = gemv_vn_kernel<SW, CL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  vn_config<SW, CL>(cfg, attr, grid, smem, s);
  return cudaLaunchKernelEx(&cfg, k, p);
}

// CTAs of clusters of CL that can be resident at once (one CTA per SM);
// cached per (device, CL, shared memory).
template <int CL>
int64_t vn_resident_ctas(const DeviceInfo &dev, uint32_t smem) {
  if (CL == 1) return dev.sm_count;
  static std::mutex mu;
  static std::map<std::pair<int, uint32_t>, int64_t> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev.device, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  auto k = gemv_vn_kernel<false, CL>;
  int64_t ctas = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) == cudaSuccess) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    vn_config<false, CL>(cfg, attr, static_cast<unsigned>(CL * dev.sm_count), smem, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess) ctas = static_cast<int64_t>(n) * CL;
  }
  (void)cudaGetLastError();  // a failed query leaves no error behind; the caller then runs without clusters
  cache[key] = ctas;
  return ctas;
}

}  // namespace

// Called by gemv_launch (gemv.cu) for Q4_K with 2..8 vectors.  Geometry:
// x operands of up to KC superblocks per chunk (all of the row when they fit
// next to the other buffers, else the fewest equal chunks that fit; the
// tuning cap EPQ_TUNE_VN_CHUNK lowers KC), one CTA per SM in clusters of CL
// (each CTA converts 1/CL of the operands for all of them; EPQ_TUNE_VN_CLUSTER
// picks CL), and the row groups split like the block-diagonal engine's (RG
// groups per CTA iteration, the 16 warps splitting the chunk's superblocks
// KP = 16 / RG ways).
epq_status gemv_vn_launch(const void *blocks, const float *x, float *y, int64_t rows, int64_t cols, int nvec,
                          const epq_gemv_opts &o, int64_t x_stride, const DeviceInfo &dev, cudaStream_t s) {
  const bool sw = o.swiglu != 0;
  const int64_t rows_out = sw ? rows / 2 : rows;
  const int nsb = static_cast<int>(cols / 256);
  const int64_t ngroups = (rows_out + (sw ? 7 : 15)) / (sw ? 8 : 16);
  const uint32_t budget = static_cast<uint32_t>(dev.max_smem_optin);
  int cl = tune_vn_cluster() > 0 ? tune_vn_cluster() : 2;
  // chunk: the whole row when its x operands fit (the partial-sum buffer,
  // a few KB, counted at its largest), else the fewest equal chunks that do
  int kc = nsb;
  if (tune_vn_chunk() > 0) kc = std::min(kc, tune_vn_chunk());
  int nchunks = (nsb + kc - 1) / kc;
  const int64_t sms = dev.sm_count;
  auto fits = [&](int kc_, int nch_) {
    return vn_layout(kc_, nch_, kVnWarps, static_cast<int>((ngroups + sms - 1) / sms), cl).total <= budget;
  };
  while (!fits(kc, nchunks) && kc > 1) {
    kc = (nsb + nchunks) / (nchunks + 1);
    nchunks = (nsb + kc - 1) / kc;
  }
  const uint32_t smem_bound = vn_layout(kc, nchunks, kVnWarps, static_cast<int>((ngroups + sms - 1) / sms), cl).total;
  if (smem_bound > budget) return EPQ_ERR_SHAPE;
  // resident CTAs: clusters may leave SMs of a GPC unused
  int64_t cap = cl == 4 ? vn_resident_ctas<4>(dev, smem_bound) : cl == 2 ? vn_resident_ctas<2>(dev, smem_bound) : sms;
  if (cap < cl) {
    cl = 1;
    cap = sms;
  }
  // RG among those that give every resident CTA a block: the fewest per-CTA
  // iterations x (superblocks per warp + one reduction per chunk), ties to
  // the larger RG; RG = 1 when none fills the GPU
  int rg = 1;
  int64_t best = -1;
  for (int r = kVnWarps; r >= 1; r >>= 1) {
    const int64_t blocks = (ngroups + r - 1) / r;
    if (blocks < cap) continue;
    const int64_t kpr = kVnWarps / r;
    const int64_t cost = (blocks + cap - 1) / cap * ((kc + kpr - 1) / kpr * nchunks + nchunks);
    if (best < 0 || cost < best) {
      best = cost;
      rg = r;
    }
  }
  int64_t g = std::min<int64_t>((ngroups + rg - 1) / rg, cap);
  g = std::max<int64_t>(cl, g / cl * cl);  // whole clusters (CTAs past the rows only convert operands)
  const unsigned grid = static_cast<unsigned>(g);
  const int iters_max =
      static_cast<int>((ngroups + static_cast<int64_t>(grid) * rg - 1) / (static_cast<int64_t>(grid) * rg));
  const VnLayout L = vn_layout(kc, nchunks, rg, iters_max, cl);
  if (L.total > budget) return EPQ_ERR_SHAPE;
  VnParams p;
  p.W = static_cast<const uint8_t *>(blocks);
  p.rows_out = rows_out;
  p.up_rows = sw ? rows_out : 0;
  p.row_bytes = epq_row_bytes(EPQ_Q4_K, cols);
  p.nsb = nsb;
  p.kc = kc;
  p.nchunks = nchunks;
  p.rg = rg;
  p.kp = kVnWarps / rg;
  p.iters_max = iters_max;
  p.x_stride = x_stride;
  p.y_stride = rows_out;
  p.rms = o.rms_prenorm;
  p.rms_eps = o.rms_eps;
  p.x_group = o.x_group > 1 ? o.x_group : 1;
  p.x_head_dim = o.x_head_dim;
  p.early = o.weights_ready ? 1 : 0;
  for (int v0 = 0; v0 < nvec; v0 += 8) {
    p.nv = std::min(8, nvec - v0);
    p.x = x + v0 * x_stride;
    p.y = y + v0 * rows_out;
    p.residual = o.residual ? o.residual + v0 * rows_out : nullptr;
    cudaError_t e;
    if (cl == 4) e = sw ? launch_vn<true, 4>(p, grid, L.total, s) : launch_vn<false, 4>(p, grid, L.total, s);
    else if (cl == 2) e = sw ? launch_vn<true, 2>(p, grid, L.total, s) : launch_vn<false, 2>(p, grid, L.total, s);
    else e = sw ? launch_vn<true, 1>(p, grid, L.total, s) : launch_vn<false, 1>(p, grid, L.total, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return EPQ_OK;
}

}  // namespace epq

// Decode-step attention over a Q8_0 key/value cache with a skip threshold
// (epq_attention_decode).
//
// "smolmaxxing", compute table, row "带阈值的 Q8_0 注意力": the keys and values
// of the cache are held in Q8_0 blocks; every key dot product of the step is
// computed first, so the softmax maximum M is known before any exponential,
// and positions whose score falls below M + ln(1e-4) are skipped -- no
// exponential and no read of their value row.  The kept positions get the
// usual softmax weights exp(s - M) / sum exp(s - M) over the kept set.
//
// One token (batch 1), grouped heads: query head hq reads key/value head
// hq / group.  A step appends the token's own key and value (quantized to
// Q8_0 with the packer's arithmetic) at position `pos` and attends over
// positions 0..pos.
//
// Organisation: one thread-block cluster of C CTAs per key/value head (the
// positions split evenly over the C CTAs).
//   entry    before the grid-dependency wait the CTA asks L2 for its cached
//            key and value rows (written by earlier steps; a prefetch hint
//            only); after it, every thread issues asynchronous 8-byte copies
//            of those rows into shared memory (keys and values as two copy
//            groups, in chunks when the rows do not fit), so that one round
//            trip brings every row the CTA reads;
//   phase 0  the query elements a lane uses go straight into registers; the
//            CTA whose positions include `pos` quantizes the step's key and
//            value rows into the cache and keeps a shared-memory copy for its
//            own scan (no other CTA reads them in this step);
//   phase 1  each warp takes runs of 8 consecutive positions: lane l holds 4
//            consecutive elements of a key row (one 32-bit word of codes plus
//            its block's fp16 factor, from shared memory) and multiplies them
//            with the `group` query heads; one reduce-scatter gives the run's
//            dot products; scores stay in shared memory (and optionally go to
//            scores_out); each CTA writes its per-head maximum into every
//            cluster CTA's shared memory (distributed shared memory), one
//            cluster barrier;
//   phase 2  each CTA forms the weights of its positions against the
//            cluster-wide maximum, skips the positions below the threshold
//            (for every query head of the group: no exponential, no value
//            arithmetic), accumulates the weighted value rows and the weight
//            sums, reduces over its warps and writes the partial into cluster
//            rank 0's shared memory; after a cluster barrier rank 0 adds the C
//            partials in rank order and writes out = sum w v / sum w.
// The value rows of skipped positions are copied with the others: the copy
// is one round trip either way, and the page's saving is the arithmetic.
// Every sum runs in a fixed order, so the result is bitwise reproducible.
// There is no spin wait in this kernel (asynchronous copies waited with
// cp.async.wait_group, cluster barriers that every thread reaches).
//
// Cache row layout (this library's own byte order; the values are Q8_0
// blocks of 32 elements, fp16 factor d and int8 codes q, element = d * q):
// position p of key/value head h is the D + D/16 byte row at
// (h * max_pos + p) * (D + D/16): the D/32 fp16 factors first, then the D
// int8 codes, so that a lane's 4 codes are one aligned 32-bit word.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace epq {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxGroup = 8;       // query heads per key/value head
constexpr int kMaxCluster = 8;
constexpr int kMaxPosPerCta = 2048;
constexpr int kRunMax = 8;         // positions per warp step

struct AttnParams {
  const float *q;               // [n_heads][D]
  const float *k_new, *v_new;   // [n_kv][D] (the step's key and value)
  uint8_t *k_cache, *v_cache;   // [n_kv][max_pos][row]
  float *out;                   // [n_heads][D]
  float *scores;                // NULL or [n_heads][max_pos]
  int n_kv, D, group, pos, max_pos, C;
  int nsp;    // score stride per query head (>= positions of a CTA)
  int chunk;  // rows of one shared-memory copy chunk
  float scale, skip_log;
};

__host__ __device__ inline uint32_t al16b(uint32_t v) { return (v + 15u) & ~15u; }

// Shared-memory plan of one CTA (byte offsets, 16-byte aligned).
struct AttnSmem {
  uint32_t sc, cmax, red, part, newrow, stage, total;
};

__host__ __device__ inline AttnSmem attn_smem(int G, int D, int C, int nsp, int chunk) {
  AttnSmem L;
  const uint32_t rb = static_cast<uint32_t>(D + D / 16);
  uint32_t o = 0;
  L.sc = o;  // [G][nsp] scores, then weights
  o = al16b(o + 4u * G * nsp);
  L.cmax = o;  // [kMaxCluster][G] maxima from every cluster CTA
  o = al16b(o + 4u * kMaxCluster * G);
  L.red = o;  // [warp][G][D + 1] warp partials (warp maxima first)
  o = al16b(o + 4u * kAttnWarps * G * (D + 1));
  L.part = o;  // [C][G][D + 1] partials of every CTA (rank 0 only)
  o = al16b(o + 4u * C * G * (D + 1));
  L.newrow = o;  // [2][row] the step's key and value rows
  o = al16b(o + 2u * rb);
  L.stage = o;  // [2][chunk][row] copied key rows, value rows
  o = al16b(o + 2u * static_cast<uint32_t>(chunk) * rb);
  L.total = o;
  return L;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v at the shared-memory address `local` of cluster CTA `rank`.
__device__ __forceinline__ void st_cluster(const float *local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Q8_0 of one 32-element run held one element per lane (the packer's
// arithmetic: factor fp16(max|x| / 127), codes rint(x / factor) clamped to
// +-127, zero codes for a zero factor).
__device__ __forceinline__ void q8_block_lane(float x, uint16_t *d_out, int8_t *q_out) {
  x = __fadd_rn(x, 0.0f);  // -0 -> +0
  float a = fabsf(x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const __half dh = __float2half_rn(__fdiv_rn(a, 127.0f));
  const float d = __half2float(dh);
  float q = 0.0f;
  if (d != 0.0f) q = fminf(fmaxf(rintf(__fdiv_rn(x, d)), -127.0f), 127.0f);
  *q_out = static_cast<int8_t>(q);
  if ((threadIdx.x & 31) == 0) *d_out = __half_as_ushort(dh);
}

// 8-byte asynchronous copy global -> shared (L1-allocating form), and the
// per-thread copy groups.
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)),
               "l"(static_cast<uint64_t>(__cvta_generic_to_global(src)))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Sum over the warp of N values per lane (N a power of two <= 32): a
// reduce-scatter that halves the set of values each lane carries at every
// level (offsets 16, 8, ...), then plain butterflies once one value is left.
// Lane l returns the warp total of value l / (32 / N) (the high bits of the
// lane pick the value; the 32 / N lanes of a run hold the same total).
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
  int n = N;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (n > 1) {
      const bool up = (lane & o) != 0;
      const int half = n / 2;
#pragma unroll
      for (int j = 0; j < N / 2; ++j) {
        if (j >= half) break;
        const float send = up ? v[j] : v[j + half];
        const float keep = up ? v[j + half] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

// Exact float of int8 code b of a word: with u = q + 128 (the code's byte
// with its top bit flipped), the bit pattern 0x4B0000uu is the float 2^23 + u.
__device__ __forceinline__ float i8(uint32_t wflip, int b) {
  const uint32_t sel = static_cast<uint32_t>(b) | 0x7540u;  // byte b, then zero, zero, 0x4B
  return __uint_as_float(__byte_perm(wflip, 0x4B000000u, sel)) - 8388736.0f;
}

template <int G>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_decode_kernel(const __grid_constant__ AttnParams p) {
  // kRun positions per warp step, so that a step's kRun x G dot products fit one reduce-scatter
  constexpr int kRun = kRunMax * G <= 32 ? kRunMax : 32 / G;
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D;
  const int C = p.C;
  const uint32_t rank = cluster_rank();
  const int h = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row_bytes = D + D / 16;
  const int nblk = D / 32;
  // positions of this CTA; those below `pos` come from the cache
  const int npos = p.pos + 1;
  const int p0 = static_cast<int>((static_cast<int64_t>(rank) * npos) / C);
  const int p1 = static_cast<int>((static_cast<int64_t>(rank + 1) * npos) / C);
  const int n = p1 - p0;
  const int ncached = min(p1, p.pos) - p0;
  const int chunk = p.chunk;
  const int nsp = p.nsp;

  const AttnSmem L = attn_smem(G, D, C, nsp, chunk);
  float *sc = reinterpret_cast<float *>(smem + L.sc);
  float *cmax = reinterpret_cast<float *>(smem + L.cmax);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *part = reinterpret_cast<float *>(smem + L.part);
  uint8_t *newrow = smem + L.newrow;
  uint8_t *stk = smem + L.stage;                // [chunk][row] key rows
  uint8_t *stv = stk + chunk * row_bytes;       // [chunk][row] value rows
  const int64_t head_row0 = static_cast<int64_t>(h) * p.max_pos + p0;
  const uint8_t *kc = p.k_cache + head_row0 * row_bytes;
  const uint8_t *vc = p.v_cache + head_row0 * row_bytes;

  // L2 hint for the cached rows (a prefetch cannot expose stale data: the
  // rows are read only after the grid-dependency wait)
  {
    const int lines = (ncached * row_bytes + 127) / 128;
    for (int i = tid; i < 2 * lines; i += kAttnThreads) {
      const uint8_t *a = (i < lines ? kc : vc) + 128 * static_cast<int64_t>(i < lines ? i : i - lines);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<uint64_t>(__cvta_generic_to_global(a))));
    }
  }
  pdl_launch_dependents();
  pdl_wait();  // q, k_new and v_new come from the preceding projection

  // rows [c0, c0 + cn) of this CTA's positions -> dst, 8-byte copies (rows
  // are 8-byte multiples; the step's own position is never copied)
  auto stage_rows = [&](const uint8_t *src_rows, uint8_t *dst, int c0, int cn) {
    const int pieces = max(0, min(cn, ncached - c0)) * row_bytes / 8;
    const uint8_t *src = src_rows + static_cast<int64_t>(c0) * row_bytes;
    for (int i = tid; i < pieces; i += kAttnThreads) cp_async8(dst + 8 * i, src + 8 * i);
  };
  const bool one_chunk = n <= chunk;
  stage_rows(kc, stk, 0, chunk);
  cp_async_commit();
  if (one_chunk) stage_rows(vc, stv, 0, chunk);
  cp_async_commit();

  // ---------------------------------------------------------------- phase 0
  // Arrive on the cluster barrier now and wait on it only before the first
  // store into another CTA's shared memory: every CTA of the cluster has
  // then started.  The lane's query elements go into registers for the whole
  // scan.  The CTA whose range holds position `pos` quantizes the step's key
  // and value rows, stores them into the cache and keeps a shared-memory
  // copy for its scan.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const int nch = D / 128;
  float4 qr[G][2];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int c = 0; c < 2; ++c)
      qr[g][c] = c < nch ? *reinterpret_cast<const float4 *>(p.q + (h * G + g) * D + 128 * c + 4 * lane)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
  const bool owner = p0 <= p.pos && p.pos < p1;
  if (owner) {
    uint8_t *krow_new = p.k_cache + (static_cast<int64_t>(h) * p.max_pos + p.pos) * row_bytes;
    uint8_t *vrow_new = p.v_cache + (static_cast<int64_t>(h) * p.max_pos + p.pos) * row_bytes;
    // warps 0..nblk-1 quantize the key blocks, the next nblk warps the value blocks
    for (int b = warp; b < 2 * nblk; b += kAttnWarps) {
      const bool isv = b >= nblk;
      const int bb = isv ? b - nblk : b;
      const float x = (isv ? p.v_new : p.k_new)[h * D + 32 * bb + lane];
      uint8_t *row = isv ? vrow_new : krow_new;
      uint8_t *copy = newrow + (isv ? row_bytes : 0);
      uint16_t d;
      int8_t q;
      q8_block_lane(x, &d, &q);
      row[2 * nblk + 32 * bb + lane] = copy[2 * nblk + 32 * bb + lane] = static_cast<uint8_t>(q);
      if (lane == 0) {
        *reinterpret_cast<uint16_t *>(row + 2 * bb) = d;
        *reinterpret_cast<uint16_t *>(copy + 2 * bb) = d;
      }
    }
  }
  cp_async_wait<1>();  // this thread's key copies (the value group may still be in flight)
  __syncthreads();

  // ---------------------------------------------------------------- phase 1
  // Warp w takes runs of kRun consecutive positions (w*kRun + 8*kRun*j ...)
  // of each chunk.  Lane l: elements 4l..4l+3 of each 128-element chunk.
  float wmax[G];
#pragma unroll
  for (int g = 0; g < G; ++g) wmax[g] = -INFINITY;
#pragma unroll 1
  for (int c0 = 0; c0 < n; c0 += chunk) {
    const int cend = min(n, c0 + chunk);
    if (c0 > 0) {  // a later chunk (long contexts): the previous one is no longer read
      __syncthreads();
      stage_rows(kc, stk, c0, chunk);
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
    }
#pragma unroll 1
    for (int i0 = c0 + warp * kRun; i0 < cend; i0 += kAttnWarps * kRun) {
      uint32_t wk[kRun][2];
      float dk[kRun][2];
#pragma unroll
      for (int u = 0; u < kRun; ++u) {
        const int i = min(i0 + u, cend - 1);  // past the end: a repeat of the last row, not used
        const uint8_t *row = p0 + i == p.pos ? newrow : stk + (i - c0) * row_bytes;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c >= nch) break;
          const int e0 = 128 * c + 4 * lane;
          wk[u][c] = *reinterpret_cast<const unsigned int *>(row + 2 * nblk + e0);
          dk[u][c] = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short *>(row + 2 * (e0 / 32))));
        }
      }
      // partial dots of the run's kRun x G (position, head) pairs, then one
      // reduce-scatter over the warp: lane l ends with the full sum of pair
      // l / (32 / (kRun G)) (index u G + g), instead of one butterfly per pair
      float acc[kRun * G];
#pragma unroll
      for (int u = 0; u < kRun; ++u) {
#pragma unroll
        for (int g = 0; g < G; ++g) acc[u * G + g] = 0.0f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c >= nch) break;
          // the lane's 4 elements share one Q8_0 block: the factor d multiplies their sum
          const uint32_t w = wk[u][c] ^ 0x80808080u;
          const float k0 = i8(w, 0), k1 = i8(w, 1), k2 = i8(w, 2), k3 = i8(w, 3);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float4 qv = qr[g][c];
            acc[u * G + g] = fmaf(dk[u][c], fmaf(k0, qv.x, fmaf(k1, qv.y, fmaf(k2, qv.z, k3 * qv.w))), acc[u * G + g]);
          }
        }
      }
      const float sum = reduce_scatter<kRun * G>(acc, lane);
      constexpr int kPairs = kRun * G;
      constexpr int kCopies = 32 / kPairs;  // lanes holding the same pair
      const int pr = lane / kCopies;        // pair held by this lane
      const int u = pr / G, g = pr % G;
      const float sv = sum * p.scale;
      if (i0 + u < cend) {
        if (lane % kCopies == 0) sc[g * nsp + i0 + u] = sv;
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
          if (gg == g) wmax[gg] = fmaxf(wmax[gg], sv);  // constant indices keep wmax in registers
      }
    }
  }
  // CTA maxima -> every cluster CTA's cmax[rank][g]
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float m = wmax[g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp * G + g] = m;  // red holds the warp maxima until phase 2
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every cluster CTA has started
  if (tid < G) {
    float m = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) m = fmaxf(m, red[w * G + tid]);
    for (int r = 0; r < C; ++r) st_cluster(&cmax[rank * G + tid], static_cast<uint32_t>(r), m);
  }
  if (p.scores) {
    for (int idx = tid; idx < G * n; idx += kAttnThreads) {
      const int g = idx / n, i = idx % n;
      p.scores[static_cast<int64_t>(h * G + g) * p.max_pos + p0 + i] = sc[g * nsp + i];
    }
  }
  cluster_sync();

  // ---------------------------------------------------------------- phase 2
  // weights once per (head, position), in place of the scores: exp(s - M)
  // for kept positions, 0 for skipped ones
  for (int idx = tid; idx < G * n; idx += kAttnThreads) {
    const int g = idx / n, i = idx - g * n;
    float m = -INFINITY;  // the cluster maximum of head g (from shared memory: g is not a constant here)
    for (int r = 0; r < C; ++r) m = fmaxf(m, cmax[r * G + g]);
    const float sv = sc[g * nsp + i];
    sc[g * nsp + i] = sv >= m + p.skip_log ? expf(sv - m) : 0.0f;
  }
  if (one_chunk) cp_async_wait<0>();  // this thread's value copies
  __syncthreads();
  float o[G][4 * 2];  // up to D = 256: two 128-element chunks of 4 per lane
  float ws[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    ws[g] = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) o[g][j] = 0.0f;
  }
  // the same runs of positions; a position that no query head keeps costs
  // no value arithmetic
#pragma unroll 1
  for (int c0 = 0; c0 < n; c0 += chunk) {
    const int cend = min(n, c0 + chunk);
    if (!one_chunk) {
      __syncthreads();
      stage_rows(vc, stv, c0, chunk);
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
    }
#pragma unroll 1
    for (int i0 = c0 + warp * kRun; i0 < cend; i0 += kAttnWarps * kRun) {
      float w[kRun][G];
      bool need[kRun];
#pragma unroll
      for (int u = 0; u < kRun; ++u) {
        need[u] = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          w[u][g] = i0 + u < cend ? sc[g * nsp + i0 + u] : 0.0f;
          need[u] = need[u] || w[u][g] != 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < kRun; ++u) {
        if (!need[u]) continue;  // warp-uniform: every lane read the same weights
        const uint8_t *row = p0 + i0 + u == p.pos ? newrow + row_bytes : stv + (i0 + u - c0) * row_bytes;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (c >= nch) break;
          const int e0 = 128 * c + 4 * lane;
          const uint32_t wq = *reinterpret_cast<const unsigned int *>(row + 2 * nblk + e0) ^ 0x80808080u;
          const float dv = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short *>(row + 2 * (e0 / 32))));
          const float v0 = i8(wq, 0), v1 = i8(wq, 1), v2 = i8(wq, 2), v3 = i8(wq, 3);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float wd = w[u][g] * dv;  // weight times the block factor of the lane's elements
            o[g][4 * c + 0] = fmaf(wd, v0, o[g][4 * c + 0]);
            o[g][4 * c + 1] = fmaf(wd, v1, o[g][4 * c + 1]);
            o[g][4 * c + 2] = fmaf(wd, v2, o[g][4 * c + 2]);
            o[g][4 * c + 3] = fmaf(wd, v3, o[g][4 * c + 3]);
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) ws[g] += w[u][g];
      }
    }
  }
  // warp partials -> shared memory, then the CTA sum (warp order) -> rank 0
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float *rw = red + (warp * G + g) * (D + 1);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (c >= nch) break;
#pragma unroll
      for (int j = 0; j < 4; ++j) rw[128 * c + 4 * lane + j] = o[g][4 * c + j];
    }
    if (lane == 0) rw[D] = ws[g];
  }
  __syncthreads();
  for (int idx = tid; idx < G * (D + 1); idx += kAttnThreads) {
    float s = 0.0f;
    for (int w = 0; w < kAttnWarps; ++w) s += red[w * G * (D + 1) + idx];
    st_cluster(&part[rank * G * (D + 1) + idx], 0u, s);
  }
  cluster_sync();
  if (rank == 0) {
    for (int idx = tid; idx < G * D; idx += kAttnThreads) {
      const int g = idx / D, e = idx % D;
      float num = 0.0f, den = 0.0f;
      for (int r = 0; r < C; ++r) {
        num += part[(r * G + g) * (D + 1) + e];
        den += part[(r * G + g) * (D + 1) + D];
      }
      p.out[(h * G + g) * D + e] = num / den;
    }
  }
}

template <int G>
cudaError_t launch_attn(const AttnParams &p, cudaStream_t s) {
  auto k = attn_decode_kernel<G>;
  const size_t smem = attn_smem(G, p.D, p.C, p.nsp, p.chunk).total;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_kv * p.C));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace
}  // namespace epq

using namespace epq;

extern "C" int64_t epq_kv_row_bytes(int head_dim) {
  if (head_dim <= 0 || head_dim % 128 || head_dim > 256) return -1;
  return head_dim + head_dim / 16;
}

extern "C" epq_status epq_attention_decode(const float *q, const float *k_new, const float *v_new, void *k_cache,
                                           void *v_cache, int n_heads, int n_kv_heads, int head_dim, int pos,
                                           int max_pos, float scale, float skip_log, float *out, float *scores_out,
                                           epq_stream_t stream) {
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !out) return EPQ_ERR_ARG;
  if (n_kv_heads < 1 || n_heads < n_kv_heads || n_heads % n_kv_heads) return EPQ_ERR_SHAPE;
  const int G = n_heads / n_kv_heads;
  if (G > kMaxGroup || (G & (G - 1))) return EPQ_ERR_SHAPE;
  if (epq_kv_row_bytes(head_dim) < 0) return EPQ_ERR_SHAPE;
  if (max_pos < 1 || pos < 0 || pos >= max_pos) return EPQ_ERR_ARG;
  if (!(scale > 0.0f) || std::isnan(skip_log)) return EPQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(out) || (scores_out && !aligned16(scores_out)))
    return EPQ_ERR_ALIGN;
  // cluster size: enough CTAs that each has at most 64 positions (up to 8
  // CTAs); positions per CTA bounded by its shared-memory score buffer
  int C = 1;
  while (C < kMaxCluster && (pos + 1 + C - 1) / C > 64) C *= 2;
  if ((pos + 1 + C - 1) / C > kMaxPosPerCta) return EPQ_ERR_SHAPE;
  DeviceInfo dev;
  if (!current_device(&dev) || dev.major * 10 + dev.minor < 100) return EPQ_ERR_DEVICE;
  AttnParams p;
  p.q = q;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_cache = static_cast<uint8_t *>(k_cache);
  p.v_cache = static_cast<uint8_t *>(v_cache);
  p.out = out;
  p.scores = scores_out;
  p.n_kv = n_kv_heads;
  p.D = head_dim;
  p.group = G;
  p.pos = pos;
  p.max_pos = max_pos;
  p.C = C;
  // scores: positions of the largest CTA range, rounded to 4; key/value
  // rows copied in chunks that fit the rest of the shared memory (the whole
  // range in one chunk whenever it fits)
  const int nmax = (pos + 1 + C - 1) / C;
  p.nsp = (nmax + 3) & ~3;
  const int64_t fixed = attn_smem(G, head_dim, C, p.nsp, 0).total;
  const int64_t fit = (static_cast<int64_t>(dev.max_smem_optin) - fixed) / (2 * epq_kv_row_bytes(head_dim));
  int64_t chunk = std::min<int64_t>((nmax + 7) & ~7, fit & ~int64_t(7));
  if (tune_attn_chunk() > 0) chunk = std::min<int64_t>(chunk, tune_attn_chunk());
  p.chunk = static_cast<int>(chunk);
  if (p.chunk < 8) return EPQ_ERR_SHAPE;
  p.scale = scale;
  p.skip_log = skip_log;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaErrorInvalidValue;
  switch (G) {
    case 1: e = launch_attn<1>(p, s); break;
    case 2: e = launch_attn<2>(p, s); break;
    case 4: e = launch_attn<4>(p, s); break;
    case 8: e = launch_attn<8>(p, s); break;
  }
  return e == cudaSuccess ? EPQ_OK : cuda_fail(e);
}

// Shared part of the MoE layer (moe.cu, moe_tc.cu): limits, workspace
// layout, kernel arguments, the routing (softmax + top-K + grouping, run
// inside a CTA) and the routing reload of the down kernels.
//
// "Flash-MoE：在笔记本上运行 397B 参数大模型", section "每层流水线": the router
// matvec, then softmax and top-K over its logits, then the selected experts.
#pragma once

#include "gemv_core.cuh"

namespace epq {

// Arguments of every MoE kernel (one definition for both translation units).
struct MoeArgs {
  // router
  const float *R;
  const float *bias;
  const float *gvec;
  int E, H, I, ntok, topk, norm_topk, rms;
  float eps;
  int has_shared;
  // experts
  const uint8_t *gate_up;
  int64_t gu_stride;
  const uint8_t *down;
  int64_t dn_stride;
  const uint8_t *sh_gate_up;
  const uint8_t *sh_down;
  int64_t gu_row_bytes, dn_row_bytes;
  // io
  const float *x;
  float *y;
  int32_t *out_idx;
  float *out_w;
  // workspace views
  float *logits;
  float *xstat;      // [ntok][2]: max|x| (as float), rms factor
  float *gshared;    // [ntok]
  int32_t *idx;      // [ntok][topk]
  float *w;          // [ntok][topk]
  int32_t *meta;     // [0] = n_active, [1] = n_slots
  int32_t *active;   // [slots] expert id
  int32_t *cnt;      // [slots] entries
  int32_t *list;     // [slots][ntok] entry = t*32 + k (k == topk: shared)
  uint32_t *hmax;    // [ntok][topk+1] bits of max|h|
  float *h;          // [ntok][topk+1][I]
  unsigned *err;
};

namespace {


constexpr int kMaxTok = 16;
constexpr int kMaxTopk = 16;
constexpr int kMaxExperts = 1024;
constexpr int kRouterThreads = 128;
constexpr int kMaxConsumers = 512;

// ------------------------------------------------------------------ workspace
struct WsLayout {
  size_t logits, xstat, gshared, idx, w, meta, active, cnt, list, hmax, h, total;
};

inline size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(int ntok, int topk, int E, int I) {
  WsLayout L;
  size_t o = 0;
  const size_t slots = static_cast<size_t>(ntok) * topk + 1;
  L.logits = o; o = al256(o + 4ull * ntok * E);
  L.xstat = o; o = al256(o + 8ull * ntok);
  L.gshared = o; o = al256(o + 4ull * ntok);
  L.idx = o; o = al256(o + 4ull * ntok * topk);
  L.w = o; o = al256(o + 4ull * ntok * topk);
  L.meta = o; o = al256(o + 16);
  L.active = o; o = al256(o + 4ull * slots);
  L.cnt = o; o = al256(o + 4ull * slots);
  L.list = o; o = al256(o + 4ull * slots * ntok);
  L.hmax = o; o = al256(o + 4ull * ntok * (topk + 1));
  L.h = o; o = al256(o + 4ull * ntok * (topk + 1) * I);
  L.total = o;
  return L;
}


// ------------------------------------------------------------------ routing
// Shared-memory copy of the routing results.
struct Meta {
  int *nact, *nslots, *active, *cnt, *list, *expo, *idx;
  float *w, *gs, *rms;
  unsigned *sel, *base, *tmask;
  int slots;
  __device__ Meta(uint8_t *mem, int ntok, int topk) {
    slots = ntok * topk + 1;
    int *i = reinterpret_cast<int *>(mem);
    nact = i;
    nslots = i + 1;
    active = i + 2;
    cnt = active + slots;
    list = cnt + slots;
    w = reinterpret_cast<float *>(list + slots * ntok);
    gs = w + ntok * topk;
    expo = reinterpret_cast<int *>(gs + ntok);
    rms = reinterpret_cast<float *>(expo + ntok * (topk + 1));
    idx = reinterpret_cast<int *>(rms + ntok);
    sel = reinterpret_cast<unsigned *>(idx + ntok * topk);
    base = sel + 32;
    tmask = base + 32;
  }
  // the bit sets route_tokens() accumulates into; before a __syncthreads()
  __device__ void clear(int tid, int nthr) {
    for (int i = tid; i < 32; i += nthr) sel[i] = 0u;
    for (int i = tid; i < slots; i += nthr) tmask[i] = 0u;
  }
};

// ints/floats of Meta
__host__ __device__ inline int meta_words(int ntok, int topk) {
  const int slots = ntok * topk + 1;
  return 2 + 2 * slots + slots * ntok + ntok * topk + ntok + ntok * (topk + 1) + ntok + ntok * topk + 64 + slots;
}

// Integer key with the order of the logits: larger logit, larger key; -0
// and +0 equal.
__device__ __forceinline__ unsigned order_key(float f) {
  const unsigned b = __float_as_uint(__fadd_rn(f, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Selection scratch (32-bit words), at least kSelScratchWords: candidates
// of up to kCandMax (key, expert) pairs, per-chunk softmax statistics and
// the selected keys.
constexpr int kCandMax = 2048;
constexpr int kSelScratchWords = 2 * kCandMax + 2 * kMaxTok * (kMaxExperts / 32) + kMaxTok * kMaxTopk;

// (key, expert) packed so that a larger value comes first: larger key,
// then lower expert index.
__device__ __forceinline__ unsigned long long cand_pack(unsigned key, int e) {
  return (static_cast<unsigned long long>(key) << 32) | (0xffffffffu - static_cast<unsigned>(e));
}

// Softmax + top-K of every token, by all threads of the CTA (after a
// __syncthreads), in batches of tokens whose candidates fit kCandMax.
// Level 1: warp per (token, 32-expert chunk): the chunk's best topk entries
// in order, by rounds of warp max + ballot (equal keys: lowest lane, i.e.
// lowest expert, first), and the chunk's softmax statistics (max, sum of
// exp(l - max)).  Level 2: thread per candidate: its rank among the
// token's candidates is the count of those that come first; rank < topk
// places it.  Then warp per token: the softmax denominator from the chunk
// statistics and the selected probabilities (renormalised when norm_topk).
// Writes m.idx, m.w (and the caller's outputs when `publish`), m.sel bits.
__device__ void select_topk(const MoeArgs &a, Meta &m, uint32_t *scratch, bool publish) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarps = nthr >> 5;
  const int E = a.E, K = a.topk;
  const int nch = (E + 31) / 32;
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(scratch);  // [tb][nch][K]
  float *cmax = reinterpret_cast<float *>(scratch + 2 * kCandMax);             // [tb][nch]
  float *cden = cmax + kMaxTok * (kMaxExperts / 32);                           // [tb][nch]
  unsigned *skey = reinterpret_cast<unsigned *>(cden + kMaxTok * (kMaxExperts / 32));  // [tb][K]
  const int tb = max(1, min(a.ntok, kCandMax / (nch * K)));
#pragma unroll 1
  for (int t0 = 0; t0 < a.ntok; t0 += tb) {
    const int nt = min(tb, a.ntok - t0);
    // level 1
#pragma unroll 1
    for (int job = nwarps - 1 - warp; job < nt * nch; job += nwarps) {  // the last warps first
      const int tl = job / nch, c = job - tl * nch;
      const int e = c * 32 + lane;
      const float v = e < E ? __ldcg(a.logits + static_cast<int64_t>(t0 + tl) * E + e) : 0.0f;
      unsigned key = e < E ? max(order_key(v), 1u) : 0u;  // 0: absent or taken
      const unsigned k0 = __reduce_max_sync(0xffffffffu, key);
      const float mc = key_value(k0);
      float d = e < E ? expf(v - mc) : 0.0f;
      unsigned long long mine = 0ull;
#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        const unsigned kmax = k == 0 ? k0 : __reduce_max_sync(0xffffffffu, key);
        const int w = __ffs(__ballot_sync(0xffffffffu, key == kmax && kmax != 0u)) - 1;
        if (lane == k) mine = w >= 0 ? cand_pack(kmax, c * 32 + w) : 0ull;
        if (lane == w) key = 0u;
      }
      d = warp_sum_xor<32>(d);
      if (lane < K) cand[job * K + lane] = mine;
      if (lane == 0) {
        cmax[job] = mc;
        cden[job] = d;
      }
    }
    __syncthreads();
    // level 2
    const int C = nch * K;
#pragma unroll 1
    for (int i = tid; i < nt * C; i += nthr) {
      const int tl = i / C;
      const unsigned long long ci = cand[i];
      if (ci == 0ull) continue;
      const unsigned long long *ct = cand + tl * C;  // 16-byte aligned when C is even
      int r = 0, j = 0;
      if ((C & 1) == 0) {
        const ulonglong2 *c2 = reinterpret_cast<const ulonglong2 *>(ct);
#pragma unroll 4
        for (; j < C / 2; ++j) {
          const ulonglong2 v = c2[j];
          r += (v.x > ci ? 1 : 0) + (v.y > ci ? 1 : 0);
        }
        j = C;
      }
#pragma unroll 4
      for (; j < C; ++j) r += ct[j] > ci ? 1 : 0;
      if (r < K) {
        m.idx[(t0 + tl) * K + r] = static_cast<int>(0xffffffffu - static_cast<unsigned>(ci));
        skey[tl * K + r] = static_cast<unsigned>(ci >> 32);
      }
    }
    __syncthreads();
    // softmax: warp per token
#pragma unroll 1
    for (int tl = nwarps - 1 - warp; tl < nt; tl += nwarps) {
      const int t = t0 + tl;
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = lane; c < nch; c += 32) mx = fmaxf(mx, cmax[tl * nch + c]);
      mx = warp_max_all(mx);
      float den = 0.0f;
#pragma unroll 1
      for (int c = lane; c < nch; c += 32) den += cden[tl * nch + c] * expf(cmax[tl * nch + c] - mx);
      den = warp_sum_xor<32>(den);
      const float p = lane < K ? __fdiv_rn(expf(key_value(skey[tl * K + lane]) - mx), den) : 0.0f;
      const float sel_sum = warp_sum_xor<32>(p);
      if (lane < K) {
        const float wk = a.norm_topk ? __fdiv_rn(p, sel_sum) : p;
        const int e = m.idx[t * K + lane];
        m.w[t * K + lane] = wk;
        atomicOr(&m.sel[e >> 5], 1u << (e & 31));
        if (publish) {
          const int o = t * K + lane;
          a.idx[o] = e;
          a.w[o] = wk;
          if (a.out_idx) a.out_idx[o] = e;
          if (a.out_w) a.out_w[o] = wk;
        }
      }
    }
    if (t0 + tb < a.ntok) __syncthreads();  // the next batch reuses the scratch
  }
}

// Softmax + top-K of a single token by one warp (the calling warp; ntok ==
// 1), the same rule as select_topk -- larger logit first, equal logits to
// the lower expert, weights exp(l - max) / sum_e exp(l_e - max), renormalised
// over the chosen when norm_topk -- in one pass: lane l holds the logits of
// experts l, l + 32, ...; round r takes the warp's largest key with one
// redux.sync max and the lowest expert holding it with one redux.sync min.
// Writes m.idx, m.w (and the caller's outputs when `publish`).
template <int kPer>
__device__ void select_single_n(const MoeArgs &a, Meta &m, bool publish, int lane) {
  const int E = a.E, K = a.topk;
  unsigned key[kPer];  // 0: absent or taken
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = j * 32 + lane;
    key[j] = 0u;
    if (j * 32 < E && e < E) key[j] = max(order_key(__ldcg(a.logits + e)), 1u);
  }
  unsigned kl = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) kl = max(kl, key[j]);
  const float mx = key_value(__reduce_max_sync(0xffffffffu, kl));
  float den = 0.0f;
#pragma unroll
  for (int j = 0; j < kPer; ++j) den += key[j] != 0u ? expf(key_value(key[j]) - mx) : 0.0f;
  den = warp_sum_xor<32>(den);
  int sel_e = 0;
  unsigned sel_k = 0u;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    // the lane's largest key by a tree of adjacent pairs (log2 kPer levels
    // instead of a chain of kPer compares): slot j of level w holds the best
    // of keys [j, j + 2w), and on equal keys the left, lower expert wins
    unsigned tk[kPer];
    int tj[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      tk[j] = key[j];
      tj[j] = j;
    }
#pragma unroll
    for (int w = 1; w < kPer; w <<= 1)
#pragma unroll
      for (int j = 0; j + w < kPer; j += 2 * w) {
        const bool right = tk[j + w] > tk[j];
        tk[j] = right ? tk[j + w] : tk[j];
        tj[j] = right ? tj[j + w] : tj[j];
      }
    const unsigned lb = tk[0];
    const int lj = tj[0];
    const unsigned kmax = __reduce_max_sync(0xffffffffu, lb);
    const unsigned cand = kmax != 0u && lb == kmax ? static_cast<unsigned>(lj * 32 + lane) : 0xffffffffu;
    const unsigned emin = __reduce_min_sync(0xffffffffu, cand);
    if (lane == static_cast<int>(emin & 31u)) {
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (j == static_cast<int>(emin >> 5)) key[j] = 0u;  // constant indices keep key in registers
    }
    if (lane == r) {
      sel_e = static_cast<int>(emin);
      sel_k = kmax;
    }
  }
  const float p = lane < K ? __fdiv_rn(expf(key_value(sel_k) - mx), den) : 0.0f;
  const float sel_sum = warp_sum_xor<32>(p);
  if (lane < K) {
    const float wk = a.norm_topk ? __fdiv_rn(p, sel_sum) : p;
    m.idx[lane] = sel_e;
    m.w[lane] = wk;
    if (publish) {
      a.idx[lane] = sel_e;
      a.w[lane] = wk;
      if (a.out_idx) a.out_idx[lane] = sel_e;
      if (a.out_w) a.out_w[lane] = wk;
    }
  }
}

// The per-lane key count fixed by E (up to 64, 128 or 256 experts), so
// that every loop over a lane's keys unrolls and the keys stay in registers.
// Routers of more experts take select_topk: with 16+ keys per lane the
// single warp's serial exponentials and scans were slower than the CTA-wide
// selection (512 experts, top-4: 3.8 against 3.2 us per gate/up launch;
// 256 experts, top-8: 3.3 against 3.8 us).
constexpr int kSingleMaxExperts = 256;
__device__ void select_single(const MoeArgs &a, Meta &m, bool publish, int lane) {
  if (a.E <= 64) select_single_n<2>(a, m, publish, lane);
  else if (a.E <= 128) select_single_n<4>(a, m, publish, lane);
  else select_single_n<8>(a, m, publish, lane);
}

// What the down kernel reads of the routing, from the CTA's copy.
__device__ void publish_routing(const MoeArgs &a, const Meta &m, int tid, int nthr) {
  const int nact = *m.nact, nslots = *m.nslots;
  if (tid == 0) {
    a.meta[0] = nact;
    a.meta[1] = nslots;
  }
#pragma unroll 1
  for (int s = tid; s < nslots; s += nthr) {
    a.active[s] = s < nact ? m.active[s] : -1;
    a.cnt[s] = m.cnt[s];
  }
#pragma unroll 1
  for (int i = tid; i < nslots * a.ntok; i += nthr)
    if (i % a.ntok < m.cnt[i / a.ntok]) a.list[i] = m.list[i];
}

// Routing of all tokens inside one CTA; every thread of the CTA calls it,
// after Meta::clear() and a __syncthreads(); `scratch` holds
// kSelScratchWords.  Softmax + top-K of every token (select_topk), then
// grouping: the distinct selected experts in
// ascending order become slots 0..nact-1 and the shared expert (if any) slot
// nact; list[s*ntok + j] holds the entries t*32 + k of slot s in ascending
// token order.  `publish`: also write the routing to global memory (the
// caller's top-K outputs and what the down kernel reads).
__device__ void route_tokens(const MoeArgs &a, Meta &m, uint32_t *scratch, bool publish) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarps = nthr >> 5;
  // per-token factors: loaded before the selection, stored after it
  float tg = 1.0f, tr = 0.0f, tx = 0.0f;
  if (tid < a.ntok) {  // ntok <= 16 < threads
    if (a.gvec) tg = __ldcg(a.gshared + tid);
    tr = __ldcg(a.xstat + 2 * tid + 1);
    tx = __ldcg(a.xstat + 2 * tid);
  }
  const int rwarp = nwarps - 1 - warp;  // rwarp 0 runs token 0's softmax
  if (a.ntok == 1 && a.E <= kSingleMaxExperts) {
    if (rwarp == 0) select_single(a, m, publish, lane);  // the other warps go straight to the barrier below
  } else {
    select_topk(a, m, scratch, publish);
  }
  if (tid < a.ntok) {
    m.gs[tid] = tg;
    m.rms[tid] = tr;
    m.expo[tid] = bound_exponent(tx);
  }
  if (a.ntok == 1) {
    // one token: its topk distinct experts are the slots, in ascending
    // order (rank among the chosen), one entry each
    if (rwarp == 0) {  // m.idx / m.w of token 0 are this warp's own writes
      __syncwarp();
      const int e = lane < a.topk ? m.idx[lane] : 0x7fffffff;
      int rank = 0;
#pragma unroll 1
      for (int j = 0; j < a.topk; ++j) rank += __shfl_sync(0xffffffffu, e, j) < e ? 1 : 0;
      if (lane < a.topk) {
        m.active[rank] = e;
        m.list[rank] = lane;
        m.cnt[rank] = 1;
      }
      if (lane == 0) {
        *m.nact = a.topk;
        *m.nslots = a.topk + (a.has_shared ? 1 : 0);
        if (a.has_shared) {
          m.list[a.topk] = a.topk;
          m.cnt[a.topk] = 1;
        }
      }
    }
    __syncthreads();
    if (publish) publish_routing(a, m, tid, nthr);
    return;
  }
  __syncthreads();
  if (warp == 0) {
    // slots: exclusive scan of the per-word counts of selected experts
    const unsigned word = m.sel[lane];
    const int c = __popc(word);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    m.base[lane] = static_cast<unsigned>(incl - c);
    int pos = incl - c;
#pragma unroll 1
    for (unsigned b = word; b; b &= b - 1u) m.active[pos++] = lane * 32 + __ffs(static_cast<int>(b)) - 1;
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      *m.nact = total;
      *m.nslots = total + (a.has_shared ? 1 : 0);
      if (a.has_shared) m.tmask[total] = (1u << a.ntok) - 1u;
    }
  }
  __syncthreads();
  const int nsel = a.ntok * a.topk;
  auto slot_of = [&](int e) {
    return static_cast<int>(m.base[e >> 5]) + __popc(m.sel[e >> 5] & ((1u << (e & 31)) - 1u));
  };
#pragma unroll 1
  for (int i = tid; i < nsel; i += nthr) atomicOr(&m.tmask[slot_of(m.idx[i])], 1u << (i / a.topk));
  __syncthreads();
  const int nact = *m.nact, nslots = *m.nslots;
#pragma unroll 1
  for (int i = tid; i < nsel; i += nthr) {
    const int t = i / a.topk, k = i - t * a.topk;
    const int s = slot_of(m.idx[i]);
    m.list[s * a.ntok + __popc(m.tmask[s] & ((1u << t) - 1u))] = t * 32 + k;
  }
  if (a.has_shared)
#pragma unroll 1
    for (int t = tid; t < a.ntok; t += nthr) m.list[nact * a.ntok + t] = t * 32 + a.topk;
#pragma unroll 1
  for (int s = tid; s < nslots; s += nthr) m.cnt[s] = __popc(m.tmask[s]);
  __syncthreads();
  if (publish) publish_routing(a, m, tid, nthr);
}

// Fill the metadata copy from the routing the gate/up kernel published, with
// the h exponents from the max|h| accumulators (threads [0, nthr) of the CTA).
__device__ void load_meta(const MoeArgs &a, Meta &m, int tid, int nthr) {
  // first item of every array: all loads are issued before the first store
  // (a store waits for its load, and issue is in order)
  const int i = tid;
  const int nl = m.slots * a.ntok, nw = a.ntok * a.topk, ne = a.ntok * (a.topk + 1);
  int n0 = 0, n1 = 0, va = 0, vc = 0, vl = 0;
  float vw = 0.0f, vg = 1.0f, vr = 0.0f;
  unsigned vh = 0u;
  if (i == 0) {
    n0 = __ldcg(a.meta);
    n1 = __ldcg(a.meta + 1);
  }
  if (i < m.slots) {
    va = __ldcg(a.active + i);
    vc = __ldcg(a.cnt + i);
  }
  if (i < nl) vl = __ldcg(a.list + i);
  if (i < nw) vw = __ldcg(a.w + i);
  if (i < a.ntok) {
    if (a.gvec) vg = __ldcg(a.gshared + i);
    vr = __ldcg(a.xstat + 2 * i + 1);
  }
  if (i < ne) vh = __ldcg(a.hmax + i);
  if (i == 0) {
    *m.nact = n0;
    *m.nslots = n1;
  }
  if (i < m.slots) {
    m.active[i] = va;
    m.cnt[i] = vc;
  }
  if (i < nl) m.list[i] = vl;
  if (i < nw) m.w[i] = vw;
  if (i < a.ntok) {
    m.gs[i] = vg;
    m.rms[i] = vr;
  }
  if (i < ne) m.expo[i] = bound_exponent(__uint_as_float(vh));
  // the rest (large token counts only)
#pragma unroll 1
  for (int j = tid + nthr; j < m.slots; j += nthr) {
    m.active[j] = __ldcg(a.active + j);
    m.cnt[j] = __ldcg(a.cnt + j);
  }
#pragma unroll 4
  for (int j = tid + nthr; j < nl; j += nthr) m.list[j] = __ldcg(a.list + j);
#pragma unroll 1
  for (int j = tid + nthr; j < nw; j += nthr) m.w[j] = __ldcg(a.w + j);
#pragma unroll 1
  for (int j = tid + nthr; j < ne; j += nthr) m.expo[j] = bound_exponent(__uint_as_float(__ldcg(a.hmax + j)));
}

}  // namespace
}  // namespace epq

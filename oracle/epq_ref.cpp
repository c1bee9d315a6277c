// Plain C++ CPU oracle of the block formats and of the dequant-GEMV.
// TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
// baseline load it; the CUDA library never does, and this file includes no
// CUDA header and shares no source with it.
//
// Sources (web pages, cited by title and section):
//   "端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch" (edge-inference handbook),
//     section "GGUF 的量化格式": the four block formats -- 32-weight blocks
//     with an fp16 scale and symmetric 8-bit codes (Q8_0), 32-weight blocks
//     whose fp16 scale puts the signed largest-magnitude weight on code -8
//     (Q4_0), 32-weight blocks with an fp16 scale and an fp16 minimum and
//     codes 0..15 (Q4_1), and 256-weight superblocks of eight 32-weight
//     sub-blocks whose own scale and minimum are coded in 6 bits against
//     two fp16 superblock factors (the page's simplified Q4_K);
//     section "速度上限：带宽 ÷ 权重字节数": a decode step multiplies every
//     weight once by the activation vector(s).
//   "smolmaxxing": guided row scheduling of a multithreaded CPU matmul (each
//     grab takes remaining / (2 * threads) rows).
//
// Arithmetic: every quantizer decision is IEEE float32 with round to nearest
// even (true division, rintf, clamping in float before the integer cast),
// taken against the fp16 factors as stored.  Build without fast-math and
// with -ffp-contract=off so that no multiply-add is fused.
//
// Readings where the page is silent (the same readings as the numpy oracle):
//   * -0 inputs are mapped to +0 before anything else;
//   * a zero factor codes every weight as 0 (Q4_K: scale codes 1, min codes 0);
//   * Q4_0's largest magnitude takes the first index on ties;
//   * byte layouts are this project's own (sizes fixed by the page):
//       Q8_0  34 B: f16 d, int8 q[32]
//       Q4_0  18 B: f16 d, u8 qs[16]            (code + 8 in each nibble)
//       Q4_1  20 B: f16 d, f16 m, u8 qs[16]
//       Q4_K 144 B: f16 d, f16 dmin, u8 sc[12], u8 qs[128]
//     fp16 little-endian; weight j of a 32-run in byte j>>1, low nibble for
//     even j; Q4_K sub-block s owns qs[16s..16s+15]; its 6-bit codes c_0..c_7
//     then k_0..k_7 form a little-endian 96-bit stream (code t at bits
//     6t..6t+5).
//   * Q2_K and Q6_K (named by "smolmaxxing" and by "EPM ... 記憶體怎麼配置的",
//     which fixes Q6_K at 210 B per 256 weights) follow the same two-level
//     idea with 16-weight sub-blocks; their rows are stored plane by plane
//     (nsb superblocks per row):
//       Q2_K  codes[64 nsb] | sub-block codes c | k << 4 [16 nsb] | f16 d, dmin [nsb]
//       Q6_K  low nibbles[128 nsb] | high 2 bits[64 nsb] | int8 scales[16 nsb] | f16 d[nsb]
//     A sub-block's sixteen 2-bit fields (Q2_K codes, Q6_K high parts) share
//     one little-endian 32-bit word; position i starts at bit kField[i].
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

enum { kQ8_0 = 0, kQ4_0 = 1, kQ4_1 = 2, kQ4_K = 3, kQ2_K = 4, kQ6_K = 5 };

int block_weights(int fmt) { return fmt >= kQ4_K && fmt <= kQ6_K ? 256 : (fmt >= 0 && fmt <= 2 ? 32 : -1); }
int block_bytes(int fmt) {
  switch (fmt) {
    case kQ8_0: return 34;
    case kQ4_0: return 18;
    case kQ4_1: return 20;
    case kQ4_K: return 144;
    case kQ2_K: return 84;
    case kQ6_K: return 210;
  }
  return -1;
}
bool planar(int fmt) { return fmt == kQ2_K || fmt == kQ6_K; }

// ---------------------------------------------------------------- fp16
// IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
// Encoding from float32 by round to nearest, ties to even; values below the
// smallest subnormal half-way point become signed zero, values at or above
// 65520 become infinity, NaN stays NaN (quiet).
uint16_t f32_to_f16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const uint32_t sign = (u >> 16) & 0x8000u;
  const uint32_t ef = (u >> 23) & 0xFFu;   // float32 biased exponent
  const uint32_t mf = u & 0x7FFFFFu;       // float32 fraction
  if (ef == 0xFFu) return static_cast<uint16_t>(sign | 0x7C00u | (mf ? 0x200u | (mf >> 13) : 0u));
  // the value is (1.mf) * 2^(ef-127) (or 0.mf * 2^-126 when ef == 0)
  const int e = static_cast<int>(ef) - 127;
  if (e >= 16) return static_cast<uint16_t>(sign | 0x7C00u);  // |f| >= 65536: overflow
  if (e >= -14) {
    // normal range of fp16: keep 10 fraction bits, round the other 13 away
    uint32_t mant = mf >> 13;
    const uint32_t rest = mf & 0x1FFFu;
    uint32_t h = (static_cast<uint32_t>(e + 15) << 10) | mant;
    if (rest > 0x1000u || (rest == 0x1000u && (mant & 1u))) ++h;  // may carry into the exponent
    return static_cast<uint16_t>(sign | h);                      // 0x7C00 after a carry = inf
  }
  // subnormal fp16 (or zero): the result counts units of 2^-24
  if (ef == 0) return static_cast<uint16_t>(sign);  // float32 subnormals are far below 2^-25
  const uint32_t full = mf | 0x800000u;              // 24-bit significand, value full * 2^(e-23)
  // in units of 2^-24 the value is full * 2^(e - 23 + 24) = full >> (-e - 1)
  const int shift = -e - 1;
  if (shift > 24) return static_cast<uint16_t>(sign);  // below 2^-25 (half of the smallest subnormal)
  const uint32_t q = full >> shift;
  const uint32_t rem = full & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  uint32_t h = q;
  if (rem > half || (rem == half && (q & 1u))) ++h;  // may become the smallest normal: still right
  return static_cast<uint16_t>(sign | h);
}

// Exact float32 value of an fp16.
float f16_to_f32(uint16_t h) {
  const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
  const uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
  uint32_t u;
  if (e == 0x1Fu) {
    u = sign | 0x7F800000u | (m << 13);
  } else if (e == 0) {
    // subnormal: m * 2^-24, exact in float32
    float v = static_cast<float>(m) * 5.9604644775390625e-08f;  // 2^-24
    std::memcpy(&u, &v, 4);
    u |= sign;
  } else {
    u = sign | ((e + 112u) << 23) | (m << 13);
  }
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

void put_f16(uint8_t *p, uint16_t h) {
  p[0] = static_cast<uint8_t>(h & 0xFFu);
  p[1] = static_cast<uint8_t>(h >> 8);
}
uint16_t get_f16(const uint8_t *p) { return static_cast<uint16_t>(p[0] | (p[1] << 8)); }

// round to nearest even, clamp to [lo, hi] in float, then to an integer
int code_of(float q, float lo, float hi) {
  float r = std::rint(q);
  if (r < lo) r = lo;
  if (r > hi) r = hi;
  return static_cast<int>(r);
}

// ---------------------------------------------------------------- Q8_0
// One scale per 32 weights, chosen so that the largest magnitude maps to 127;
// codes are the nearest integers to w / scale.
void q8_0_encode(const float *w, uint8_t *out) {
  float top = 0.0f;
  for (int j = 0; j < 32; ++j) top = std::fmax(top, std::fabs(w[j]));
  const uint16_t dh = f32_to_f16(top / 127.0f);
  const float d = f16_to_f32(dh);
  put_f16(out, dh);
  for (int j = 0; j < 32; ++j) {
    const int c = d == 0.0f ? 0 : code_of(w[j] / d, -127.0f, 127.0f);
    out[2 + j] = static_cast<uint8_t>(static_cast<int8_t>(c));
  }
}

void q8_0_decode(const uint8_t *in, float *w) {
  const float d = f16_to_f32(get_f16(in));
  for (int j = 0; j < 32; ++j) w[j] = d * static_cast<float>(static_cast<int8_t>(in[2 + j]));
}

// ---------------------------------------------------------------- Q4_0
// One scale per 32 weights: the weight of largest magnitude, with its sign,
// divided by -8 (so that weight lands exactly on code -8); codes -8..7 are
// kept with an offset of 8.
void set_nibble(uint8_t *qs, int j, int n) {
  if (j & 1) qs[j >> 1] = static_cast<uint8_t>((qs[j >> 1] & 0x0Fu) | (n << 4));
  else qs[j >> 1] = static_cast<uint8_t>((qs[j >> 1] & 0xF0u) | n);
}
int get_nibble(const uint8_t *qs, int j) { return (j & 1) ? (qs[j >> 1] >> 4) : (qs[j >> 1] & 0x0F); }

void q4_0_encode(const float *w, uint8_t *out) {
  int peak = 0;
  for (int j = 1; j < 32; ++j)
    if (std::fabs(w[j]) > std::fabs(w[peak])) peak = j;  // strict: the first index wins ties
  const uint16_t dh = f32_to_f16(w[peak] / -8.0f);
  const float d = f16_to_f32(dh);
  put_f16(out, dh);
  std::memset(out + 2, 0, 16);
  for (int j = 0; j < 32; ++j) {
    const int c = d == 0.0f ? 0 : code_of(w[j] / d, -8.0f, 7.0f);
    set_nibble(out + 2, j, c + 8);
  }
}

void q4_0_decode(const uint8_t *in, float *w) {
  const float d = f16_to_f32(get_f16(in));
  for (int j = 0; j < 32; ++j) w[j] = d * static_cast<float>(get_nibble(in + 2, j) - 8);
}

// ---------------------------------------------------------------- Q4_1
// Per 32 weights an fp16 minimum m and an fp16 step d = (max - min) / 15;
// codes 0..15 are the nearest integers to (w - m) / d.
void q4_1_encode(const float *w, uint8_t *out) {
  float lo = w[0], hi = w[0];
  for (int j = 1; j < 32; ++j) {
    lo = std::fmin(lo, w[j]);
    hi = std::fmax(hi, w[j]);
  }
  const uint16_t dh = f32_to_f16((hi - lo) / 15.0f);
  const uint16_t mh = f32_to_f16(lo);
  const float d = f16_to_f32(dh), m = f16_to_f32(mh);
  put_f16(out, dh);
  put_f16(out + 2, mh);
  std::memset(out + 4, 0, 16);
  for (int j = 0; j < 32; ++j) {
    const int c = d == 0.0f ? 0 : code_of((w[j] - m) / d, 0.0f, 15.0f);
    set_nibble(out + 4, j, c);
  }
}

void q4_1_decode(const uint8_t *in, float *w) {
  const float d = f16_to_f32(get_f16(in)), m = f16_to_f32(get_f16(in + 2));
  for (int j = 0; j < 32; ++j) w[j] = static_cast<float>(get_nibble(in + 4, j)) * d + m;
}

// ---------------------------------------------------------------- Q4_K
// A superblock of 256 weights = 8 sub-blocks of 32.  Each sub-block has an
// affine code: a step (its range over 15 levels, the range measured from
// min(sub-block minimum, 0)) and an offset (minus that clamped minimum).
// The eight steps share one fp16 factor d (largest step / 63) and each is
// stored as a 6-bit multiple c of it (1..63); the eight offsets likewise
// share dmin (largest offset / 63) with 6-bit multiples k (0..63).  The
// 4-bit code of a weight is the nearest integer to (w + k*dmin) / (c*d).
void put_code6(uint8_t *sc, int t, int v) {
  for (int b = 0; b < 6; ++b) {
    const int bit = 6 * t + b;
    if ((v >> b) & 1) sc[bit >> 3] = static_cast<uint8_t>(sc[bit >> 3] | (1u << (bit & 7)));
  }
}
int get_code6(const uint8_t *sc, int t) {
  int v = 0;
  for (int b = 0; b < 6; ++b) {
    const int bit = 6 * t + b;
    v |= ((sc[bit >> 3] >> (bit & 7)) & 1) << b;
  }
  return v;
}

void q4_k_encode(const float *w, uint8_t *out) {
  float step[8], offs[8];
  float step_top = 0.0f, offs_top = 0.0f;
  for (int s = 0; s < 8; ++s) {
    const float *v = w + 32 * s;
    float lo = 0.0f, hi = v[0];  // the minimum is clamped to <= 0 from the start
    for (int j = 0; j < 32; ++j) {
      lo = std::fmin(lo, v[j]);
      hi = std::fmax(hi, v[j]);
    }
    step[s] = (hi - lo) / 15.0f;
    offs[s] = 0.0f - lo;
    step_top = std::fmax(step_top, step[s]);
    offs_top = std::fmax(offs_top, offs[s]);
  }
  const uint16_t dh = f32_to_f16(step_top / 63.0f), mh = f32_to_f16(offs_top / 63.0f);
  const float d = f16_to_f32(dh), dmin = f16_to_f32(mh);
  put_f16(out, dh);
  put_f16(out + 2, mh);
  uint8_t *sc = out + 4;
  std::memset(sc, 0, 12 + 128);
  for (int s = 0; s < 8; ++s) {
    const int c = d == 0.0f ? 1 : code_of(step[s] / d, 1.0f, 63.0f);
    const int k = dmin == 0.0f ? 0 : code_of(offs[s] / dmin, 0.0f, 63.0f);
    put_code6(sc, s, c);
    put_code6(sc, 8 + s, k);
    const float S = d * static_cast<float>(c);     // exact (11 x 6 significant bits)
    const float M = dmin * static_cast<float>(k);  // exact
    uint8_t *qs = out + 16 + 16 * s;
    for (int j = 0; j < 32; ++j) {
      const int n = S == 0.0f ? 0 : code_of((w[32 * s + j] + M) / S, 0.0f, 15.0f);
      set_nibble(qs, j, n);
    }
  }
}

void q4_k_decode(const uint8_t *in, float *w) {
  const float d = f16_to_f32(get_f16(in)), dmin = f16_to_f32(get_f16(in + 2));
  for (int s = 0; s < 8; ++s) {
    const float S = d * static_cast<float>(get_code6(in + 4, s));
    const float M = dmin * static_cast<float>(get_code6(in + 4, 8 + s));
    for (int j = 0; j < 32; ++j) w[32 * s + j] = static_cast<float>(get_nibble(in + 16 + 16 * s, j)) * S - M;
  }
}

const int kField[16] = {4, 8, 6, 10, 20, 24, 22, 26, 28, 0, 30, 2, 12, 16, 14, 18};

uint32_t get_word(const uint8_t *p) {
  return static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) | (static_cast<uint32_t>(p[2]) << 16) |
         (static_cast<uint32_t>(p[3]) << 24);
}
void put_word(uint8_t *p, uint32_t v) {
  for (int b = 0; b < 4; ++b) p[b] = static_cast<uint8_t>(v >> (8 * b));
}
int get_field(const uint8_t *words, int i) { return (get_word(words + 4 * (i >> 4)) >> kField[i & 15]) & 3; }
void or_field(uint8_t *words, int i, int v) {
  uint8_t *p = words + 4 * (i >> 4);
  put_word(p, get_word(p) | (static_cast<uint32_t>(v) << kField[i & 15]));
}

// ---------------------------------------------------------------- Q2_K
// A superblock of 256 weights = 16 sub-blocks of 16, each an affine grid of
// four levels from min(sub-block minimum, 0); the sixteen steps are 4-bit
// multiples c (1..15) of one fp16 factor d = largest step / 15, the lifts
// 4-bit multiples k (0..15) of dmin = largest lift / 15.  The superblock's
// entries go to three planes of the row: codes (64 B), sub-block codes
// (16 B), factors (4 B).
void q2_k_encode(const float *w, uint8_t *codes, uint8_t *sub, uint8_t *fac) {
  float step[16], lift[16], step_top = 0.0f, lift_top = 0.0f;
  for (int s = 0; s < 16; ++s) {
    float lo = 0.0f, hi = w[16 * s];
    for (int j = 0; j < 16; ++j) {
      lo = std::fmin(lo, w[16 * s + j]);
      hi = std::fmax(hi, w[16 * s + j]);
    }
    step[s] = (hi - lo) / 3.0f;
    lift[s] = 0.0f - lo;
    step_top = std::fmax(step_top, step[s]);
    lift_top = std::fmax(lift_top, lift[s]);
  }
  const uint16_t dh = f32_to_f16(step_top / 15.0f), mh = f32_to_f16(lift_top / 15.0f);
  const float d = f16_to_f32(dh), dmin = f16_to_f32(mh);
  put_f16(fac, dh);
  put_f16(fac + 2, mh);
  std::memset(codes, 0, 64);
  for (int s = 0; s < 16; ++s) {
    const int c = d == 0.0f ? 1 : code_of(step[s] / d, 1.0f, 15.0f);
    const int k = dmin == 0.0f ? 0 : code_of(lift[s] / dmin, 0.0f, 15.0f);
    sub[s] = static_cast<uint8_t>(c | (k << 4));
    const float S = d * static_cast<float>(c), M = dmin * static_cast<float>(k);  // exact
    for (int j = 0; j < 16; ++j) {
      const int i = 16 * s + j;
      const int n = S == 0.0f ? 0 : code_of((w[i] + M) / S, 0.0f, 3.0f);
      or_field(codes, i, n);
    }
  }
}

void q2_k_decode(const uint8_t *codes, const uint8_t *sub, const uint8_t *fac, float *w) {
  const float d = f16_to_f32(get_f16(fac)), dmin = f16_to_f32(get_f16(fac + 2));
  for (int s = 0; s < 16; ++s) {
    const float S = d * static_cast<float>(sub[s] & 15), M = dmin * static_cast<float>(sub[s] >> 4);
    for (int j = 0; j < 16; ++j) {
      const int i = 16 * s + j;
      w[i] = static_cast<float>(get_field(codes, i)) * S - M;
    }
  }
}

// ---------------------------------------------------------------- Q6_K
// A superblock of 256 weights = 16 sub-blocks of 16, symmetric: a
// sub-block's scale is its signed weight of largest magnitude (first index on
// ties) over -32, so that weight lands on code -32; the scales are int8
// multiples of one fp16 factor d = largest |scale| / 127; codes -32..31
// stored as u = code + 32 in two planes (low nibbles, high 2 bits).
void q6_k_encode(const float *w, uint8_t *ql, uint8_t *qh, uint8_t *sc, uint8_t *dp) {
  float scale[16], top = 0.0f;
  for (int s = 0; s < 16; ++s) {
    int peak = 16 * s;
    for (int j = 1; j < 16; ++j)
      if (std::fabs(w[16 * s + j]) > std::fabs(w[peak])) peak = 16 * s + j;
    scale[s] = w[peak] / -32.0f;
    top = std::fmax(top, std::fabs(scale[s]));
  }
  const uint16_t dh = f32_to_f16(top / 127.0f);
  const float d = f16_to_f32(dh);
  put_f16(dp, dh);
  std::memset(ql, 0, 128);
  std::memset(qh, 0, 64);
  for (int s = 0; s < 16; ++s) {
    const int c = d == 0.0f ? 0 : code_of(scale[s] / d, -127.0f, 127.0f);
    sc[s] = static_cast<uint8_t>(static_cast<int8_t>(c));
    const float S = d * static_cast<float>(c);  // exact
    for (int j = 0; j < 16; ++j) {
      const int i = 16 * s + j;
      const int u = (S == 0.0f ? 0 : code_of(w[i] / S, -32.0f, 31.0f)) + 32;
      set_nibble(ql, i, u & 15);
      or_field(qh, i, u >> 4);
    }
  }
}

void q6_k_decode(const uint8_t *ql, const uint8_t *qh, const uint8_t *sc, const uint8_t *dp, float *w) {
  const float d = f16_to_f32(get_f16(dp));
  for (int s = 0; s < 16; ++s) {
    const float S = d * static_cast<float>(static_cast<int8_t>(sc[s]));
    for (int j = 0; j < 16; ++j) {
      const int i = 16 * s + j;
      const int u = get_nibble(ql, i) | (get_field(qh, i) << 4);
      w[i] = static_cast<float>(u - 32) * S;
    }
  }
}

// Superblock b of a planar row (nsb superblocks): encode / decode in place.
void encode_planar(int fmt, const float *w, uint8_t *row, int64_t nsb, int64_t b) {
  if (fmt == kQ2_K)
    q2_k_encode(w, row + 64 * b, row + 64 * nsb + 16 * b, row + 80 * nsb + 4 * b);
  else
    q6_k_encode(w, row + 128 * b, row + 128 * nsb + 64 * b, row + 192 * nsb + 16 * b, row + 208 * nsb + 2 * b);
}

void decode_planar(int fmt, const uint8_t *row, int64_t nsb, int64_t b, float *w) {
  if (fmt == kQ2_K)
    q2_k_decode(row + 64 * b, row + 64 * nsb + 16 * b, row + 80 * nsb + 4 * b, w);
  else
    q6_k_decode(row + 128 * b, row + 128 * nsb + 64 * b, row + 192 * nsb + 16 * b, row + 208 * nsb + 2 * b, w);
}

void encode_block(int fmt, const float *w, uint8_t *out) {
  switch (fmt) {
    case kQ8_0: q8_0_encode(w, out); break;
    case kQ4_0: q4_0_encode(w, out); break;
    case kQ4_1: q4_1_encode(w, out); break;
    case kQ4_K: q4_k_encode(w, out); break;
  }
}

void decode_block(int fmt, const uint8_t *in, float *w) {
  switch (fmt) {
    case kQ8_0: q8_0_decode(in, w); break;
    case kQ4_0: q4_0_decode(in, w); break;
    case kQ4_1: q4_1_decode(in, w); break;
    case kQ4_K: q4_k_decode(in, w); break;
  }
}

bool shape_ok(int fmt, int64_t rows, int64_t cols) {
  const int bw = block_weights(fmt);
  return bw > 0 && rows >= 0 && cols > 0 && cols % bw == 0;
}

// Run body(r0, r1) over row ranges on `threads` threads with the guided
// split: each grab takes max(1, remaining / (2 * threads)) rows.
template <typename F>
void guided_rows(int64_t rows, int threads, F body) {
  if (threads <= 1 || rows < 2) {
    body(int64_t{0}, rows);
    return;
  }
  std::atomic<int64_t> next{0};
  auto work = [&]() {
    for (;;) {
      int64_t r0 = next.load();
      int64_t take, r1;
      do {
        if (r0 >= rows) return;
        take = (rows - r0) / (2 * threads);
        if (take < 1) take = 1;
        r1 = r0 + take;
      } while (!next.compare_exchange_weak(r0, r1));
      body(r0, r1);
    }
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < threads; ++t) pool.emplace_back(work);
  work();
  for (auto &th : pool) th.join();
}

}  // namespace

extern "C" {

uint16_t eref_f32_to_f16(float f) { return f32_to_f16(f); }
float eref_f16_to_f32(uint16_t h) { return f16_to_f32(h); }

// The fp16 encodings of the float32 values whose bit patterns are
// first, first + 1, ..., first + n - 1 (for the exhaustive check).
void eref_f16_of_bits(uint32_t first, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t u = first + static_cast<uint32_t>(i);
    float f;
    std::memcpy(&f, &u, 4);
    out[i] = f32_to_f16(f);
  }
}

int eref_block_weights(int fmt) { return block_weights(fmt); }
int eref_block_bytes(int fmt) { return block_bytes(fmt); }

// W float32 [rows][cols] -> packed [rows][cols / bw * block_bytes].  0 on success.
int eref_quantize(int fmt, const float *W, int64_t rows, int64_t cols, uint8_t *out, int threads) {
  if (!shape_ok(fmt, rows, cols)) return -1;
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  const int64_t nb = cols / bw;
  guided_rows(rows, threads, [&](int64_t r0, int64_t r1) {
    float buf[256];
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t b = 0; b < nb; ++b) {
        const float *src = W + r * cols + b * bw;
        for (int j = 0; j < bw; ++j) buf[j] = src[j] + 0.0f;  // -0 -> +0
        if (planar(fmt)) encode_planar(fmt, buf, out + r * nb * bb, nb, b);
        else encode_block(fmt, buf, out + (r * nb + b) * bb);
      }
  });
  return 0;
}

int eref_dequantize(int fmt, const uint8_t *blocks, int64_t rows, int64_t cols, float *out) {
  if (!shape_ok(fmt, rows, cols)) return -1;
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  const int64_t nb = cols / bw;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      if (planar(fmt)) decode_planar(fmt, blocks + r * nb * bb, nb, b, out + r * cols + b * bw);
      else decode_block(fmt, blocks + (r * nb + b) * bb, out + r * cols + b * bw);
    }
  return 0;
}

// y[v][i] = sum_j deq(W)[i][j] * x[v][j] in float64 (terms in column order),
// bound[v][i] = sum_j |deq(W)[i][j] * x[v][j]|.  x float32 [nvec][cols].
int eref_gemv_f64(int fmt, const uint8_t *blocks, const float *x, int64_t rows, int64_t cols, int nvec, double *y,
                  double *bound, int threads) {
  if (!shape_ok(fmt, rows, cols) || nvec < 1) return -1;
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  const int64_t nb = cols / bw;
  guided_rows(rows, threads, [&](int64_t r0, int64_t r1) {
    float w[256];
    for (int64_t r = r0; r < r1; ++r)
      for (int v = 0; v < nvec; ++v) {
        double acc = 0.0, mag = 0.0;
        const float *xv = x + v * cols;
        for (int64_t b = 0; b < nb; ++b) {
          if (planar(fmt)) decode_planar(fmt, blocks + r * nb * bb, nb, b, w);
          else decode_block(fmt, blocks + (r * nb + b) * bb, w);
          for (int j = 0; j < bw; ++j) {
            const double t = static_cast<double>(w[j]) * static_cast<double>(xv[b * bw + j]);
            acc += t;
            mag += std::fabs(t);
          }
        }
        y[v * rows + r] = acc;
        if (bound) bound[v * rows + r] = mag;
      }
  });
  return 0;
}

// The CPU baseline: y[v][i] = sum_j deq(W)[i][j] * x[v][j] in float32, each
// block dequantized into a small buffer and multiplied in place (eight
// running partial sums per row, added in a fixed order).  Rows are spread
// over `threads` threads by the guided split.
int eref_gemv_f32(int fmt, const uint8_t *blocks, const float *x, int64_t rows, int64_t cols, int nvec, float *y,
                  int threads) {
  if (!shape_ok(fmt, rows, cols) || nvec < 1 || nvec > 8) return -1;
  const int bw = block_weights(fmt), bb = block_bytes(fmt);
  const int64_t nb = cols / bw;
  guided_rows(rows, threads, [&](int64_t r0, int64_t r1) {
    float w[256];
    for (int64_t r = r0; r < r1; ++r) {
      float part[8][8] = {};
      for (int64_t b = 0; b < nb; ++b) {
        if (planar(fmt)) decode_planar(fmt, blocks + r * nb * bb, nb, b, w);
        else decode_block(fmt, blocks + (r * nb + b) * bb, w);
        for (int v = 0; v < nvec; ++v) {
          const float *xv = x + v * cols + b * bw;
          for (int j = 0; j < bw; j += 8)
            for (int l = 0; l < 8; ++l) part[v][l] += w[j + l] * xv[j + l];
        }
      }
      for (int v = 0; v < nvec; ++v)
        y[v * rows + r] = ((part[v][0] + part[v][1]) + (part[v][2] + part[v][3])) +
                          ((part[v][4] + part[v][5]) + (part[v][6] + part[v][7]));
    }
  });
  return 0;
}

int eref_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? static_cast<int>(n) : 1;
}

}  // extern "C"

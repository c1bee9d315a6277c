/*
 * epq.h -- C ABI of the block-quantized decode library (GB300, sm_103a).
 *
 * The library computes the batch-1 decode hot path over block-quantized
 * weights: packing float32 weights into the Q8_0 / Q4_0 / Q4_1 / Q4_K block
 * formats, the fused dequantize-and-matrix-vector product y = deq(W) x (one to
 * eight activation vectors), and the mixture-of-experts layer built on it
 * (router softmax + top-K, gate/up with SwiGLU, down, weighted combine plus
 * residual).
 *
 * Sources, cited by page title and section:
 *   [H]  "端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch" (edge-inference handbook),
 *        sections "速度上限：带宽 ÷ 权重字节数" and "GGUF 的量化格式".
 *   [F]  "Flash-MoE：在笔记本上运行 397B 参数大模型", sections
 *        "核心技术 / 3. Metal 计算着色器" and "每层流水线".
 *   [E]  "EPM：MiniCPM-V-4.7-35B-A3B 的 8 GiB 專家分頁 CPU 推論", sections
 *        "記憶體怎麼配置的" and "正確性".
 *
 * Conventions for every call:
 *   - Pointers named W, x, y, blocks, ... are DEVICE pointers on the current
 *     CUDA device unless a parameter says otherwise.  The caller owns all
 *     memory; no call allocates device memory.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     and return after the launches are queued.
 *   - Every call returns an epq_status and never aborts.  Argument errors are
 *     detected on the host before anything is launched.  EPQ_ERR_CUDA reports
 *     a CUDA runtime error of a launch (its code: epq_last_cuda_error()).
 *   - Kernels never wait without bound.  A pipeline wait that exceeds its
 *     time limit makes the kernel record an error and return;
 *     epq_device_error() reads and clears that record.
 *   - Results are bitwise reproducible run to run (no floating-point atomics).
 */
#ifndef EPQ_H
#define EPQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *epq_stream_t; /* same type as cudaStream_t */

typedef enum {
  EPQ_OK = 0,
  EPQ_ERR_ARG = 1,       /* null pointer or value out of range */
  EPQ_ERR_FORMAT = 2,    /* unknown block format */
  EPQ_ERR_SHAPE = 3,     /* a dimension the kernels do not support */
  EPQ_ERR_ALIGN = 4,     /* pointer not 16-byte aligned */
  EPQ_ERR_WORKSPACE = 5, /* workspace missing or too small */
  EPQ_ERR_CUDA = 6,      /* CUDA runtime error; see epq_last_cuda_error() */
  EPQ_ERR_DEVICE = 7     /* no usable device of compute capability 10.3 */
} epq_status;

/* Block formats of [H] "GGUF 的量化格式".  Packed byte layouts (the page fixes
 * the sizes; the byte order is this library's own definition):
 *   EPQ_Q8_0  32 weights,  34 B: f16 d | int8 q[32]             w = d*q
 *   EPQ_Q4_0  32 weights,  18 B: f16 d | u8 qs[16]              w = d*(n-8)
 *   EPQ_Q4_1  32 weights,  20 B: f16 d | f16 m | u8 qs[16]      w = d*n + m
 *   EPQ_Q4_K 256 weights, 144 B: f16 d | f16 dmin | u8 sc[12] | u8 qs[128]
 *             sub-block s (weights 32s..32s+31): w = d*c_s*n - dmin*k_s
 * fp16 little-endian; weight j of a 32-run lives in byte j>>1 (low nibble for
 * even j); Q4_K sub-block s owns qs[16s..16s+15]; its 6-bit codes c_0..c_7,
 * k_0..k_7 form a little-endian 96-bit stream, code t at bits 6t..6t+5.  A
 * row is a contiguous run of blocks in column order; rows are contiguous.
 *
 * Two K-quants with 16-weight sub-blocks, sized by "EPM ... 記憶體怎麼配置的"
 * (Q6_K: 210 B per 256 weights) and the 2-bit experts of "smolmaxxing":
 *   EPQ_Q2_K 256 weights,  84 B: sub-block s (weights 16s..16s+15) has
 *             step code c_s (1..15) and lift code k_s (0..15) against fp16
 *             d and dmin; codes n 0..3:  w = d*c_s*n - dmin*k_s
 *   EPQ_Q6_K 256 weights, 210 B: int8 scale code c_s against fp16 d; codes
 *             m -32..31:  w = d*c_s*m   (exact in float32)
 * Their rows are stored plane by plane (nsb = cols/256 superblocks):
 *   Q2_K  u8 codes[64 nsb] | u8 (c | k<<4)[16 nsb] | f16 (d, dmin)[nsb]
 *   Q6_K  u8 low nibbles[128 nsb] | u8 high parts[64 nsb] | int8 c[16 nsb]
 *         | f16 d[nsb]
 * with u = m + 32 for Q6_K: u & 15 of superblock weight j in byte j>>1 of
 * the superblock's 128 (low nibble when j is even); the 2-bit fields (Q2_K
 * codes n, Q6_K high parts u >> 4) of sub-block s fill its little-endian
 * 32-bit word s, position i at bit FIELD[i], FIELD = {4, 8, 6, 10, 20, 24,
 * 22, 26, 28, 0, 30, 2, 12, 16, 14, 18}. */
typedef enum { EPQ_Q8_0 = 0, EPQ_Q4_0 = 1, EPQ_Q4_1 = 2, EPQ_Q4_K = 3, EPQ_Q2_K = 4, EPQ_Q6_K = 5 } epq_fmt;

const char *epq_status_string(epq_status s);

/* cudaError_t of the most recent EPQ_ERR_CUDA returned on this host thread. */
int epq_last_cuda_error(void);

/* Reads and clears the device-side error record of the current device:
 * 0 = none; otherwise a code naming the pipeline wait that timed out.
 * Synchronizes the device. */
int epq_device_error(void);

/* Same, and where the first timeout happened: the CTA index, the pipeline
 * step (tile or work-unit index) and the thread index (any pointer may be
 * NULL). */
int epq_device_error_detail(int *block, int *where, int *thread);

/* Weights per block (32 or 256), bytes per block, and packed bytes per row:
 * cols/block_weights*block_bytes, or -1 when cols is not a positive multiple
 * of the block size or fmt is unknown.  Host-only, no device needed. */
int64_t epq_block_weights(epq_fmt fmt);
int64_t epq_block_bytes(epq_fmt fmt);
int64_t epq_row_bytes(epq_fmt fmt, int64_t cols);

/* Tuning hooks (host-only, process-wide; the defaults suit GB300).
 *   EPQ_TUNE_TILE_BYTES  target packed bytes per pipeline stage of the GEMV
 *                        engines (4096 .. 131072)
 *   EPQ_TUNE_RING_BYTES  shared-memory ring budget per CTA (32768 .. 200704)
 *   EPQ_TUNE_GEMV_ENGINE engine of the Q4_K GEMVs and MoE experts:
 *                        0 automatic (the block-diagonal tensor-core engine
 *                        of the Q2_K / Q6_K GEMV for one vector; for two or
 *                        more the vector-column engine from 5 vectors, else
 *                        the ring tensor-core engine; the ring engine for
 *                        the MoE expert stages), 1 CUDA-core engines only
 *                        (also for the MoE experts), 2 the ring tensor-core
 *                        engine wherever it applies (one vector under 2 MiB:
 *                        CUDA cores), 3 the block-diagonal engine for every
 *                        Q4_K GEMV (the MoE experts as in 0), 4 the
 *                        vector-column engine for two or more Q4_K vectors
 *                        (one weight pass for up to 8; MoE as in 0)
 *   EPQ_TUNE_EARLY_STAGES pipeline stages the tensor-core GEMV issues before
 *                        its grid-dependency wait when weights_ready is set
 *                        (0 .. 16, default 4)
 *   EPQ_TUNE_TC_SPLIT    warps that share one 8-row block of the tensor-core
 *                        GEMV (1, 2, 4, 8 or 16; 0 = chosen by shape, the
 *                        default: 8 for rows of 8..32 superblocks)
 *   EPQ_TUNE_ATTN_CHUNK  most cached key (value) rows epq_attention_decode
 *                        copies into shared memory at a time: 0 = as many
 *                        as fit (the default), else 8 .. 4096, a multiple
 *                        of 8 (smaller chunks: more copy round trips, the
 *                        same result)
 *   EPQ_TUNE_VN_CHUNK    most superblocks of x operands the vector-column
 *                        engine holds at a time: 0 = as many as fit (the
 *                        default), else 1 .. 64 (longer rows run in chunks
 *                        with partial sums in shared memory)
 *   EPQ_TUNE_VN_CLUSTER  CTAs per thread-block cluster of the vector-column
 *                        engine, which share the conversion of x: 0 =
 *                        automatic (the default), 1, 2 or 4
 * Returns the previous value, or -1 for an unknown key or a value out of
 * range (nothing changes then).  Affects launches issued afterwards. */
enum { EPQ_TUNE_TILE_BYTES = 1, EPQ_TUNE_RING_BYTES = 2, EPQ_TUNE_GEMV_ENGINE = 3, EPQ_TUNE_EARLY_STAGES = 4,
       EPQ_TUNE_TC_SPLIT = 5, EPQ_TUNE_ATTN_CHUNK = 6, EPQ_TUNE_VN_CHUNK = 7,
       EPQ_TUNE_VN_CLUSTER = 8 };
int epq_set_tuning(int key, int value);

/* ---------------------------------------------------------------- packing
 * epq_quantize: [H] "GGUF 的量化格式" (the four quantizers).
 *   W       float32 [rows][cols], row-major, finite values.
 *   blocks  output, rows*epq_row_bytes(fmt, cols) bytes.
 * Decisions follow the page in IEEE float32 (true division, round half to
 * even) against the stored fp16 factors; a zero factor gives zero codes
 * (Q4_K: scale codes 1, min codes 0); Q4_0 takes the first index of the
 * largest magnitude; -0 inputs are treated as +0.  The output is bit-exact
 * with the CPU oracle.  Requirements: cols % 256 == 0 (EPQ_ERR_SHAPE),
 * rows >= 1, W and blocks 16-byte aligned (EPQ_ERR_ALIGN). */
epq_status epq_quantize(epq_fmt fmt, const float *W, int64_t rows, int64_t cols,
                        void *blocks, epq_stream_t stream);

/* epq_dequantize: the inverse map of [H] "GGUF 的量化格式" (each weight is
 * formed with a single rounding), W_out float32 [rows][cols].  Same shape and
 * alignment rules as epq_quantize.  Bit-exact with the CPU oracle. */
epq_status epq_dequantize(epq_fmt fmt, const void *blocks, int64_t rows, int64_t cols,
                          float *W_out, epq_stream_t stream);

/* ---------------------------------------------------------------- GEMV
 * epq_gemv: [H] "速度上限：带宽 ÷ 权重字节数" -- batch-1 decode streams every
 * weight once per token; nvec > 1 multiplies the same weight pass by up to 8
 * speculative-verify vectors.
 *   x  float32 [nvec][cols]   y  float32 [nvec][rows]   (contiguous)
 *   y[v][i] = sum_j deq(W)[i][j] * x[v][j], accumulated in float32.
 * Accuracy: |y - y_ref| <= 1e-4 * sum_j |deq(W)[i][j] x[v][j]| (float64 ref).
 * The entries of x must be finite with max|x| < 2^100; entries more than
 * about 2^100 below max|x| count as zero.  Q4_K through the tensor-core
 * engine (see EPQ_TUNE_GEMV_ENGINE): x is split into fp16 hi + lo parts
 * scaled per 256-column block, so entries more than about 2^38 below the
 * largest |x| of their 256-column block keep less precision (their fp16
 * parts become subnormal); the bound can fail only for inputs whose tiny
 * entries carry the result.
 * Requirements: 1 <= nvec <= 8, rows >= 1, cols % 256 == 0 and
 * 256 <= cols <= 16384 (EPQ_ERR_SHAPE), blocks/x/y 16-byte aligned.
 * y must not overlap x or blocks. */
epq_status epq_gemv(epq_fmt fmt, const void *blocks, const float *x, float *y,
                    int64_t rows, int64_t cols, int nvec, epq_stream_t stream);

/* Options of epq_gemv_ex (all-zero = plain epq_gemv).
 *   residual     NULL or float32 [nvec][rows_out]: y = residual + result.
 *                May equal y (in-place residual update).
 *   rms_prenorm  1: each x vector is replaced by x / sqrt(mean(x^2) + rms_eps)
 *                before the product (a weightless RMS norm, [F] "3. Metal 计算
 *                着色器"); the norm is folded into the output scale.
 *   swiglu       1: the matrix holds 2*I rows, the I gate rows then the I up
 *                rows; the output has rows_out = I = rows/2 rows:
 *                y[v][i] = silu(g_i) * u_i, silu(g) = g / (1 + exp(-g))
 *                ([F] "3. Metal 计算着色器", fused SwiGLU).  rows must be even.
 *   x_group, x_head_dim   when x_group > 1: column j of the product reads
 *                x[(j / (x_head_dim*x_group)) * x_head_dim + j % x_head_dim]
 *                (each head of x repeated x_group times, as a grouped-query
 *                attention output over a one-token context).  x then holds
 *                cols / x_group floats per vector; x_head_dim % 32 == 0.
 *   x_ld         floats between consecutive x vectors (0 = the vector length);
 *                a multiple of 4, so that a slice of a wider buffer can be
 *                read in place.
 *   weights_ready  1: the packed weights were not written by work that may
 *                still be running on the stream, so the kernel may start
 *                streaming them into shared memory before the preceding
 *                kernel has finished (programmatic dependent launch).  x and
 *                residual are always read only after it has finished. */
typedef struct {
  const float *residual;
  int rms_prenorm;
  float rms_eps;
  int swiglu;
  int x_group;
  int x_head_dim;
  int64_t x_ld;
  int weights_ready;
} epq_gemv_opts;

epq_status epq_gemv_ex(epq_fmt fmt, const void *blocks, const float *x, float *y,
                       int64_t rows, int64_t cols, int nvec, const epq_gemv_opts *opts,
                       epq_stream_t stream);

/* ---------------------------------------------------------------- GEMV chain
 * epq_gemv_chain: a sequence of dependent dequant-GEMVs in one persistent
 * launch -- the decode step of a dense decoder ([H] "速度上限：带宽 ÷
 * 权重字节数": a step streams every weight once, so the bound is bandwidth /
 * weight bytes).  Op k computes exactly what epq_gemv_ex computes with the
 * same fields (y = [residual +] W x with the RMS pre-norm, SwiGLU and
 * grouped-head options), and it sees every output of ops 0..k-1: x,
 * residual and y of op k may be outputs of earlier ops.  The weights of
 * later ops are streamed while earlier ops finish; between ops a grid-wide
 * barrier makes the outputs visible.
 *   fmt      EPQ_Q4_K only (EPQ_ERR_FORMAT otherwise).
 *   ops      host array of nops (1 .. EPQ_CHAIN_MAX_OPS) descriptors; read
 *            during the call only (it may be reused afterwards, also under
 *            stream capture).  Per op: rows, cols as in epq_gemv (cols % 256
 *            == 0, 256 <= cols <= 16384), blocks/x/y/residual device
 *            pointers, 16-byte aligned; x_ld floats between the two vectors
 *            of x (0 = the vector length).
 *   nvec     1 or 2 (vectors per op; y and residual are [nvec][rows_out]).
 *   ws, ws_bytes  device workspace of >= epq_gemv_chain_workspace_bytes()
 *            bytes, 16-byte aligned, zero-filled before its first use and
 *            not shared by chains that may run at the same time.  A call
 *            leaves it ready for the next call; after a device-side wait
 *            timeout (epq_device_error) zero it again.
 * Accuracy per op as epq_gemv.  Deterministic.  The launch is cooperative
 * (one CTA per SM, all resident): EPQ_ERR_CUDA if the device cannot host it. */
#define EPQ_CHAIN_MAX_OPS 256
typedef struct {
  const void *blocks;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows;
  int64_t cols;
  int swiglu;
  int rms_prenorm;
  float rms_eps;
  int x_group;
  int x_head_dim;
  int64_t x_ld;
} epq_gemv_op;

size_t epq_gemv_chain_workspace_bytes(void);
epq_status epq_gemv_chain(epq_fmt fmt, const epq_gemv_op *ops, int nops, int nvec, void *ws,
                          size_t ws_bytes, epq_stream_t stream);

/* ---------------------------------------------------------------- MoE layer
 * [F] "每层流水线" and "3. Metal 计算着色器"; shapes from [F] "模型架构" and
 * [E] "記憶體怎麼配置的".  For every token t (x_t = row t of x):
 *   xin_t  = x_t, or x_t / sqrt(mean(x_t^2) + rms_eps) with rms_prenorm
 *   l_t    = R xin_t + bias                       (router logits, float32)
 *   S_t    = the topk experts of largest l_t (ties -> lower expert index)
 *   p_t    = softmax(l_t) over all experts; w_tk = p_t[e_k], divided by
 *            sum_k p_t[e_k] when norm_topk
 *   E_e(v) = down_e( silu(gate_e v) * (up_e v) )  (silu(g) = g/(1+exp(-g)))
 *   y_t    = x_t + sum_k w_tk E_{e_k}(xin_t) + g_t E_shared(xin_t)
 *            g_t = 1, or sigmoid(shared_gate_vec . xin_t) when given.
 * Tokens that pick the same expert share one pass over its weights, except
 * that a Q4_K call of three or more tokens running all stages is processed
 * as chunks of two tokens on the tensor-core kernels (an expert chosen in
 * two chunks is read once per chunk); EPQ_TUNE_GEMV_ENGINE = 1 keeps one
 * pass for all tokens on the CUDA-core kernels. */
typedef struct {
  const float *weight; /* [n_experts][hidden] float32, 16-byte aligned */
  const float *bias;   /* [n_experts] or NULL */
  int n_experts;       /* 1..1024 */
  int norm_topk;       /* 1: renormalize the selected probabilities */
} epq_router;

typedef struct {
  epq_fmt fmt;
  int n_experts; /* must equal the router's */
  int hidden;    /* H: multiple of 256, 256..16384 */
  int inter;     /* I: multiple of 256, 256..16384 */
  /* expert e: gate_up + e*gate_up_stride holds 2*I packed rows of H weights
   * (the I gate rows, then the I up rows); down + e*down_stride holds H
   * packed rows of I weights.  A stride of 0 means the packed size.  Strides
   * must be multiples of 16 bytes. */
  const void *gate_up;
  int64_t gate_up_stride;
  const void *down;
  int64_t down_stride;
  const void *shared_gate_up;    /* NULL: no shared expert */
  const void *shared_down;
  const float *shared_gate_vec;  /* NULL: shared weight 1; else [H] */
  /* Mixed per-tensor recipe ("EPM ... 記憶體怎麼配置的": Q4_K gate/up with
   * Q6_K down): when down_fmt_set is 1 the down projections (routed and
   * shared) are stored in down_fmt and the gate/up matrices in fmt; when 0
   * (zero-initialised struct) both use fmt. */
  int down_fmt_set;
  epq_fmt down_fmt;
} epq_experts;

typedef struct {
  int rms_prenorm;
  float rms_eps;
  float *logits_out; /* NULL or [ntok][n_experts]: the router logits */
  float *h_out;      /* NULL or [ntok][topk+1][I]: silu(g)*u per token and
                        slot (slot k = k-th choice, slot topk = shared) */
  int stages;        /* 0 = all; else a mask of EPQ_MOE_ROUTE, EPQ_MOE_GATE_UP,
                        EPQ_MOE_DOWN: the selected kernels only.  Stages of
                        one layer may be issued by separate calls in order
                        with the same arguments and workspace (the workspace
                        carries the logits, routing and h between them).
                        Separate stage calls are never split into chunks of
                        two tokens, so for a Q4_K call of more than two
                        tokens they run the CUDA-core kernels (same result
                        within the GEMV bound, not bit for bit).
                        The gate/up stage computes the routing; a call with
                        the router stage but not the gate/up stage adds a
                        one-CTA routing kernel when it returns topk_idx /
                        topk_w or runs the down stage. */
} epq_moe_opts;

enum { EPQ_MOE_ROUTE = 1, EPQ_MOE_GATE_UP = 2, EPQ_MOE_DOWN = 4 };

/* Workspace bytes epq_moe_forward needs for these shapes (0 on bad input).
 * Host-only. */
size_t epq_moe_workspace_bytes(const epq_router *router, const epq_experts *experts, int ntok, int topk);

/* One MoE layer for ntok tokens (1..16) and topk (1..16, <= n_experts).
 *   x          float32 [ntok][H]            y  float32 [ntok][H] (may equal x)
 *   topk_idx   NULL or int32 [ntok][topk]   (selected experts, best first)
 *   topk_w     NULL or float32 [ntok][topk] (their combine weights)
 *   workspace  device scratch of epq_moe_workspace_bytes(); no
 *              initialisation is needed and nothing carries over between
 *              calls, except between the stages of one layer (see stages).
 *              Calls that share a workspace must be ordered on one stream.
 * Three kernels are queued: router logits; routing (softmax, top-K,
 * grouping) + gate/up + SwiGLU; down + combine + residual.  No host
 * synchronisation.  Logits must be finite (a NaN logit ranks above all
 * others; the selection is then unspecified by the method). */
epq_status epq_moe_forward(const epq_router *router, const epq_experts *experts, const float *x, int ntok,
                           int topk, const epq_moe_opts *opts, float *y, int32_t *topk_idx, float *topk_w,
                           void *workspace, size_t workspace_bytes, epq_stream_t stream);

/* epq_moe_forward_noalloc: the same MoE layer, for callers that cannot
 * allocate device memory -- for instance a runtime that plans all of its
 * device memory up front and hands out no scratch, or code that must not
 * call the CUDA allocator from its decode loop.  (The source pages have no
 * counterpart; this is an interface convenience.)
 *
 * Instead of a caller workspace it uses one fixed 1 MiB array compiled into
 * the library (a file-scope __device__ array; every GPU that loads the
 * library holds it until the process exits).  Inputs and outputs are still
 * passed by the caller, exactly as for epq_moe_forward.
 *   - Shapes whose workspace (epq_moe_workspace_bytes) exceeds 1 MiB are
 *     rejected with EPQ_ERR_WORKSPACE before anything is queued.
 *   - No cudaMalloc / cudaFree or other allocating call is made.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - All calls on a device share the array.  Calls that may overlap on
 *     the GPU (different streams without ordering) race on the array and
 *     must not be issued. */
epq_status epq_moe_forward_noalloc(const epq_router *router, const epq_experts *experts, const float *x,
                                   int ntok, int topk, const epq_moe_opts *opts, float *y, int32_t *topk_idx,
                                   float *topk_w, epq_stream_t stream);

/* ---------------------------------------------------------------- attention
 * epq_attention_decode: one decode step of attention over a Q8_0 key/value
 * cache with a skip threshold ("smolmaxxing", compute table, row
 * "带阈值的 Q8_0 注意力": all key dot products first, so the softmax maximum M
 * is known; positions with score < M + skip_log skip the exponential and the
 * value read).  Batch 1; query head hq reads key/value head hq / group with
 * group = n_heads / n_kv_heads (1, 2, 4 or 8).
 *   q             float32 [n_heads][head_dim]
 *   k_new, v_new  float32 [n_kv_heads][head_dim]: the step's key and value;
 *                 they are quantized to Q8_0 (32-element blocks, the
 *                 packer's arithmetic) and stored at position `pos` first.
 *   k_cache, v_cache  [n_kv_heads][max_pos][epq_kv_row_bytes(head_dim)]:
 *                 row (h, p) holds the head_dim/32 fp16 block factors, then
 *                 the head_dim int8 codes (element = factor * code).  Rows
 *                 0..pos-1 must hold earlier positions; row pos is written.
 *   scores s_p = scale * sum_e q[e] * k_p[e] (k dequantized, float32 sums);
 *   M = max_p s_p; kept positions: s_p >= M + skip_log (skip_log = -inf
 *   keeps all); out[hq] = sum_kept exp(s_p - M) v_p / sum_kept exp(s_p - M).
 *   out           float32 [n_heads][head_dim]
 *   scores_out    NULL or float32 [n_heads][max_pos]: the scores of
 *                 positions 0..pos (for checking).
 * Requirements: head_dim 128 or 256, 0 <= pos < max_pos, pos < 16384,
 * scale > 0, 16-byte aligned pointers.  Deterministic (fixed summation
 * order).  One launch: a cluster of up to 8 CTAs per key/value head. */
int64_t epq_kv_row_bytes(int head_dim);
epq_status epq_attention_decode(const float *q, const float *k_new, const float *v_new, void *k_cache,
                                void *v_cache, int n_heads, int n_kv_heads, int head_dim, int pos, int max_pos,
                                float scale, float skip_log, float *out, float *scores_out, epq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EPQ_H */

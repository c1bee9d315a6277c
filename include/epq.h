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
 * row is a contiguous run of blocks in column order; rows are contiguous. */
typedef enum { EPQ_Q8_0 = 0, EPQ_Q4_0 = 1, EPQ_Q4_1 = 2, EPQ_Q4_K = 3 } epq_fmt;

const char *epq_status_string(epq_status s);

/* cudaError_t of the most recent EPQ_ERR_CUDA returned on this host thread. */
int epq_last_cuda_error(void);

/* Reads and clears the device-side error record of the current device:
 * 0 = none; otherwise a code naming the pipeline wait that timed out.
 * Synchronizes the device. */
int epq_device_error(void);

/* Weights per block (32 or 256), bytes per block, and packed bytes per row:
 * cols/block_weights*block_bytes, or -1 when cols is not a positive multiple
 * of the block size or fmt is unknown.  Host-only, no device needed. */
int64_t epq_block_weights(epq_fmt fmt);
int64_t epq_block_bytes(epq_fmt fmt);
int64_t epq_row_bytes(epq_fmt fmt, int64_t cols);

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
 * about 2^100 below max|x| count as zero.
 * Requirements: 1 <= nvec <= 8, rows >= 1, cols % 256 == 0 and
 * 256 <= cols <= 32768 (EPQ_ERR_SHAPE), blocks/x/y 16-byte aligned.
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
 *                cols / x_group floats per vector; x_head_dim % 32 == 0. */
typedef struct {
  const float *residual;
  int rms_prenorm;
  float rms_eps;
  int swiglu;
  int x_group;
  int x_head_dim;
} epq_gemv_opts;

epq_status epq_gemv_ex(epq_fmt fmt, const void *blocks, const float *x, float *y,
                       int64_t rows, int64_t cols, int nvec, const epq_gemv_opts *opts,
                       epq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EPQ_H */

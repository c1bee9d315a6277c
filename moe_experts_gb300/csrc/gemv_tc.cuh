// Host interface of the tensor-core Q4_K dequant-GEMV (gemv_tc.cu).
#pragma once

#include "common.cuh"

namespace epq {

// Launch geometry chosen on the host for one matrix shape.
struct TcPlan {
  int nsb_tmpl;          // superblocks per warp (template value 1, 2 or 4)
  bool full;             // every warp has all NSB superblocks (no bounds test)
  int kp, nb, nbs, stages;
  uint32_t stage_bytes, smem;
  unsigned grid;
};

// Arguments of one launch (one or two vectors).
struct TcArgs {
  const uint8_t *W;
  const float *x;
  float *y;
  const float *residual;
  int64_t rows_out, row_bytes;
  int cols, nv;
  int64_t x_stride, y_stride;
  int swiglu, rms;
  float rms_eps;
  int x_group, x_head_dim;
  int early_weights;
  unsigned *err;
};

// False when the shape is outside the kernel's range (cols % 256, 256..16384)
// or the shared-memory budget cannot hold two stages.
bool gemv_tc_plan(int64_t row_bytes, int cols, int64_t rows_out, bool swiglu, const DeviceInfo &dev,
                  TcPlan *pl);

cudaError_t gemv_tc_launch(const TcPlan &pl, const TcArgs &a, cudaStream_t s);

// 3..8 vectors in one weight pass (rows of 4096 weights); false when the
// shape is not covered (the caller then runs one pass per vector pair).
bool gemv_tc_multi_launch(const TcArgs &a, int nvec, const DeviceInfo &dev, cudaStream_t s, cudaError_t *err);

// Q4_K with 2..8 vectors in one weight pass, the vectors in the MMA's n
// dimension (gemv_vn.cu): the whole epq_gemv_ex call after the common checks.
epq_status gemv_vn_launch(const void *blocks, const float *x, float *y, int64_t rows, int64_t cols, int nvec,
                          const epq_gemv_opts &o, int64_t x_stride, const DeviceInfo &dev, cudaStream_t s);

// Q2_K / Q6_K (gemv_k16.cu): the whole epq_gemv_ex call after the common
// argument checks (x_stride = floats between x vectors).
epq_status gemv_k16_launch(epq_fmt fmt, const void *blocks, const float *x, float *y, int64_t rows, int64_t cols,
                           int nvec, const epq_gemv_opts &o, int64_t x_stride, const DeviceInfo &dev,
                           cudaStream_t s);

}  // namespace epq

// Tensor-core Q4_K expert kernels of the MoE layer for one or two tokens per
// call (moe_tc.cu).  epq_moe_forward uses them when moe_tc_plan accepts the
// call's shapes; everything else keeps the CUDA-core kernels of moe.cu.
#pragma once

#include "moe_common.cuh"

namespace epq {

struct MoeTcPlan {
  unsigned grid;
  // gate/up + SwiGLU: KP k-parts of NSB superblocks each, FULL when they
  // cover the H/256 superblocks exactly; ring of `stages` stages of 8 gate
  // rows + 8 up rows
  int g_kp, g_nsbw, g_full, g_stages, g_sep;
  uint32_t g_stage_bytes, g_smem;
  // down + combine: the x operand spans up to d_nsbx superblocks (every
  // slot's I/256); a stage holds 8 rows of every slot's down matrix
  int d_kp, d_nsbw, d_stages, d_nsbx, d_sep;
  uint32_t d_stage_bytes, d_smem;
};

// Plans both kernels for the call described by `a` (Q4_K experts, 1 or 2
// tokens, H and I multiples of 256) with at most `max_slots` slots (distinct
// routed experts plus the shared expert).  False when the shapes do not fit.
bool moe_tc_plan(const MoeArgs &a, int max_slots, const DeviceInfo &dev, MoeTcPlan *pl);

// gate/up: routes in every CTA (publishing from CTA 0), writes h.
cudaError_t moe_tc_gateup_launch(const MoeTcPlan &pl, const MoeArgs &a, cudaStream_t s);
// down + weighted combine + residual: reads the published routing and h, writes y.
cudaError_t moe_tc_down_launch(const MoeTcPlan &pl, const MoeArgs &a, cudaStream_t s);

}  // namespace epq

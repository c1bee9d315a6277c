// Q2_K / Q6_K expert kernels of the MoE layer, one or two tokens per call
// (moe_k16.cu).  epq_moe_forward runs them for a stage whose matrices are
// stored in one of these formats; the other stage may use any engine (the
// kernels follow the shared workspace protocol: routing published by the
// gate/up kernel's CTA 0, h and the max |h| words in the workspace).
#pragma once

#include "moe_common.cuh"

namespace epq {

// Whether the kernels' shared memory holds the call's operands (H/256
// superblocks of x per token for gate/up, max_slots * I/256 for down).
bool moe_k16_fits(const MoeArgs &a, int max_slots, bool gateup, bool down, const DeviceInfo &dev);

// gate/up + SwiGLU: routes in every CTA (publishing from CTA 0), writes h
// (and the max |h| words when want_hmax).
cudaError_t moe_k16_gateup_launch(epq_fmt fmt, const MoeArgs &a, int max_slots, bool want_hmax,
                                  const DeviceInfo &dev, cudaStream_t s);
// down + weighted combine + residual: reads the published routing and h, writes y.
cudaError_t moe_k16_down_launch(epq_fmt fmt, const MoeArgs &a, int max_slots, const DeviceInfo &dev,
                                cudaStream_t s);

}  // namespace epq

"""epq: block-quantized decode kernels for GB300 (sm_103a).

The compute lives in libepq.so (hand-written CUDA, C ABI in include/epq.h);
this package only marshals torch tensors into that ABI.
"""
from ._lib import (  # noqa: F401
    EPQ_Q8_0, EPQ_Q4_0, EPQ_Q4_1, EPQ_Q4_K, EPQ_Q2_K, EPQ_Q6_K, FORMATS, EpqError, declared_symbols, load,
    epq_row_bytes, epq_block_weights, epq_block_bytes, epq_status_string, epq_device_error, epq_device_error_detail,
    epq_quantize, epq_dequantize, epq_gemv, epq_gemv_ex, epq_set_tuning, EPQ_TUNE_TILE_BYTES, EPQ_TUNE_RING_BYTES, EPQ_TUNE_GEMV_ENGINE, EPQ_TUNE_EARLY_STAGES, EPQ_TUNE_TC_SPLIT, EPQ_TUNE_ATTN_CHUNK, EPQ_TUNE_VN_CHUNK, EPQ_TUNE_VN_CLUSTER,
    GemvOp, gemv_op, epq_gemv_chain, epq_gemv_chain_workspace_bytes, EPQ_CHAIN_MAX_OPS,
    KVCache, epq_kv_row_bytes, epq_attention_decode,
    MoELayer, epq_moe_workspace_bytes, epq_moe_forward, epq_moe_forward_noalloc, EPQ_MOE_ROUTE, EPQ_MOE_GATE_UP, EPQ_MOE_DOWN,
)

"""CPU oracle for the block-quantized decode path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy restatements of what the CUDA library
computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import it; the library itself never does,
and nothing here imports the library.

Sources (web pages, cited by title and section):

* "端侧推理：llama.cpp 与 GGUF、MLX、ExecuTorch" (edge-inference handbook),
  section "GGUF 的量化格式": the four block formats Q8_0, Q4_0, Q4_1 and the
  simplified Q4_K, the long-tailed weight sample and the printed table of
  bits/weight and relative errors.
* "Flash-MoE：在笔记本上运行 397B 参数大模型", sections "核心技术 / 3. Metal
  计算着色器" and "每层流水线": the expert layer (router softmax + top-K,
  gate/up with SwiGLU, down, weighted combine + residual, optional sigmoid
  gate on the shared expert).
* "EPM：MiniCPM-V-4.7-35B-A3B 的 8 GiB 專家分頁 CPU 推論", section
  "記憶體怎麼配置的": per-expert Q4_K byte sizes that fix the 144-byte superblock.

Precision: quantizer decisions are taken in IEEE float32 (round to nearest
even, true division), as the handbook's listing computes them; GEMV and MoE
reference values are float64.

Pins (tests/test_oracle_*.py): the page's printed relative errors, closed-form
bits/weight, the EPM expert byte sizes, hand-built blocks with exact expected
bytes, brute-force nearest-code checks, brute-force float64 matvec and
top-K-by-sort on tiny shapes, and closed forms for every MoE and attention
step (router logits with a bias, softmax, the combine with and without
renormalising the top-K weights, the sigmoid shared gate, an expert built
from diagonal matrices, the pre-norm).  The pages print no numeric MoE
output, so those pins are closed forms rather than printed values; whether
the top-K weights are renormalised is a reading of the pages (both variants
are pinned and the library takes either).
"""
from .formats import (  # noqa: F401
    Q8_0, Q4_0, Q4_1, Q4_K, Q2_K, Q6_K, FORMATS, BLOCK_WEIGHTS, BLOCK_BYTES,
    row_bytes, bits_per_weight, quantize, dequantize, quantize_dequantize,
)
from .gemv import gemv_f64, gemv_bound  # noqa: F401
from .moe import (  # noqa: F401
    rmsnorm_f64, router_logits_f64, topk_select, softmax_f64, combine_weights,
    expert_forward_f64, moe_forward_f64, MoEWeights, MoEResult,
)

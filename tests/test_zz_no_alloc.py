"""The MoE entry point for callers that cannot allocate device memory.

epq_moe_forward_noalloc takes no workspace: it runs the same three kernels
on a fixed scratch array compiled into the library.  This checks it through
the C ABI against the workspace entry point (epq_moe_forward) on the same
inputs, with the MoE tolerance of tests/test_gpu_moe.py, on two calls in a
row (the second call finds the first call's leftovers in the shared array).
Collected last on purpose, so that a failure here cannot hide the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle.moe import MoEWeights

pytestmark = pytest.mark.gpu


def _layer(epq, dev, fmt, E, H, I, seed):
    R = synthetic.student_t((E, H), seed=seed).numpy()
    gu = np.stack([oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=seed + 1 + e).numpy())
                   for e in range(E)])
    dn = np.stack([oracle.quantize(fmt, synthetic.student_t((H, I), seed=seed + 100 + e).numpy())
                   for e in range(E)])
    sgu = oracle.quantize(fmt, synthetic.student_t((2 * I, H), seed=seed + 200).numpy())
    sdn = oracle.quantize(fmt, synthetic.student_t((H, I), seed=seed + 201).numpy())
    mw = MoEWeights(fmt=fmt, hidden=H, inter=I, router=R, gate_up=gu, down=dn, shared_gate_up=sgu,
                    shared_down=sdn)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    layer = epq.MoELayer(fmt, t(R), t(gu), t(dn), shared_gate_up=t(sgu), shared_down=t(sdn))
    return mw, layer


def _bound(mw, x, ref):
    """Per-element end-to-end scale |x| + sum_k w_k A_k + A_s (float64 oracle)."""
    fmt, H, I = mw.fmt, mw.hidden, mw.inter
    b = np.abs(x.astype(np.float64)).copy()
    for t in range(x.shape[0]):
        slots = [(ref.w[t, k], mw.gate_up[e], mw.down[e]) for k, e in enumerate(ref.idx[t])]
        slots.append((1.0, mw.shared_gate_up, mw.shared_down))
        for wk, GU, D in slots:
            h = oracle.expert_forward_f64(fmt, GU, D, H, I, ref.xin[t])[3]
            b[t] += abs(wk) * oracle.gemv_bound(fmt, D, h[0], I)[0]
    return b


# fmt, E, H, I, topk, ntok, engine (EPQ_TUNE_GEMV_ENGINE)
CASES = [
    (oracle.Q4_K, 16, 1024, 512, 4, 3, 0),    # Q4_K, 3 tokens: chunks of two on the tensor-core kernels
    (oracle.Q4_K, 16, 1024, 512, 4, 3, 1),    # the same on the CUDA-core kernels, one pass
    (oracle.Q4_0, 16, 1024, 512, 4, 3, 0),    # another format: CUDA-core kernels
    (oracle.Q4_0, 32, 1024, 1792, 8, 16, 0),  # workspace 1,046,784 B: all but 1.8 KB of the array
    (oracle.Q2_K, 16, 1024, 512, 4, 3, 0),    # 2-bit experts: the 16-weight sub-block kernels, chunks of two
    (oracle.Q6_K, 12, 1280, 768, 3, 2, 0),    # Q6_K rows of an odd number of superblocks
]


@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_workspace_entry(epq_lib, cuda_dev, case):
    fmt, E, H, I, topk, ntok, engine = case
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, engine)
    try:
        _noalloc_case(epq_lib, cuda_dev, fmt, E, H, I, topk, ntok)
    finally:
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


def _noalloc_case(epq_lib, cuda_dev, fmt, E, H, I, topk, ntok):
    mw, layer = _layer(epq_lib, cuda_dev, fmt, E, H, I, seed=4321 + I)
    assert layer.workspace_bytes(ntok, topk) <= (1 << 20)
    x = synthetic.normal((ntok, H), seed=99, scale=2.0).numpy()
    xs = torch.from_numpy(x).to(cuda_dev)

    idx_ref = torch.empty((ntok, topk), dtype=torch.int32, device=cuda_dev)
    w_ref = torch.empty((ntok, topk), dtype=torch.float32, device=cuda_dev)
    y_ref, _, _ = epq_lib.epq_moe_forward(layer, xs, topk, topk_idx=idx_ref, topk_w=w_ref)
    torch.cuda.synchronize()
    y_ref = y_ref.cpu().numpy()

    ref = oracle.moe_forward_f64(mw, x, topk)
    tol = 1e-3 * _bound(mw, x, ref)
    for call in range(2):
        y = torch.full_like(xs, float("nan"))
        idx = torch.full((ntok, topk), -1, dtype=torch.int32, device=cuda_dev)
        w = torch.zeros((ntok, topk), dtype=torch.float32, device=cuda_dev)
        epq_lib.epq_moe_forward_noalloc(layer, xs, topk, y, topk_idx=idx, topk_w=w)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert torch.equal(idx, idx_ref), f"call {call}: top-K differs"
        assert np.allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=1e-6, atol=0), f"call {call}: weights"
        err = np.abs(got.astype(np.float64) - y_ref)
        assert (err <= tol).all(), f"call {call}: worst {(err / tol).max():.3g} of the tolerance"
    assert epq_lib.epq_device_error() == 0


def test_noalloc_rejects_oversized_shapes(epq_lib, cuda_dev):
    """A shape whose workspace exceeds the fixed 1 MiB is refused up front."""
    from moe_experts_gb300._lib import Experts, MoeOpts, Router, load
    lib = load()
    dummy = torch.zeros(4096, dtype=torch.uint8, device=cuda_dev)
    x = torch.zeros((16, 256), device=cuda_dev)
    r = Router(dummy.data_ptr(), None, 64, 1)
    e = Experts(3, 64, 256, 16384, dummy.data_ptr(), 0, dummy.data_ptr(), 0, None, None, None)
    o = MoeOpts(0, 0.0, None, None, 0)
    need = lib.epq_moe_workspace_bytes(ctypes.byref(r), ctypes.byref(e), 16, 16)
    assert need > (1 << 20)
    st = lib.epq_moe_forward_noalloc(ctypes.byref(r), ctypes.byref(e), ctypes.c_void_p(x.data_ptr()), 16, 16,
                                     ctypes.byref(o), ctypes.c_void_p(x.data_ptr()), None, None,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 5  # EPQ_ERR_WORKSPACE

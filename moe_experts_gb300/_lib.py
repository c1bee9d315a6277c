"""ctypes binding of libepq.so (include/epq.h): argument marshalling only.

Every function here forwards to the C ABI of the same name.  Tensors are
torch CUDA tensors; their device pointers and torch's current CUDA stream are
passed through.  Output tensors that the caller does not supply are
allocated with torch (device memory is torch's business; the library itself
never allocates).  There is no fallback: if the shared library is missing or
a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libepq.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "epq.h")

EPQ_Q8_0, EPQ_Q4_0, EPQ_Q4_1, EPQ_Q4_K, EPQ_Q2_K, EPQ_Q6_K = 0, 1, 2, 3, 4, 5
FORMATS = {"Q8_0": EPQ_Q8_0, "Q4_0": EPQ_Q4_0, "Q4_1": EPQ_Q4_1, "Q4_K": EPQ_Q4_K, "Q2_K": EPQ_Q2_K,
           "Q6_K": EPQ_Q6_K}

_lib = None


class EpqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _lib.epq_status_string(status).decode() if _lib else str(status)
        extra = f" (cudaError {_lib.epq_last_cuda_error()})" if _lib and status == 6 else ""
        super().__init__(f"{fn} failed: {msg}{extra}")
        self.status = status


class GemvOpts(ctypes.Structure):
    _fields_ = [("residual", ctypes.c_void_p), ("rms_prenorm", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("swiglu", ctypes.c_int), ("x_group", ctypes.c_int), ("x_head_dim", ctypes.c_int),
                ("x_ld", ctypes.c_int64), ("weights_ready", ctypes.c_int)]


class GemvOp(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("swiglu", ctypes.c_int), ("rms_prenorm", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("x_group", ctypes.c_int), ("x_head_dim", ctypes.c_int), ("x_ld", ctypes.c_int64)]


class Router(ctypes.Structure):
    _fields_ = [("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("n_experts", ctypes.c_int),
                ("norm_topk", ctypes.c_int)]


class Experts(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("n_experts", ctypes.c_int), ("hidden", ctypes.c_int),
                ("inter", ctypes.c_int), ("gate_up", ctypes.c_void_p), ("gate_up_stride", ctypes.c_int64),
                ("down", ctypes.c_void_p), ("down_stride", ctypes.c_int64), ("shared_gate_up", ctypes.c_void_p),
                ("shared_down", ctypes.c_void_p), ("shared_gate_vec", ctypes.c_void_p),
                ("down_fmt_set", ctypes.c_int), ("down_fmt", ctypes.c_int)]


class MoeOpts(ctypes.Structure):
    _fields_ = [("rms_prenorm", ctypes.c_int), ("rms_eps", ctypes.c_float), ("logits_out", ctypes.c_void_p),
                ("h_out", ctypes.c_void_p), ("stages", ctypes.c_int)]


EPQ_MOE_ROUTE, EPQ_MOE_GATE_UP, EPQ_MOE_DOWN = 1, 2, 4


def declared_symbols() -> list[str]:
    """Every function the public header declares."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(epq_[a-z0-9_]+)\s*\(", text)))


def load(path: str | None = None):
    """Load libepq.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with moe_experts_gb300.build.build()")
    lib = ctypes.CDLL(path)
    i64, vp, i32, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "epq_status_string": (ctypes.c_char_p, [i32]),
        "epq_last_cuda_error": (i32, []),
        "epq_device_error": (i32, []),
        "epq_device_error_detail": (i32, [ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "epq_block_weights": (i64, [i32]),
        "epq_block_bytes": (i64, [i32]),
        "epq_row_bytes": (i64, [i32, i64]),
        "epq_set_tuning": (i32, [i32, i32]),
        "epq_quantize": (i32, [i32, vp, i64, i64, vp, vp]),
        "epq_dequantize": (i32, [i32, vp, i64, i64, vp, vp]),
        "epq_gemv": (i32, [i32, vp, vp, vp, i64, i64, i32, vp]),
        "epq_gemv_ex": (i32, [i32, vp, vp, vp, i64, i64, i32, ctypes.POINTER(GemvOpts), vp]),
        "epq_moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Router), ctypes.POINTER(Experts), i32, i32]),
        "epq_moe_forward": (i32, [ctypes.POINTER(Router), ctypes.POINTER(Experts), vp, i32, i32,
                                  ctypes.POINTER(MoeOpts), vp, vp, vp, vp, ctypes.c_size_t, vp]),
        "epq_gemv_chain_workspace_bytes": (ctypes.c_size_t, []),
        "epq_gemv_chain": (i32, [i32, ctypes.POINTER(GemvOp), i32, i32, vp, ctypes.c_size_t, vp]),
        "epq_moe_forward_noalloc": (i32, [ctypes.POINTER(Router), ctypes.POINTER(Experts), vp, i32, i32,
                                          ctypes.POINTER(MoeOpts), vp, vp, vp, vp]),
        "epq_kv_row_bytes": (i64, [i32]),
        "epq_attention_decode": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, f32, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, st: int):
    if st != 0:
        raise EpqError(fn, st)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------------ host-only queries
def epq_row_bytes(fmt: int, cols: int) -> int:
    return int(load().epq_row_bytes(fmt, cols))


def epq_block_weights(fmt: int) -> int:
    return int(load().epq_block_weights(fmt))


def epq_block_bytes(fmt: int) -> int:
    return int(load().epq_block_bytes(fmt))


EPQ_TUNE_TILE_BYTES, EPQ_TUNE_RING_BYTES, EPQ_TUNE_GEMV_ENGINE, EPQ_TUNE_EARLY_STAGES, EPQ_TUNE_TC_SPLIT = 1, 2, 3, 4, 5
EPQ_TUNE_ATTN_CHUNK, EPQ_TUNE_VN_CHUNK, EPQ_TUNE_VN_CLUSTER = 6, 7, 8


def epq_set_tuning(key: int, value: int) -> int:
    return int(load().epq_set_tuning(key, value))


def epq_status_string(st: int) -> str:
    return load().epq_status_string(st).decode()


def epq_device_error() -> int:
    return int(load().epq_device_error())


def epq_device_error_detail() -> tuple[int, int, int, int]:
    """(code, block, pipeline step, thread) of the first wait timeout; clears it."""
    b, w, t = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    code = load().epq_device_error_detail(ctypes.byref(b), ctypes.byref(w), ctypes.byref(t))
    return int(code), b.value, w.value, t.value


# ------------------------------------------------------------------ packing
def epq_quantize(fmt: int, W: torch.Tensor, blocks: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """W float32 [rows, cols] (CUDA) -> packed uint8 [rows, row_bytes]."""
    lib = load()
    rows, cols = W.shape
    rb = lib.epq_row_bytes(fmt, cols)
    if blocks is None:
        blocks = torch.empty((rows, max(rb, 0)), dtype=torch.uint8, device=W.device)
    _check("epq_quantize", lib.epq_quantize(fmt, _ptr(W), rows, cols, _ptr(blocks), _stream(stream)))
    return blocks


def epq_dequantize(fmt: int, blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    lib = load()
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=blocks.device)
    _check("epq_dequantize", lib.epq_dequantize(fmt, _ptr(blocks), rows, cols, _ptr(out), _stream(stream)))
    return out


# ------------------------------------------------------------------ GEMV
def epq_gemv(fmt: int, blocks: torch.Tensor, x: torch.Tensor, rows: int, cols: int, y: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """x float32 [nvec, cols] (or [cols]) -> y float32 [nvec, rows]."""
    lib = load()
    x2 = x if x.dim() == 2 else x.view(1, -1)
    nvec = x2.shape[0]
    if y is None:
        y = torch.empty((nvec, rows), dtype=torch.float32, device=x.device)
    _check("epq_gemv", lib.epq_gemv(fmt, _ptr(blocks), _ptr(x2), _ptr(y), rows, cols, nvec, _stream(stream)))
    return y


def epq_gemv_ex(fmt: int, blocks: torch.Tensor, x: torch.Tensor, rows: int, cols: int, y: torch.Tensor | None = None,
                residual: torch.Tensor | None = None, rms_prenorm: bool = False, rms_eps: float = 0.0,
                swiglu: bool = False, x_group: int = 0, x_head_dim: int = 0, weights_ready: bool = False,
                stream=None) -> torch.Tensor:
    lib = load()
    x2 = x if x.dim() == 2 else x.view(1, -1)
    nvec = x2.shape[0]
    if x2.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    x_ld = x2.stride(0) if nvec > 1 else 0
    rows_out = rows // 2 if swiglu else rows
    if y is None:
        y = torch.empty((nvec, rows_out), dtype=torch.float32, device=x.device)
    o = GemvOpts(residual.data_ptr() if residual is not None else None, int(rms_prenorm), float(rms_eps),
                 int(swiglu), int(x_group), int(x_head_dim), int(x_ld), int(weights_ready))
    _check("epq_gemv_ex", lib.epq_gemv_ex(fmt, _ptr(blocks), _ptr(x2), _ptr(y), rows, cols, nvec,
                                          ctypes.byref(o), _stream(stream)))
    return y


EPQ_CHAIN_MAX_OPS = 256


def epq_gemv_chain_workspace_bytes() -> int:
    return int(load().epq_gemv_chain_workspace_bytes())


def gemv_op(blocks: torch.Tensor, x: torch.Tensor, y: torch.Tensor, rows: int, cols: int,
            residual: torch.Tensor | None = None, swiglu: bool = False, rms_prenorm: bool = False,
            rms_eps: float = 0.0, x_group: int = 0, x_head_dim: int = 0) -> GemvOp:
    """One op of epq_gemv_chain; x and y are [nvec, n] views (rows contiguous)."""
    x2 = x if x.dim() == 2 else x.view(1, -1)
    if x2.stride(1) != 1:
        raise ValueError("x rows must be contiguous")
    x_ld = x2.stride(0) if x2.shape[0] > 1 else 0
    return GemvOp(_ptr(blocks), _ptr(x2), _ptr(y), residual.data_ptr() if residual is not None else None,
                  int(rows), int(cols), int(swiglu), int(rms_prenorm), float(rms_eps), int(x_group),
                  int(x_head_dim), int(x_ld))


def epq_gemv_chain(fmt: int, ops: list, nvec: int, workspace: torch.Tensor, stream=None) -> None:
    """Run the ops (GemvOp list) in order in one persistent launch."""
    lib = load()
    arr = (GemvOp * len(ops))(*ops)
    _check("epq_gemv_chain", lib.epq_gemv_chain(fmt, arr, len(ops), nvec, _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream(stream)))


# ------------------------------------------------------------------ MoE layer
def _addr(t):
    return None if t is None else t.data_ptr()


class MoELayer:
    """Device-resident MoE weights in the layout epq_moe_forward expects.

    router [E, H] float32; gate_up uint8 [E, 2*I, row_bytes(H)] (gate rows
    then up rows); down uint8 [E, H, row_bytes(I)]; optional shared expert
    (same shapes without E) and shared gate vector [H].  down_fmt: the
    format of the down projections when it differs from fmt (a mixed
    per-tensor recipe).
    """

    def __init__(self, fmt, router, gate_up, down, router_bias=None, shared_gate_up=None, shared_down=None,
                 shared_gate_vec=None, norm_topk=True, down_fmt=None):
        self.fmt = int(fmt)
        self.down_fmt = self.fmt if down_fmt is None else int(down_fmt)
        self.router, self.router_bias = router, router_bias
        self.gate_up, self.down = gate_up, down
        self.shared_gate_up, self.shared_down, self.shared_gate_vec = shared_gate_up, shared_down, shared_gate_vec
        self.E, self.H = router.shape
        self.I = down.shape[2] * epq_block_weights(self.down_fmt) // epq_block_bytes(self.down_fmt)
        self.norm_topk = bool(norm_topk)
        self._r = Router(_addr(router), _addr(router_bias), self.E, int(self.norm_topk))
        self._x = Experts(self.fmt, self.E, self.H, self.I, _addr(gate_up), gate_up[0].numel(), _addr(down),
                          down[0].numel(), _addr(shared_gate_up), _addr(shared_down), _addr(shared_gate_vec),
                          int(self.down_fmt != self.fmt), self.down_fmt)

    def workspace_bytes(self, ntok: int, topk: int) -> int:
        return int(load().epq_moe_workspace_bytes(ctypes.byref(self._r), ctypes.byref(self._x), ntok, topk))


def epq_moe_workspace_bytes(layer: MoELayer, ntok: int, topk: int) -> int:
    return layer.workspace_bytes(ntok, topk)


def epq_moe_forward(layer: MoELayer, x: torch.Tensor, topk: int, y: torch.Tensor | None = None,
                    topk_idx: torch.Tensor | None = None, topk_w: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, rms_prenorm: bool = False, rms_eps: float = 0.0,
                    logits_out: torch.Tensor | None = None, h_out: torch.Tensor | None = None, stages: int = 0,
                    stream=None):
    """x float32 [ntok, H] -> y float32 [ntok, H]; returns (y, topk_idx, topk_w)."""
    lib = load()
    ntok = x.shape[0]
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = torch.empty(layer.workspace_bytes(ntok, topk), dtype=torch.uint8, device=x.device)
    o = MoeOpts(int(rms_prenorm), float(rms_eps), _addr(logits_out), _addr(h_out), int(stages))
    _check("epq_moe_forward", lib.epq_moe_forward(
        ctypes.byref(layer._r), ctypes.byref(layer._x), _ptr(x), ntok, topk, ctypes.byref(o), _ptr(y),
        _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y, topk_idx, topk_w


def epq_moe_forward_noalloc(layer: MoELayer, x: torch.Tensor, topk: int, y: torch.Tensor,
                            topk_idx: torch.Tensor | None = None, topk_w: torch.Tensor | None = None,
                            rms_prenorm: bool = False, rms_eps: float = 0.0, stream=None):
    """The MoE layer with the library's fixed scratch instead of a workspace.

    For callers that cannot allocate device memory: nothing is allocated
    here either, so y (and the optional top-K outputs) must be supplied.
    """
    lib = load()
    o = MoeOpts(int(rms_prenorm), float(rms_eps), None, None, 0)
    _check("epq_moe_forward_noalloc", lib.epq_moe_forward_noalloc(
        ctypes.byref(layer._r), ctypes.byref(layer._x), _ptr(x), x.shape[0], topk, ctypes.byref(o), _ptr(y),
        _ptr(topk_idx), _ptr(topk_w), _stream(stream)))
    return y


# ------------------------------------------------------------------ attention
def epq_kv_row_bytes(head_dim: int) -> int:
    return int(load().epq_kv_row_bytes(head_dim))


class KVCache:
    """Device Q8_0 key and value caches of one layer: uint8
    [n_kv_heads, max_pos, epq_kv_row_bytes(head_dim)] each."""

    def __init__(self, n_kv_heads: int, head_dim: int, max_pos: int, device):
        rb = epq_kv_row_bytes(head_dim)
        if rb < 0:
            raise ValueError(f"head_dim {head_dim} not supported")
        self.n_kv_heads, self.head_dim, self.max_pos = n_kv_heads, head_dim, max_pos
        self.k = torch.zeros((n_kv_heads, max_pos, rb), dtype=torch.uint8, device=device)
        self.v = torch.zeros_like(self.k)


def epq_attention_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cache: KVCache, n_heads: int,
                         pos: int, scale: float, skip_log: float = float("-inf"), out: torch.Tensor | None = None,
                         scores_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q [n_heads*D], k_new/v_new [n_kv*D] (float32, device) -> out [n_heads*D]."""
    lib = load()
    if out is None:
        out = torch.empty(n_heads * cache.head_dim, dtype=torch.float32, device=q.device)
    _check("epq_attention_decode", lib.epq_attention_decode(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cache.k), _ptr(cache.v), n_heads, cache.n_kv_heads, cache.head_dim,
        int(pos), cache.max_pos, float(scale), float(skip_log), _ptr(out), _ptr(scores_out), _stream(stream)))
    return out

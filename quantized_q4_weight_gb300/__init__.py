"""Python binding of libqgemv (include/qgemv.h): the Q4_0-weight x
Q8_0-activation decode GEMV on one GB300.

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors supply device pointers; work is enqueued on the current torch CUDA
stream.  The library is loaded from this directory (libqgemv.so, built by
``quantized_q4_weight_gb300._build.build()``); if it is missing, every call
raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

QK = 32
Q4_0_BYTES = 18
W_GGML, W_PACKED = 0, 1

STATUS = {0: "QGEMV_OK", 1: "QGEMV_ERR_INVALID_ARG", 2: "QGEMV_ERR_MISALIGNED", 3: "QGEMV_ERR_UNSUPPORTED",
          4: "QGEMV_ERR_WORKSPACE", 5: "QGEMV_ERR_CUDA", 6: "QGEMV_ERR_TIMEOUT", 7: "QGEMV_ERR_BAD_ID",
          8: "QGEMV_ERR_INTERNAL"}


class QgemvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class SeqItem(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("xq", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class SeqF32Item(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class SeqEpItem(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p)]


class GatherMatrix(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("expert_stride", ctypes.c_int64), ("xq", ctypes.c_void_p),
                ("xq_stride", ctypes.c_int64), ("y", ctypes.c_void_p), ("y_stride", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class GatherF32Matrix(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("expert_stride", ctypes.c_int64), ("x", ctypes.c_void_p),
                ("x_stride", ctypes.c_int64), ("y", ctypes.c_void_p), ("y_stride", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


_lib = None

_VP, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "qgemv_status_string": ([_I32], ctypes.c_char_p),
    "qgemv_version": ([], _I32),
    "qgemv_q4_0_bytes": ([_I64, _I64], _SZ),
    "qgemv_xq_bytes": ([_I32, _I64], _SZ),
    "qgemv_pack_q4_0": ([_VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_unpack_q4_0": ([_VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_quantize_q8_0": ([_VP, _VP, _I32, _I64, _I32, _VP], _I32),
    "qgemv_workspace_bytes": ([_I64, _I64, _I32], _SZ),
    "qgemv_q4_0": ([_VP, _I32, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_q4_0_f32": ([_VP, _I32, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_q4_0_argmax": ([_VP, _I32, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_q4_0_argmax_f32": ([_VP, _I32, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_q4_0_argmax_noalloc": ([_VP, _I32, _VP, _VP, _VP, _I64, _I64, _I32, _VP], _I32),
    "qgemv_q4_0_top2": ([_VP, _I32, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_q4_0_top2_f32": ([_VP, _I32, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_verify_commit": ([_VP, _VP, _I32, _I32, _VP, _VP], _I32),
    "qgemv_q4_0_verify_f32": ([_VP, _I32, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_ffn_workspace_bytes": ([_I64, _I64, _I32], _SZ),
    "qgemv_q4_0_ffn": ([_VP, _VP, _VP, _I32, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_q4_0_ffn_residual": ([_VP, _VP, _VP, _I32, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_debug_silu_mul_q8": ([_VP, _VP, _VP, _I32, _I64, _VP], _I32),
    "qgemv_pack_q8_0": ([_VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_unpack_q8_0": ([_VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_requant_f32_q4_0": ([_VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_requant_q8_0_q4_0": ([_VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_q8_0_workspace_bytes": ([_I64, _I64, _I32], _SZ),
    "qgemv_q8_0": ([_VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_seq_workspace_bytes": ([ctypes.POINTER(SeqItem), _I32, _I32], _SZ),
    "qgemv_q4_0_seq": ([ctypes.POINTER(SeqItem), _I32, _I32, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_seq_f32_workspace_bytes": ([ctypes.POINTER(SeqF32Item), _I32, _I32], _SZ),
    "qgemv_q4_0_seq_f32": ([ctypes.POINTER(SeqF32Item), _I32, _I32, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_seq_ep_workspace_bytes": ([ctypes.POINTER(SeqEpItem), _I32, _I32, _I32], _SZ),
    "qgemv_q4_0_seq_ep": ([ctypes.POINTER(SeqEpItem), _I32, _I32, _I32, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_gather_workspace_bytes": ([ctypes.POINTER(GatherMatrix), _I32, _I32, _I32], _SZ),
    "qgemv_q4_0_gather": ([ctypes.POINTER(GatherMatrix), _I32, _VP, _I32, _I32, _I32, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_gather_f32_workspace_bytes": ([ctypes.POINTER(GatherF32Matrix), _I32, _I32, _I32], _SZ),
    "qgemv_q4_0_gather_f32": ([ctypes.POINTER(GatherF32Matrix), _I32, _VP, _I32, _I32, _I32, _I32, _VP, _SZ, _VP],
                              _I32),
    "qgemv_gs64_bytes": ([_I64, _I64], _SZ),
    "qgemv_pack_gs64": ([_VP, _VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_unpack_gs64": ([_VP, _VP, _VP, _I64, _I64, _VP], _I32),
    "qgemv_quantize_vec_i8": ([_VP, _VP, _VP, _I32, _I64, _VP], _I32),
    "qgemv_gs64_workspace_bytes": ([_I64, _I64, _I32], _SZ),
    "qgemv_gs64": ([_VP, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_gs64_f32": ([_VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ, _VP], _I32),
    "qgemv_debug_block_isums": ([_VP, _I32, _VP, _VP, _I64, _I64, _I32, _VP], _I32),
    "qgemv_debug_block_isums_tc": ([_VP, _I32, _VP, _VP, _I64, _I64, _I32, _I32, _VP], _I32),
    "qgemv_debug_stream_read": ([_VP, _SZ, _I32, _I32, _I32, _I32, _VP, _VP], _I32),
    "qgemv_set_tuning": ([_I32, _I32, _I32, _I32], _I32),
    "qgemv_set_tc_min_tokens": ([_I32], _I32),
    "qgemv_set_ffn_fused": ([_I32], _I32),
    "qgemv_device_status": ([ctypes.POINTER(ctypes.c_int)], _I32),
}


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libqgemv is not built ({_build.LIB} missing): run "
                               "quantized_q4_weight_gb300._build.build() first")
        L = ctypes.CDLL(_build.LIB)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(code: int, what: str):
    if code != 0:
        raise QgemvError(code, what)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


# ----------------------------------------------------------------- sizes

def q4_0_bytes(N: int, K: int) -> int:
    return int(lib().qgemv_q4_0_bytes(N, K))


def xq_bytes(R: int, K: int) -> int:
    return int(lib().qgemv_xq_bytes(R, K))


def workspace_bytes(N: int, K: int, T: int) -> int:
    return int(lib().qgemv_workspace_bytes(N, K, T))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (the library keeps its counters at zero)."""
    return torch.zeros(max(int(nbytes), 16384), dtype=torch.uint8, device=device or "cuda")


# ----------------------------------------------------------------- calls

def pack_q4_0(w_ggml: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty(q4_0_bytes(N, K), dtype=torch.uint8, device=w_ggml.device)
    _check(lib().qgemv_pack_q4_0(_ptr(w_ggml), _ptr(out), N, K, _stream(stream)), "qgemv_pack_q4_0")
    return out


def unpack_q4_0(w_packed: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None):
    out = out if out is not None else torch.empty(q4_0_bytes(N, K), dtype=torch.uint8, device=w_packed.device)
    _check(lib().qgemv_unpack_q4_0(_ptr(w_packed), _ptr(out), N, K, _stream(stream)), "qgemv_unpack_q4_0")
    return out


def quantize_q8_0(x: torch.Tensor, R: int, K: int, batch: int = 1, out: torch.Tensor | None = None, stream=None):
    """x fp32 [batch, R, K] (any shape with that many elements) -> planar Q8_0 bytes."""
    assert x.dtype == torch.float32 and x.numel() == batch * R * K
    out = out if out is not None else torch.empty(batch * xq_bytes(R, K), dtype=torch.uint8, device=x.device)
    _check(lib().qgemv_quantize_q8_0(_ptr(x), _ptr(out), R, K, batch, _stream(stream)), "qgemv_quantize_q8_0")
    return out


def gemv(W, layout: int, xq, N: int, K: int, T: int, ws, y=None, stream=None) -> torch.Tensor:
    y = y if y is not None else torch.empty((T, N), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_q4_0(_ptr(W), layout, _ptr(xq), _ptr(y), N, K, T, _ptr(ws), ws.numel(), _stream(stream)),
           "qgemv_q4_0")
    return y


def gemv_f32(W, layout: int, x, N: int, K: int, T: int, ws, y=None, stream=None) -> torch.Tensor:
    y = y if y is not None else torch.empty((T, N), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_q4_0_f32(_ptr(W), layout, _ptr(x), _ptr(y), N, K, T, _ptr(ws), ws.numel(), _stream(stream)),
           "qgemv_q4_0_f32")
    return y


def gemv_argmax(W, layout: int, xq, N: int, K: int, T: int, ws, y=None, idx=None, stream=None):
    idx = idx if idx is not None else torch.empty(T, dtype=torch.int64, device=W.device)
    _check(lib().qgemv_q4_0_argmax(_ptr(W), layout, _ptr(xq), _ptr(y), _ptr(idx), N, K, T, _ptr(ws), ws.numel(),
                                   _stream(stream)), "qgemv_q4_0_argmax")
    return idx


def gemv_argmax_f32(W, layout: int, x, N: int, K: int, T: int, ws, y=None, idx=None, stream=None):
    """Argmax of W . x over rows for fp32 x[T][K] (quantised inside the kernel)."""
    idx = idx if idx is not None else torch.empty(T, dtype=torch.int64, device=W.device)
    _check(lib().qgemv_q4_0_argmax_f32(_ptr(W), layout, _ptr(x), _ptr(y), _ptr(idx), N, K, T, _ptr(ws), ws.numel(),
                                       _stream(stream)), "qgemv_q4_0_argmax_f32")
    return idx


def gemv_top2(W, layout: int, xq, N: int, K: int, T: int, ws, y=None, idx2=None, val2=None, stream=None):
    """The two best rows per token and their outputs: (idx2 int64 [T][2], val2 fp32 [T][2])."""
    idx2 = idx2 if idx2 is not None else torch.empty((T, 2), dtype=torch.int64, device=W.device)
    val2 = val2 if val2 is not None else torch.empty((T, 2), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_q4_0_top2(_ptr(W), layout, _ptr(xq), _ptr(y), _ptr(idx2), _ptr(val2), N, K, T, _ptr(ws),
                                 ws.numel(), _stream(stream)), "qgemv_q4_0_top2")
    return idx2, val2


def gemv_top2_f32(W, layout: int, x, N: int, K: int, T: int, ws, y=None, idx2=None, val2=None, stream=None):
    """gemv_top2 for fp32 x[T][K] (quantised inside the kernel)."""
    idx2 = idx2 if idx2 is not None else torch.empty((T, 2), dtype=torch.int64, device=W.device)
    val2 = val2 if val2 is not None else torch.empty((T, 2), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_q4_0_top2_f32(_ptr(W), layout, _ptr(x), _ptr(y), _ptr(idx2), _ptr(val2), N, K, T, _ptr(ws),
                                     ws.numel(), _stream(stream)), "qgemv_q4_0_top2_f32")
    return idx2, val2


def verify_f32(W, layout: int, x, tokens, N: int, K: int, T: int, ws, idx2=None, val2=None, n_commit=None,
               stream=None):
    """A verify step in one launch: the top-2 rows of W . x per position and the
    committed count of the verify rule on (tokens, idx2[:, 0])."""
    idx2 = idx2 if idx2 is not None else torch.empty((T, 2), dtype=torch.int64, device=W.device)
    val2 = val2 if val2 is not None else torch.empty((T, 2), dtype=torch.float32, device=W.device)
    n_commit = n_commit if n_commit is not None else torch.empty(1, dtype=torch.int32, device=W.device)
    _check(lib().qgemv_q4_0_verify_f32(_ptr(W), layout, _ptr(x), _ptr(tokens), _ptr(idx2), _ptr(val2), _ptr(n_commit),
                                       N, K, T, _ptr(ws), ws.numel(), _stream(stream)), "qgemv_q4_0_verify_f32")
    return idx2, val2, n_commit


def verify_commit(tokens, pred, n_commit=None, stream=None):
    """Committed predictions of one verify step (int32 device scalar): tokens[0]
    is the current token, tokens[1:] the drafts, pred[t] the prediction after
    tokens[:t+1] (int64 device tensors; pred may be a strided column such as
    idx2[:, 0] of gemv_top2)."""
    T = tokens.numel()
    assert pred.dim() == 1 and pred.numel() == T and tokens.is_contiguous()
    n_commit = n_commit if n_commit is not None else torch.empty(1, dtype=torch.int32, device=tokens.device)
    _check(lib().qgemv_verify_commit(_ptr(tokens), ctypes.c_void_p(pred.data_ptr()), pred.stride(0), T,
                                     _ptr(n_commit), _stream(stream)), "qgemv_verify_commit")
    return n_commit


def ffn_workspace_bytes(d_model: int, d_ff: int, T: int) -> int:
    return int(lib().qgemv_ffn_workspace_bytes(d_model, d_ff, T))


def ffn(W_gate, W_up, W_down, layout: int, x, d_model: int, d_ff: int, T: int, ws, y=None, stream=None):
    """y[T][d_model] = W_down . Q8_0(SiLU(W_gate . x) * (W_up . x)) for fp32 x[T][d_model]."""
    y = y if y is not None else torch.empty((T, d_model), dtype=torch.float32, device=x.device)
    _check(lib().qgemv_q4_0_ffn(_ptr(W_gate), _ptr(W_up), _ptr(W_down), layout, _ptr(x), _ptr(y), d_model, d_ff, T,
                                _ptr(ws), ws.numel(), _stream(stream)), "qgemv_q4_0_ffn")
    return y


def ffn_residual(W_gate, W_up, W_down, layout: int, x, residual, d_model: int, d_ff: int, T: int, ws, y=None,
                 stream=None):
    """y = residual + W_down . Q8_0(SiLU(W_gate . x) * (W_up . x)); residual may be y."""
    y = y if y is not None else torch.empty((T, d_model), dtype=torch.float32, device=x.device)
    _check(lib().qgemv_q4_0_ffn_residual(_ptr(W_gate), _ptr(W_up), _ptr(W_down), layout, _ptr(x), _ptr(residual),
                                         _ptr(y), d_model, d_ff, T, _ptr(ws), ws.numel(), _stream(stream)),
           "qgemv_q4_0_ffn_residual")
    return y


def silu_mul_q8(g, u, T: int, F: int, hq=None, stream=None):
    """Test hook: planar Q8_0 codes of SiLU(g) * u (g, u fp32 [T][F])."""
    hq = hq if hq is not None else torch.empty(xq_bytes(T, F), dtype=torch.uint8, device=g.device)
    _check(lib().qgemv_debug_silu_mul_q8(_ptr(g), _ptr(u), _ptr(hq), T, F, _stream(stream)), "qgemv_debug_silu_mul_q8")
    return hq


def q8_0_bytes(N: int, K: int) -> int:
    return 34 * N * (K // QK)


def pack_q8_0(w_ggml: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """GGML Q8_0 weights (uint8 [34 N K/32]) -> the device layout (same bytes)."""
    out = out if out is not None else torch.empty(q8_0_bytes(N, K), dtype=torch.uint8, device=w_ggml.device)
    _check(lib().qgemv_pack_q8_0(_ptr(w_ggml), _ptr(out), N, K, _stream(stream)), "qgemv_pack_q8_0")
    return out


def unpack_q8_0(w_packed: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None):
    out = out if out is not None else torch.empty(q8_0_bytes(N, K), dtype=torch.uint8, device=w_packed.device)
    _check(lib().qgemv_unpack_q8_0(_ptr(w_packed), _ptr(out), N, K, _stream(stream)), "qgemv_unpack_q8_0")
    return out


def requant_f32_q4_0(w: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 weights [N][K] -> GGML Q4_0 blocks (uint8 [18 N K/32]), GGML's q4_0 encoder."""
    out = out if out is not None else torch.empty(q4_0_bytes(N, K), dtype=torch.uint8, device=w.device)
    _check(lib().qgemv_requant_f32_q4_0(_ptr(w), _ptr(out), N, K, _stream(stream)), "qgemv_requant_f32_q4_0")
    return out


def requant_q8_0_q4_0(w_q8: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None):
    """GGML Q8_0 weights (uint8 [34 N K/32]) -> GGML Q4_0 blocks (uint8 [18 N K/32])."""
    out = out if out is not None else torch.empty(q4_0_bytes(N, K), dtype=torch.uint8, device=w_q8.device)
    _check(lib().qgemv_requant_q8_0_q4_0(_ptr(w_q8), _ptr(out), N, K, _stream(stream)), "qgemv_requant_q8_0_q4_0")
    return out


def q8_0_workspace_bytes(N: int, K: int, T: int) -> int:
    return int(lib().qgemv_q8_0_workspace_bytes(N, K, T))


def gemv_q8_0(W, xq, N: int, K: int, T: int, ws=None, y=None, stream=None) -> torch.Tensor:
    """y[T][N] for packed Q8_0 weights and planar Q8_0 activations."""
    y = y if y is not None else torch.empty((T, N), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_q8_0(_ptr(W), _ptr(xq), _ptr(y), N, K, T, _ptr(ws), 0 if ws is None else ws.numel(),
                            _stream(stream)), "qgemv_q8_0")
    return y


def seq_items(entries) -> ctypes.Array:
    """entries: iterable of (W, xq, y, N, K) with CUDA tensors."""
    entries = list(entries)
    arr = (SeqItem * len(entries))()
    for i, (W, xq, y, N, K) in enumerate(entries):
        arr[i] = SeqItem(W.data_ptr(), xq.data_ptr(), y.data_ptr(), N, K)
    return arr


def seq_workspace_bytes(items: ctypes.Array, T: int) -> int:
    return int(lib().qgemv_seq_workspace_bytes(items, len(items), T))


def gemv_seq(items: ctypes.Array, layout: int, T: int, ws, stream=None):
    _check(lib().qgemv_q4_0_seq(items, len(items), layout, T, _ptr(ws), ws.numel(), _stream(stream)),
           "qgemv_q4_0_seq")


def seq_f32_items(entries) -> ctypes.Array:
    """entries: iterable of (W, x, y, N, K) with CUDA tensors (x fp32 [T, K])."""
    entries = list(entries)
    arr = (SeqF32Item * len(entries))()
    for i, (W, x, y, N, K) in enumerate(entries):
        arr[i] = SeqF32Item(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K)
    return arr


def seq_f32_workspace_bytes(items: ctypes.Array, T: int) -> int:
    return int(lib().qgemv_seq_f32_workspace_bytes(items, len(items), T))


def gemv_seq_f32(items: ctypes.Array, layout: int, T: int, ws, stream=None):
    _check(lib().qgemv_q4_0_seq_f32(items, len(items), layout, T, _ptr(ws), ws.numel(), _stream(stream)),
           "qgemv_q4_0_seq_f32")


def seq_ep_items(entries) -> ctypes.Array:
    """entries: iterable of (W, x, y, N, K, bias, residual) with CUDA tensors;
    x planar Q8_0 or fp32 [T, K] (the call's x_f32 says which); bias [N] and
    residual [T, N] fp32 or None (residual may be y)."""
    entries = list(entries)
    arr = (SeqEpItem * len(entries))()
    for i, (W, x, y, N, K, b, r) in enumerate(entries):
        arr[i] = SeqEpItem(W.data_ptr(), x.data_ptr(), y.data_ptr(), N, K,
                           None if b is None else b.data_ptr(), None if r is None else r.data_ptr())
    return arr


def seq_ep_workspace_bytes(items: ctypes.Array, T: int, x_f32: bool = False) -> int:
    return int(lib().qgemv_seq_ep_workspace_bytes(items, len(items), T, int(x_f32)))


def gemv_seq_ep(items: ctypes.Array, layout: int, T: int, ws, x_f32: bool = False, stream=None):
    """y = W . x + bias + residual for every item, in one launch per 200 items."""
    _check(lib().qgemv_q4_0_seq_ep(items, len(items), layout, T, int(x_f32), _ptr(ws), ws.numel(), _stream(stream)),
           "qgemv_q4_0_seq_ep")


def gather_mats(entries) -> ctypes.Array:
    """entries: (W, expert_stride_bytes, xq, xq_stride_bytes, y, y_stride_floats, N, K)."""
    entries = list(entries)
    arr = (GatherMatrix * len(entries))()
    for i, (W, ws_, xq, xs, y, ys, N, K) in enumerate(entries):
        arr[i] = GatherMatrix(W.data_ptr(), ws_, xq.data_ptr(), xs, y.data_ptr(), ys, N, K)
    return arr


def gather_workspace_bytes(mats: ctypes.Array, n_ids: int, T: int) -> int:
    return int(lib().qgemv_gather_workspace_bytes(mats, len(mats), n_ids, T))


def gemv_gather(mats: ctypes.Array, ids, n_experts: int, layout: int, T: int, ws, stream=None):
    _check(lib().qgemv_q4_0_gather(mats, len(mats), _ptr(ids), ids.numel(), n_experts, layout, T, _ptr(ws),
                                   ws.numel(), _stream(stream)), "qgemv_q4_0_gather")


def gather_f32_mats(entries) -> ctypes.Array:
    """entries: (W, expert_stride_bytes, x, x_stride_bytes, y, y_stride_floats, N, K), x fp32."""
    entries = list(entries)
    arr = (GatherF32Matrix * len(entries))()
    for i, (W, ws_, x, xs, y, ys, N, K) in enumerate(entries):
        arr[i] = GatherF32Matrix(W.data_ptr(), ws_, x.data_ptr(), xs, y.data_ptr(), ys, N, K)
    return arr


def gather_f32_workspace_bytes(mats: ctypes.Array, n_ids: int, T: int) -> int:
    return int(lib().qgemv_gather_f32_workspace_bytes(mats, len(mats), n_ids, T))


def gemv_gather_f32(mats: ctypes.Array, ids, n_experts: int, layout: int, T: int, ws, stream=None):
    _check(lib().qgemv_q4_0_gather_f32(mats, len(mats), _ptr(ids), ids.numel(), n_experts, layout, T, _ptr(ws),
                                       ws.numel(), _stream(stream)), "qgemv_q4_0_gather_f32")


def block_isums(W, layout: int, xq, N: int, K: int, T: int, stream=None) -> torch.Tensor:
    out = torch.empty((T, N, K // QK), dtype=torch.int32, device=W.device)
    _check(lib().qgemv_debug_block_isums(_ptr(W), layout, _ptr(xq), _ptr(out), N, K, T, _stream(stream)),
           "qgemv_debug_block_isums")
    return out


def gs64_bytes(N: int, K: int) -> int:
    return int(lib().qgemv_gs64_bytes(N, K))


def pack_gs64(wq, wscale, N: int, K: int, stream=None) -> torch.Tensor:
    """Row planes (nibbles [N][K/64][32] uint8, scales [N][K/64] fp32) -> packed device layout."""
    out = torch.empty(gs64_bytes(N, K), dtype=torch.uint8, device=wq.device)
    _check(lib().qgemv_pack_gs64(_ptr(wq), _ptr(wscale), _ptr(out), N, K, _stream(stream)), "qgemv_pack_gs64")
    return out


def unpack_gs64(W, N: int, K: int, stream=None):
    wq = torch.empty((N, K // 64, 32), dtype=torch.uint8, device=W.device)
    ws = torch.empty((N, K // 64), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_unpack_gs64(_ptr(W), _ptr(wq), _ptr(ws), N, K, _stream(stream)), "qgemv_unpack_gs64")
    return wq, ws


def quantize_vec_i8(x, R: int, K: int, stream=None):
    """fp32 x [R][K] -> (int8 codes [R][K], fp32 scales [R]), one scale per row."""
    q = torch.empty((R, K), dtype=torch.int8, device=x.device)
    s = torch.empty(R, dtype=torch.float32, device=x.device)
    _check(lib().qgemv_quantize_vec_i8(_ptr(x), _ptr(q), _ptr(s), R, K, _stream(stream)), "qgemv_quantize_vec_i8")
    return q, s


def quantize_vec_i8_into(x, q, s, R: int, K: int, stream=None):
    """quantize_vec_i8 into existing buffers."""
    _check(lib().qgemv_quantize_vec_i8(_ptr(x), _ptr(q), _ptr(s), R, K, _stream(stream)), "qgemv_quantize_vec_i8")


def gs64_workspace_bytes(N: int, K: int, T: int) -> int:
    return int(lib().qgemv_gs64_workspace_bytes(N, K, T))


def gemv_gs64(W, q, s, N: int, K: int, T: int, ws=None, y=None, stream=None) -> torch.Tensor:
    if y is None:
        y = torch.empty((T, N), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_gs64(_ptr(W), _ptr(q), _ptr(s), _ptr(y), N, K, T, _ptr(ws) if ws is not None else None,
                            ws.numel() if ws is not None else 0, _stream(stream)), "qgemv_gs64")
    return y


def gemv_gs64_f32(W, x, N: int, K: int, T: int, ws=None, y=None, stream=None) -> torch.Tensor:
    """gs64 GEMV on fp32 activations, quantised per vector inside the launch."""
    if y is None:
        y = torch.empty((T, N), dtype=torch.float32, device=W.device)
    _check(lib().qgemv_gs64_f32(_ptr(W), _ptr(x), _ptr(y), N, K, T, _ptr(ws) if ws is not None else None,
                                ws.numel() if ws is not None else 0, _stream(stream)), "qgemv_gs64_f32")
    return y


def block_isums_tc(W, layout: int, xq, N: int, K: int, T: int, f16_image: bool, stream=None) -> torch.Tensor:
    """The tensor-core path's block sums (see qgemv_debug_block_isums_tc)."""
    out = torch.empty((T, N, K // QK), dtype=torch.int32, device=W.device)
    _check(lib().qgemv_debug_block_isums_tc(_ptr(W), layout, _ptr(xq), _ptr(out), N, K, T, 1 if f16_image else 0,
                                            _stream(stream)), "qgemv_debug_block_isums_tc")
    return out


def stream_read(src, method: int, warps: int, depth: int, stage_bytes: int, sink, stream=None):
    """Measurement hook: stream all of `src` once (see qgemv_debug_stream_read)."""
    _check(lib().qgemv_debug_stream_read(_ptr(src), src.numel() * src.element_size(), method, warps, depth,
                                         stage_bytes, _ptr(sink), _stream(stream)), "qgemv_debug_stream_read")


def set_tuning(ctas_per_sm: int = 0, waves: int = 0, mma_min_T: int = 0, ring_depth: int = 0):
    """Tuning of the streaming kernel (0 = default for each); results are unchanged."""
    _check(lib().qgemv_set_tuning(ctas_per_sm, waves, mma_min_T, ring_depth), "qgemv_set_tuning")


def set_ffn_fused(on: bool = True):
    """The decode FFN step as one fused launch where it applies (else always three launches)."""
    _check(lib().qgemv_set_ffn_fused(1 if on else 0), "qgemv_set_ffn_fused")


def set_tc_min_T(tc_min_T: int = 0):
    """Token count from which packed sequences run on the tcgen05 kernel (0 = default: never; 1..8; 9 = never)."""
    _check(lib().qgemv_set_tc_min_tokens(tc_min_T), "qgemv_set_tc_min_tokens")


def device_status() -> int:
    """Read and clear the device status word (synchronises)."""
    code = ctypes.c_int(0)
    _check(lib().qgemv_device_status(ctypes.byref(code)), "qgemv_device_status")
    return int(code.value)

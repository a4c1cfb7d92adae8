"""ctypes front end of the plain-C CPU oracle (q4_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg are the only users.  The product path never
imports this package, and this package never imports the product.

Buffers cross as numpy arrays.  Activation quantisations are in GGML's Q8_0
block layout ([T][K/32][34]: fp16 d, 32 int8); weights in GGML's Q4_0 block
layout ([N][K/32][18]: fp16 d, 16 nibble bytes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q4_oracle.c")
LIB = os.path.join(HERE, "liborc.so")

# Plain C11 (ISO mode: no FMA contraction), no fast-math, OpenMP over rows.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fopenmp", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(out: str = LIB, mutant: int = 0) -> str:
    """Compile the oracle (optionally one planted mutant) into a shared library."""
    cmd = ["gcc", *CFLAGS, f"-DORC_MUTANT={int(mutant)}", SRC, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build_mutant(mutant: int, workdir: str | None = None) -> str:
    d = workdir or tempfile.mkdtemp(prefix="orc_mut_")
    return build(os.path.join(d, f"liborc_m{mutant}.so"), mutant=mutant)


_u8p = ctypes.POINTER(ctypes.c_uint8)
_i8p = ctypes.POINTER(ctypes.c_int8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


class Oracle:
    """Thin numpy wrapper around one loaded oracle library."""

    def __init__(self, path: str = LIB):
        if not os.path.exists(path):
            if path == LIB:
                build()
            else:
                raise FileNotFoundError(path)
        self.path = path
        L = ctypes.CDLL(path)
        L.orc_half_to_float.argtypes = [ctypes.c_uint16]
        L.orc_half_to_float.restype = ctypes.c_float
        L.orc_float_to_half_rn.argtypes = [ctypes.c_float]
        L.orc_float_to_half_rn.restype = ctypes.c_uint16
        L.orc_quantize_block_q8_0.argtypes = [_f32p, _u16p, _i8p]
        L.orc_quantize_q8_0.argtypes = [_f32p, ctypes.c_int, ctypes.c_int64, _u8p]
        L.orc_block_isum.argtypes = [_u8p, _u8p]
        L.orc_block_isum.restype = ctypes.c_int32
        L.orc_block_isums.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p, ctypes.c_int, _i32p]
        L.orc_gemv_f64.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p, ctypes.c_int, _f64p, _f64p]
        L.orc_gemv_rows_f64.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p, ctypes.c_int,
                                        _i64p, ctypes.c_int64, _f64p, _f64p]
        L.orc_argmax_f32.argtypes = [_f32p, ctypes.c_int64]
        L.orc_argmax_f32.restype = ctypes.c_int64
        L.orc_argmax_f64.argtypes = [_f64p, ctypes.c_int64]
        L.orc_argmax_f64.restype = ctypes.c_int64
        L.orc_block_isum_q8.argtypes = [_u8p, _u8p]
        L.orc_block_isum_q8.restype = ctypes.c_int32
        L.orc_block_isums_q8.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p, ctypes.c_int, _i32p]
        L.orc_gemv_q8_f64.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p, ctypes.c_int, _f64p, _f64p]
        L.orc_exp_f32_n.argtypes = [_f32p, ctypes.c_int64, _f32p]
        L.orc_silu_f32_n.argtypes = [_f32p, ctypes.c_int64, _f32p]
        L.orc_silu_mul_quantize.argtypes = [_f32p, _f32p, ctypes.c_int, ctypes.c_int64, _u8p, _f32p]
        L.orc_top2_f32.argtypes = [_f32p, ctypes.c_int64, _i64p]
        L.orc_top2_f32.restype = None
        L.orc_top2_f64.argtypes = [_f64p, ctypes.c_int64, _i64p]
        L.orc_top2_f64.restype = None
        L.orc_verify_commit.argtypes = [_i64p, _i64p, ctypes.c_int]
        L.orc_quantize_block_q4_0.argtypes = [_f32p, _u8p]
        L.orc_quantize_vec_i8.argtypes = [_f32p, ctypes.c_int, ctypes.c_int64, _i8p, _f32p]
        L.orc_gemv_gs64_f64.argtypes = [_u8p, _f32p, ctypes.c_int64, ctypes.c_int64, _i8p, _f32p, ctypes.c_int,
                                        _f64p, _f64p]
        L.orc_gemv_ep_f64.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p, ctypes.c_int, _f32p, _f32p,
                                      _f64p, _f64p]
        L.orc_requant_f32_q4_0.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, _u8p]
        L.orc_requant_q8_0_q4_0.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
        L.orc_verify_commit.restype = ctypes.c_int
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_set_threads.restype = ctypes.c_int
        L.orc_mutant.restype = ctypes.c_int
        L.orc_range_violations.restype = ctypes.c_long
        self.L = L

    def set_threads(self, n: int) -> int:
        """Threads of the row loops (timing only; results do not depend on it)."""
        return int(self.L.orc_set_threads(int(n)))

    # -- binary16
    def half_to_float(self, h: int) -> float:
        return float(self.L.orc_half_to_float(int(h)))

    def float_to_half(self, f: float) -> int:
        return int(self.L.orc_float_to_half_rn(ctypes.c_float(f)))

    # -- Q8_0
    def quantize_block(self, x: np.ndarray):
        x = np.ascontiguousarray(x, dtype=np.float32)
        assert x.shape == (32,)
        d = np.zeros(1, np.uint16)
        q = np.zeros(32, np.int8)
        self.L.orc_quantize_block_q8_0(_p(x, _f32p), _p(d, _u16p), _p(q, _i8p))
        return int(d[0]), q

    def quantize(self, x: np.ndarray) -> np.ndarray:
        """x fp32 [T, K] -> uint8 [T, K/32, 34] (GGML Q8_0 blocks)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        T, K = x.shape
        out = np.empty((T, K // 32, 34), np.uint8)
        self.L.orc_quantize_q8_0(_p(x, _f32p), T, K, _p(out, _u8p))
        return out

    # -- block sums and GEMV
    def block_isum(self, wblk: np.ndarray, xblk: np.ndarray) -> int:
        wblk = np.ascontiguousarray(wblk, np.uint8)
        xblk = np.ascontiguousarray(xblk, np.uint8)
        return int(self.L.orc_block_isum(_p(wblk, _u8p), _p(xblk, _u8p)))

    def block_isums(self, W: np.ndarray, N: int, K: int, xq: np.ndarray, T: int) -> np.ndarray:
        W = np.ascontiguousarray(W, np.uint8)
        xq = np.ascontiguousarray(xq, np.uint8)
        out = np.empty((T, N, K // 32), np.int32)
        self.L.orc_block_isums(_p(W, _u8p), N, K, _p(xq, _u8p), T, _p(out, _i32p))
        return out

    def gemv(self, W: np.ndarray, N: int, K: int, xq: np.ndarray, T: int):
        """-> (y64 [T, N], S [T, N]) in fp64."""
        W = np.ascontiguousarray(W, np.uint8)
        xq = np.ascontiguousarray(xq, np.uint8)
        y = np.empty((T, N), np.float64)
        S = np.empty((T, N), np.float64)
        self.L.orc_gemv_f64(_p(W, _u8p), N, K, _p(xq, _u8p), T, _p(y, _f64p), _p(S, _f64p))
        return y, S

    def gemv_rows(self, W: np.ndarray, N: int, K: int, xq: np.ndarray, T: int, rows):
        W = np.ascontiguousarray(W, np.uint8)
        xq = np.ascontiguousarray(xq, np.uint8)
        rows = np.ascontiguousarray(rows, np.int64)
        y = np.empty((T, rows.size), np.float64)
        S = np.empty((T, rows.size), np.float64)
        self.L.orc_gemv_rows_f64(_p(W, _u8p), N, K, _p(xq, _u8p), T, _p(rows, _i64p), rows.size,
                                 _p(y, _f64p), _p(S, _f64p))
        return y, S

    # -- Q8_0 weights
    def block_isum_q8(self, wblk: np.ndarray, xblk: np.ndarray) -> int:
        wblk = np.ascontiguousarray(wblk, np.uint8)
        xblk = np.ascontiguousarray(xblk, np.uint8)
        return int(self.L.orc_block_isum_q8(_p(wblk, _u8p), _p(xblk, _u8p)))

    def block_isums_q8(self, W: np.ndarray, N: int, K: int, xq: np.ndarray, T: int) -> np.ndarray:
        W = np.ascontiguousarray(W, np.uint8)
        xq = np.ascontiguousarray(xq, np.uint8)
        out = np.empty((T, N, K // 32), np.int32)
        self.L.orc_block_isums_q8(_p(W, _u8p), N, K, _p(xq, _u8p), T, _p(out, _i32p))
        return out

    def gemv_q8(self, W: np.ndarray, N: int, K: int, xq: np.ndarray, T: int):
        """Q8_0 weights (GGML blocks [N][nb][34]) -> (y64 [T, N], S [T, N]) in fp64."""
        W = np.ascontiguousarray(W, np.uint8)
        xq = np.ascontiguousarray(xq, np.uint8)
        y = np.empty((T, N), np.float64)
        S = np.empty((T, N), np.float64)
        self.L.orc_gemv_q8_f64(_p(W, _u8p), N, K, _p(xq, _u8p), T, _p(y, _f64p), _p(S, _f64p))
        return y, S

    # -- FFN chain
    def exp_f32(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, np.float32)
        out = np.empty_like(x)
        self.L.orc_exp_f32_n(_p(x, _f32p), x.size, _p(out, _f32p))
        return out

    def silu_f32(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, np.float32)
        out = np.empty_like(x)
        self.L.orc_silu_f32_n(_p(x, _f32p), x.size, _p(out, _f32p))
        return out

    def silu_mul_quantize(self, g: np.ndarray, u: np.ndarray):
        """g, u fp32 [T, F] -> (Q8_0 blocks of SiLU(g) * u [T, F/32, 34], the fp32 h [T, F])."""
        g = np.ascontiguousarray(g, np.float32)
        u = np.ascontiguousarray(u, np.float32)
        T, F = g.shape
        hq = np.empty((T, F // 32, 34), np.uint8)
        h = np.empty((T, F), np.float32)
        self.L.orc_silu_mul_quantize(_p(g, _f32p), _p(u, _f32p), T, F, _p(hq, _u8p), _p(h, _f32p))
        return hq, h

    # -- argmax
    def argmax_f32(self, y: np.ndarray) -> int:
        y = np.ascontiguousarray(y, np.float32)
        return int(self.L.orc_argmax_f32(_p(y, _f32p), y.size))

    def argmax_f64(self, y: np.ndarray) -> int:
        y = np.ascontiguousarray(y, np.float64)
        return int(self.L.orc_argmax_f64(_p(y, _f64p), y.size))

    def top2_f32(self, y: np.ndarray):
        """(best, second) row indices of fp32 y (second = -1 when y has one row)."""
        y = np.ascontiguousarray(y, np.float32)
        out = np.empty(2, np.int64)
        self.L.orc_top2_f32(_p(y, _f32p), y.size, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
        return int(out[0]), int(out[1])

    def top2_f64(self, y: np.ndarray):
        y = np.ascontiguousarray(y, np.float64)
        out = np.empty(2, np.int64)
        self.L.orc_top2_f64(_p(y, _f64p), y.size, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
        return int(out[0]), int(out[1])

    def verify_commit(self, tokens, pred) -> int:
        """Committed predictions of one verify step (1..T)."""
        tk = np.ascontiguousarray(tokens, np.int64)
        pr = np.ascontiguousarray(pred, np.int64)
        assert tk.size == pr.size >= 1
        P = ctypes.POINTER(ctypes.c_int64)
        return int(self.L.orc_verify_commit(tk.ctypes.data_as(P), pr.ctypes.data_as(P), tk.size))

    def gemv_ep(self, W: np.ndarray, N: int, K: int, xq: np.ndarray, T: int, bias=None, res=None):
        """-> (y64, S) [T, N] of W.x + bias[N] + res[T, N] (either may be None)."""
        W = np.ascontiguousarray(W, np.uint8)
        xq = np.ascontiguousarray(xq, np.uint8)
        b = None if bias is None else np.ascontiguousarray(bias, np.float32).reshape(N)
        r = None if res is None else np.ascontiguousarray(res, np.float32).reshape(T, N)
        y = np.empty((T, N), np.float64)
        S = np.empty((T, N), np.float64)
        self.L.orc_gemv_ep_f64(_p(W, _u8p), N, K, _p(xq, _u8p), T, None if b is None else _p(b, _f32p),
                               None if r is None else _p(r, _f32p), _p(y, _f64p), _p(S, _f64p))
        return y, S

    def quantize_vec_i8(self, x: np.ndarray):
        """fp32 x [T, K] -> (q int8 [T, K], s fp32 [T]): one scale per vector."""
        x = np.ascontiguousarray(x, np.float32)
        T, K = x.shape
        q = np.empty((T, K), np.int8)
        s = np.empty(T, np.float32)
        self.L.orc_quantize_vec_i8(_p(x, _f32p), T, K, _p(q, _i8p), _p(s, _f32p))
        return q, s

    def gemv_gs64(self, Wq: np.ndarray, Ws: np.ndarray, N: int, K: int, q: np.ndarray, s: np.ndarray):
        """gs64 planar int4 weights (nibbles [N][K/64][32], fp32 scales [N][K/64])
        against per-vector int8 activations -> (y64, S) [T, N]."""
        Wq = np.ascontiguousarray(Wq, np.uint8)
        Ws = np.ascontiguousarray(Ws, np.float32)
        q = np.ascontiguousarray(q, np.int8)
        s = np.ascontiguousarray(s, np.float32)
        T = q.shape[0]
        y = np.empty((T, N), np.float64)
        S = np.empty((T, N), np.float64)
        self.L.orc_gemv_gs64_f64(_p(Wq, _u8p), _p(Ws, _f32p), N, K, _p(q, _i8p), _p(s, _f32p), T,
                                 _p(y, _f64p), _p(S, _f64p))
        return y, S

    def quantize_block_q4_0(self, x: np.ndarray) -> np.ndarray:
        """One block of 32 fp32 values -> its 18 Q4_0 bytes."""
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(32)
        out = np.empty(18, np.uint8)
        self.L.orc_quantize_block_q4_0(_p(x, _f32p), _p(out, _u8p))
        return out

    def requant_f32_q4_0(self, w: np.ndarray, N: int, K: int) -> np.ndarray:
        """fp32 w[N][K] -> GGML Q4_0 bytes [N][K/32 * 18]."""
        w = np.ascontiguousarray(w, dtype=np.float32).reshape(N, K)
        out = np.empty((N, K // 32 * 18), np.uint8)
        self.L.orc_requant_f32_q4_0(_p(w, _f32p), N, K, _p(out, _u8p))
        return out

    def requant_q8_0_q4_0(self, w: np.ndarray, N: int, K: int) -> np.ndarray:
        """GGML Q8_0 bytes [N][K/32 * 34] -> GGML Q4_0 bytes [N][K/32 * 18]."""
        w = np.ascontiguousarray(w, dtype=np.uint8).reshape(N, K // 32 * 34)
        out = np.empty((N, K // 32 * 18), np.uint8)
        self.L.orc_requant_q8_0_q4_0(_p(w, _u8p), N, K, _p(out, _u8p))
        return out

    def num_threads(self) -> int:
        return int(self.L.orc_num_threads())

    def mutant(self) -> int:
        return int(self.L.orc_mutant())

    def range_violations(self) -> int:
        return int(self.L.orc_range_violations())


# Acceptance bound on an fp32 output against the fp64 reference:
#   |y - y64| <= 1e-5 * S + 1e-6,  S = sum_b |d_w d_x isum|.
TOL_REL, TOL_ABS = 1e-5, 1e-6


def tolerance(S: np.ndarray) -> np.ndarray:
    return TOL_REL * S + TOL_ABS


_default: Oracle | None = None


def load() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default

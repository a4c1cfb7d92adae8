"""Helpers shared by the GPU parity tests: byte-format conversions between
the library's planar Q8_0 buffers and the oracle's GGML Q8_0 blocks, and
comparisons against the oracle's fp64 reference."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def planar_to_blocks(buf: np.ndarray, R: int, K: int) -> np.ndarray:
    """Planar Q8_0 bytes (R*K int8, then R*K/32 fp16, padding) -> [R][nb][34]."""
    nb = K // 32
    qs = buf[: R * K].reshape(R, nb, 32)
    d = buf[R * K: R * K + 2 * R * nb].reshape(R, nb, 2)
    return np.concatenate([d, qs], axis=2)


def blocks_to_planar(blocks: np.ndarray, xq_bytes: int) -> np.ndarray:
    R, nb, _ = blocks.shape
    out = np.zeros(xq_bytes, np.uint8)
    out[: R * nb * 32] = blocks[:, :, 2:].reshape(-1)
    out[R * nb * 32: R * nb * 32 + 2 * R * nb] = blocks[:, :, :2].reshape(-1)
    return out


def to_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1) if a.dtype == np.uint8 else np.ascontiguousarray(a)).to(dev)


def check_close(y_gpu: np.ndarray, y64: np.ndarray, S: np.ndarray, what: str = ""):
    """|y - y64| <= 1e-5 * S + 1e-6 element by element."""
    err = np.abs(y_gpu.astype(np.float64) - y64)
    tol = oracle.tolerance(S)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outputs outside the bound; "
                           f"worst excess {float(np.max(err - tol)):.3e}")
    return float(np.max(err / np.maximum(S, 1e-30)))

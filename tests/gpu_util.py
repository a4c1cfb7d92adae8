"""Helpers shared by the GPU parity tests: byte-format conversions between
the library's planar Q8_0 buffers and the oracle's GGML Q8_0 blocks, and
comparisons against the oracle's fp64 reference."""
from __future__ import annotations

import os

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


# Near ties of the fp64 reference.  The GPU's fp32 outputs may differ from
# y64 by up to the tolerance, so where two rows' y64 values are closer than
# the sum of their tolerances the GPU may rank them either way.  Such tokens
# are counted and reported, never passed silently: everywhere else the GPU's
# row must equal the fp64 reference's row exactly.  For lm_head-shaped rows
# (151936 outputs, gap of the top two about sigma / sqrt(2 ln N) against a
# tolerance near 3e-5) the expected rate is below 1e-3 per token; the bound
# asserted is ten times that, and at most one near tie in a test of fewer
# than 100 tokens.
NEAR_TIE_RATE_BOUND = 1e-2


def near_tie_bound(tokens: int) -> int:
    return max(1, int(NEAR_TIE_RATE_BOUND * tokens))


def _near_rows(y64_t: np.ndarray, S_t: np.ndarray, b: int, exclude=()) -> np.ndarray:
    """Rows r != b whose y64 lies within tol(r) + tol(b) of row b's."""
    tol = oracle.tolerance(S_t)
    near = np.abs(y64_t - y64_t[b]) <= tol + tol[b]
    near[b] = False
    for e in exclude:
        near[e] = False
    return np.nonzero(near)[0]


def rank_vs_fp64(got_rows: np.ndarray, ref_rows: np.ndarray, y64: np.ndarray, S: np.ndarray, what: str,
                 log: bool = True) -> int:
    """got_rows, ref_rows: [T][k] rows ranked 0..k-1 by the GPU and by the
    fp64 reference.  A (token, rank) is a near tie when another row lies
    within the summed tolerances of the reference's row; there the GPU's
    row may be any such row, elsewhere it must be the reference's row.
    Returns the number of tokens with a near tie (and reports it)."""
    got_rows = np.asarray(got_rows).reshape(y64.shape[0], -1)
    ref_rows = np.asarray(ref_rows).reshape(y64.shape[0], -1)
    ties = 0
    for t in range(y64.shape[0]):
        tok_tie = False
        for k in range(got_rows.shape[1]):
            a, b = int(got_rows[t, k]), int(ref_rows[t, k])
            if b < 0:                      # no such rank (one row)
                assert a == b, (what, t, k)
                continue
            near = _near_rows(y64[t], S[t], b)
            if near.size == 0:
                assert a == b, f"{what}: token {t} rank {k}: row {a} against the fp64 row {b} with no near tie"
            else:
                tok_tie = True
                assert a == b or a in set(near.tolist()), (
                    f"{what}: token {t} rank {k}: row {a} is not within tolerance of the fp64 row {b}")
        ties += int(tok_tie)
    if log:
        report_near_ties(what, ties, y64.shape[0])
    return ties


def report_near_ties(what: str, ties: int, tokens: int):
    line = f"NEAR-TIES {what}: {ties} of {tokens} tokens"
    print(line)
    path = os.environ.get("QGEMV_NEAR_TIE_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")
    assert ties <= near_tie_bound(tokens), f"{line}: above the bound {near_tie_bound(tokens)}"

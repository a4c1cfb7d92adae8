"""Requantisation of fp32 and Q8_0 weights to Q4_0 through the C ABI against
the CPU oracle: every output byte bit-exact (the codes are integer decisions
taken in fp32 on both sides, with the same rounded operations).  Then the
requantised lm_head feeds the packed GEMV, whose output equals the GEMV of
the oracle's blocks and stays within the bound of the oracle's fp64 GEMV.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def orc():
    from quantized_q4_weight_gb300 import _build
    _build.build()
    oracle.build()
    q.lib()
    torch.cuda.init()
    return oracle.load()


def edge_rows(K: int) -> np.ndarray:
    """Rows of hand-placed blocks: ties of the extreme in both orders, zero
    and negative-zero blocks, exact half steps, fp32 subnormals, a scale
    beyond fp16's range, a lone non-zero, and a constant block."""
    nb = K // 32
    rows = np.zeros((8, K), np.float32)
    rows[0, 3], rows[0, 9] = 8.0, -8.0                    # tie, the positive first
    rows[0, 32 + 3], rows[0, 32 + 9] = -8.0, 8.0          # tie, the negative first
    rows[1, :32] = -0.0                                   # negative zeros
    half = np.array([0.5, 1.5, -2.5, 7.5, -7.5, 3.5, -0.5, 6.5], np.float32)
    rows[2, :32] = np.resize(half, 32)
    rows[2, 0] = -8.0                                     # d = 1: x + 8.5 lands on integers
    rows[3, :32] = np.float32(1e-40) * np.arange(-16, 16, dtype=np.float32)
    rows[4, :32] = np.linspace(-1e6, 2e5, 32, dtype=np.float32)   # d = 1.25e5 overflows fp16
    rows[5, 17] = -3.0
    rows[6, :32] = 0.25
    rows[7] = np.tile(np.linspace(-1, 1, 32, dtype=np.float32), nb)
    return rows


@pytest.mark.parametrize("N,K", [(1, 32), (37, 288), (8, 1536), (1536, 8960), (2048, 11008)])
def test_requant_f32_bit_exact(orc, N, K):
    w = synth.f32_weights(900 + N + K, N, K)
    if N >= 8:
        w[:8] = edge_rows(K)
    got = q.requant_f32_q4_0(torch.from_numpy(w).to(DEV), N, K).cpu().numpy()
    ref = orc.requant_f32_q4_0(w, N, K)
    assert np.array_equal(got, ref.reshape(-1)), int(np.argmax(got != ref.reshape(-1)))
    assert q.device_status() == 0


@pytest.mark.parametrize("N,K", [(1, 32), (50, 2080), (151936, 1536)])
def test_requant_q8_0_bit_exact(orc, N, K):
    """Q8_0 -> Q4_0 at the lm_head's full size (minfer README M14)."""
    w8 = synth.q8_0_weights(950 + N, N, K)
    if N >= 4:
        blk = w8.reshape(N, K // 32, 34)
        blk[0, 0, 2:] = 0                                         # zero codes
        blk[1, 0, 2:] = np.int8(-127).view(np.uint8)              # the int8 extreme, every element
        blk[2, 0, 2:4] = np.array([127, -127], np.int8).view(np.uint8)   # a tie of magnitudes
        blk[3, 0, 0:2] = np.array([np.float16(-0.0)]).view(np.uint8)     # negative zero scale
    got = q.requant_q8_0_q4_0(to_dev(w8), N, K).cpu().numpy()
    ref = orc.requant_q8_0_q4_0(w8, N, K)
    assert np.array_equal(got, ref.reshape(-1))
    assert q.device_status() == 0


def test_requantised_head_feeds_the_gemv(orc):
    """Q8_0 lm_head -> Q4_0 -> packed GEMV with argmax, at 151936 x 1536."""
    N, K, T = 151936, 1536, 2
    w8 = synth.q8_0_weights(960, N, K)
    w4 = q.requant_q8_0_q4_0(to_dev(w8), N, K)
    ref4 = orc.requant_q8_0_q4_0(w8, N, K)
    Wp = q.pack_q4_0(w4, N, K)
    x = synth.activations(961, T, K)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), T, K)
    ws = q.new_workspace(q.workspace_bytes(N, K, T))
    y = torch.empty((T, N), dtype=torch.float32, device=DEV)
    idx = q.gemv_argmax(Wp, q.W_PACKED, xq, N, K, T, ws, y=y).cpu().numpy()
    yref = q.gemv(q.pack_q4_0(to_dev(ref4.reshape(-1)), N, K), q.W_PACKED, xq, N, K, T,
                  q.new_workspace(q.workspace_bytes(N, K, T))).cpu()
    assert torch.equal(y.cpu().view(torch.int32), yref.view(torch.int32))
    rows = np.unique(np.concatenate([idx, np.random.default_rng(962).integers(0, N, 64)]))
    y64, S = orc.gemv_rows(ref4, N, K, orc.quantize(x), T, rows)
    err = np.abs(y.cpu().numpy()[:, rows].astype(np.float64) - y64)
    assert np.all(err <= oracle.tolerance(S))
    for t in range(T):
        assert idx[t] == orc.argmax_f32(y.cpu().numpy()[t])
    assert q.device_status() == 0


def test_requant_f32_unaligned_source(orc):
    """A 4-byte (not 16-byte) aligned fp32 source takes scalar loads; the
    bytes are the same."""
    N, K = 300, 1536
    w = synth.f32_weights(970, N, K)
    buf = torch.zeros(N * K + 4, dtype=torch.float32, device=DEV)
    buf[1:1 + N * K] = torch.from_numpy(w.reshape(-1)).to(DEV)
    view = buf[1:1 + N * K]
    assert view.data_ptr() % 16 == 4
    got = q.requant_f32_q4_0(view, N, K).cpu().numpy()
    assert np.array_equal(got, orc.requant_f32_q4_0(w, N, K).reshape(-1))
    assert q.device_status() == 0

"""Q8_0-weight GEMV through the C ABI against the CPU oracle.

Bit-exact: the packed layout (against a layout written out here from its
definition), pack/unpack round trips, outputs across T, and outputs of
identical rows whether their slab is split over warps or not.  Closed forms
are exact.  Every output is within |y - y64| <= 1e-5 * S + 1e-6.
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


def expected_packed(Wg, N, K):
    """The device layout from its definition: 16-row slabs of 8-block stages;
    a full stage holds [16 rows][16 chunks of 16 code bytes], chunk c of row r
    at position c ^ (r & 7), then fp16 scales [16 rows][2 parities][4]; a
    partial stage [16][nbs][32] codes then [16][nbs] scales; tail rows as is."""
    nb = K // 32
    blk = Wg.reshape(N, nb, 34)
    out = np.empty(N * nb * 34, np.uint8)
    nslabs = N // 16
    pos = 0
    for s in range(nslabs):
        for st in range(0, nb, 8):
            nbs = min(8, nb - st)
            rows = blk[16 * s:16 * s + 16, st:st + nbs]
            if nbs == 8:
                codes = np.empty((16, 16, 16), np.uint8)
                for r in range(16):
                    chunks = rows[r, :, 2:].reshape(16, 16)          # chunk c = 2 * block + half
                    for c in range(16):
                        codes[r, c ^ (r & 7)] = chunks[c]
                scales = np.empty((16, 2, 4, 2), np.uint8)
                for r in range(16):
                    for b in range(8):
                        scales[r, b & 1, b >> 1] = rows[r, b, :2]
                part = np.concatenate([codes.reshape(-1), scales.reshape(-1)])
            else:
                part = np.concatenate([rows[:, :, 2:].reshape(-1), rows[:, :, :2].reshape(-1)])
            out[pos:pos + part.size] = part
            pos += part.size
    out[pos:] = blk[16 * nslabs:].reshape(-1)
    assert pos + blk[16 * nslabs:].size == out.size
    return out


def run(orc, seed, N, K, T, W_ggml=None):
    Wg = W_ggml if W_ggml is not None else synth.q8_0_weights(seed, N, K)
    Wp = q.pack_q8_0(to_dev(Wg), N, K)
    x = synth.activations(seed + 1, T, K)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), T, K)
    ws = q.new_workspace(q.q8_0_workspace_bytes(N, K, T))
    y = q.gemv_q8_0(Wp, xq, N, K, T, ws).cpu().numpy()
    return Wg, Wp, x, xq, ws, y


@pytest.mark.parametrize("N,K", [(16, 256), (37, 288), (48, 8960), (5, 64)])
def test_pack_layout_and_round_trip(N, K):
    Wg = synth.q8_0_weights(90 + N, N, K)
    Wp = q.pack_q8_0(to_dev(Wg), N, K)
    assert np.array_equal(Wp.cpu().numpy(), expected_packed(Wg, N, K))
    assert np.array_equal(q.unpack_q8_0(Wp, N, K).cpu().numpy(), Wg.reshape(-1))


# one and few rows, a tail of N % 16 rows, partial stages (K % 256 != 0),
# slabs split over warps (few slabs) and not (many), T = 1..8
SHAPES = [(1, 32, 1), (16, 256, 1), (17, 288, 2), (1536, 1536, 1), (2048, 11008, 8), (4000, 544, 5),
          (50, 8960, 3), (40000, 1536, 1), (3000, 2048, 7), (151, 4096, 4), (9000, 1536, 6)]


@pytest.mark.parametrize("N,K,T", SHAPES)
def test_q8_gemv_within_bound(orc, N, K, T):
    Wg, Wp, x, xq, ws, y = run(orc, 1000 + N + K + T, N, K, T)
    y64, S = orc.gemv_q8(Wg, N, K, orc.quantize(x), T)
    err = np.abs(y.astype(np.float64) - y64)
    bound = oracle.tolerance(S)
    assert np.all(err <= bound), f"worst excess {np.max(err - bound)}"
    assert q.device_status() == 0
    # the workspace counters are left at zero: a second call gives the same bits
    y2 = q.gemv_q8_0(Wp, xq, N, K, T, ws).cpu().numpy()
    assert np.array_equal(y.view(np.int32), y2.view(np.int32))


@pytest.mark.parametrize("N,K", [(1536, 1536), (2048, 8960), (37, 288)])
def test_q8_bit_identical_across_T(orc, N, K):
    Wg = synth.q8_0_weights(500 + N, N, K)
    Wp = q.pack_q8_0(to_dev(Wg), N, K)
    x = synth.activations(501 + N, 8, K)
    xd = torch.from_numpy(x).to(DEV)
    xq8 = q.quantize_q8_0(xd, 8, K)
    ws = q.new_workspace(q.q8_0_workspace_bytes(N, K, 8))
    y8 = q.gemv_q8_0(Wp, xq8, N, K, 8, ws).cpu()
    for t in (0, 3, 7):
        xq1 = q.quantize_q8_0(xd[t:t + 1].contiguous(), 1, K)
        y1 = q.gemv_q8_0(Wp, xq1, N, K, 1, q.new_workspace(q.q8_0_workspace_bytes(N, K, 1))).cpu()
        assert torch.equal(y1[0].view(torch.int32), y8[t].view(torch.int32))


def test_q8_split_and_unsplit_slabs_agree(orc):
    """The same 16 rows give the same bits when their slab is shared by
    several warps (few slabs) and when one warp takes it (many slabs)."""
    K = 4096
    W16 = synth.q8_0_weights(610, 16, K)
    few = run(orc, 611, 16, K, 2, W_ggml=W16)
    many_W = np.tile(W16, (6000, 1))                      # 96000 rows: 6000 identical slabs
    N = many_W.shape[0]
    Wp = q.pack_q8_0(to_dev(many_W), N, K)
    ws = q.new_workspace(q.q8_0_workspace_bytes(N, K, 2))
    y = q.gemv_q8_0(Wp, few[3], N, K, 2, ws).cpu().numpy()
    assert q.q8_0_workspace_bytes(16, K, 2) > 0 and q.q8_0_workspace_bytes(N, K, 2) == 0
    for s in (0, 2999, 5999):
        assert np.array_equal(y[:, 16 * s:16 * s + 16].view(np.int32), few[5].view(np.int32))


def test_q8_closed_forms(orc):
    K, N, T = 1536, 64, 1
    nb = K // 32
    for c in (-128, -127, -1, 0, 1, 127):
        blk = np.zeros((N, nb, 34), np.uint8)
        blk[:, :, 0:2] = np.array([0x00, 0x3C], np.uint8)            # d_w = 1
        blk[:, :, 2:] = np.int8(c).view(np.uint8)
        x = np.full((T, K), 127.0, np.float32)                          # q = 127, d_x = 1
        Wp = q.pack_q8_0(to_dev(blk.reshape(N, -1)), N, K)
        xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), T, K)
        y = q.gemv_q8_0(Wp, xq, N, K, T, q.new_workspace(q.q8_0_workspace_bytes(N, K, T))).cpu().numpy()
        assert np.all(y == np.float32(nb * 32 * 127 * c))


def test_q8_errors():
    N, K, T = 64, 32768, 8                                              # activations beyond shared memory
    W = torch.zeros(q.q8_0_bytes(N, K), dtype=torch.uint8, device=DEV)
    xq = torch.zeros(q.xq_bytes(T, K), dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QgemvError, match="UNSUPPORTED"):
        q.gemv_q8_0(W, xq, N, K, T, q.new_workspace(1 << 20))
    N, K, T = 32, 1536, 1                                               # few slabs: needs a workspace
    assert q.q8_0_workspace_bytes(N, K, T) > 0
    W = torch.zeros(q.q8_0_bytes(N, K), dtype=torch.uint8, device=DEV)
    xq = torch.zeros(q.xq_bytes(T, K), dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QgemvError, match="WORKSPACE"):
        q.gemv_q8_0(W, xq, N, K, T, None)
    with pytest.raises(q.QgemvError, match="INVALID_ARG"):
        q.gemv_q8_0(W, xq, N, 33, T, None)
    assert q.device_status() == 0

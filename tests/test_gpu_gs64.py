"""The grouped int4 (gs64) GEMV with per-vector int8 activations against the
CPU oracle, through the C ABI (colibri qwen36 docs: the gs64 container's
planar groups, one fp32 scale per 64 weights; the dense int8 IDOT
activation contract, one scale amax / 127 per vector).

Bit-exact: the activation codes and scales, the packed layout (against its
definition written out here), pack / unpack round trips, and y across T.
Within |y - y64| <= 1e-5 * S + 1e-6: every output against the fp64
reference, at expert shapes (512 x 2048, 2048 x 512) and dense ones, with
ragged row tails, partial stages and split-K.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests.gpu_util import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def orc():
    from quantized_q4_weight_gb300 import _build
    _build.build()
    oracle.build()
    return oracle.load()


def packed(seed, N, K):
    wq, ws = synth.gs64_weights(seed, N, K)
    W = q.pack_gs64(torch.from_numpy(wq).to(DEV), torch.from_numpy(ws).to(DEV), N, K)
    return wq, ws, W


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("R,K", [(1, 64), (1, 2048), (3, 512), (8, 11008), (5, 8960), (2, 1000)])
def test_quantize_vec_i8_bit_exact(orc, R, K):
    x = synth.activations(300 + R + K, R, K)
    x[0, K // 2] = -40.0 * (1 + R)                      # the extreme inside the row
    qd, sd = q.quantize_vec_i8(torch.from_numpy(x).to(DEV), R, K)
    qr, sr = orc.quantize_vec_i8(x)
    assert np.array_equal(qd.cpu().numpy(), qr)
    assert np.array_equal(sd.cpu().numpy().view(np.int32), sr.view(np.int32))


def test_quantize_vec_i8_edges(orc):
    K = 256
    x = np.zeros((4, K), np.float32)
    x[1] = 1e-30                                        # tiny amax
    x[2, :5] = [127.0, 2.5, -2.5, 0.5, -0.5]           # s = 1: exact halves round away from zero
    x[3, 7] = 3.0e38
    qd, sd = q.quantize_vec_i8(torch.from_numpy(x).to(DEV), 4, K)
    qr, sr = orc.quantize_vec_i8(x)
    assert np.array_equal(qd.cpu().numpy(), qr) and np.array_equal(sd.cpu().numpy().view(np.int32), sr.view(np.int32))
    assert sr[0] == 0 and not qr[0].any()
    assert list(qr[2, :5]) == [127, 3, -3, 1, -1]


# ----------------------------------------------------------------- pack

@pytest.mark.parametrize("N,K", [(1, 64), (16, 512), (17, 576), (35, 1024), (48, 64 * 19)])
def test_pack_layout_and_roundtrip(orc, N, K):
    wq, ws, W = packed(N * K + 1, N, K)
    assert W.numel() == q.gs64_bytes(N, K) == 36 * N * K // 64
    uq, us = q.unpack_gs64(W, N, K)
    assert np.array_equal(uq.cpu().numpy(), wq) and np.array_equal(us.cpu().numpy().view(np.int32), ws.view(np.int32))
    # the layout as include/qgemv.h states it
    got = W.cpu().numpy()
    ng = K // 64
    nfull = N // 16
    slab = 16 * ng * 36
    for s in range(nfull):
        for st in range((ng + 7) // 8):
            ngs = min(8, ng - 8 * st)
            base = s * slab + st * 4608
            for r in range(16):
                for gs in range(ngs):
                    g = 8 * st + gs
                    if ngs == 8:
                        for k in range(2):
                            c = 2 * gs + k
                            o = base + r * 256 + 16 * (c ^ (r & 7))
                            assert np.array_equal(got[o:o + 16], wq[16 * s + r, g, 16 * k:16 * k + 16])
                        so = base + 4096 + (r * 2 + (gs & 1)) * 16 + (gs >> 1) * 4
                    else:
                        o = base + (r * ngs + gs) * 32
                        assert np.array_equal(got[o:o + 32], wq[16 * s + r, g])
                        so = base + 16 * ngs * 32 + (r * ngs + gs) * 4
                    assert got[so:so + 4].view(np.float32)[0] == ws[16 * s + r, g]
    for t in range(N - 16 * nfull):
        tb = nfull * slab + t * ng * 36
        assert np.array_equal(got[tb:tb + 32 * ng], wq[16 * nfull + t].reshape(-1))
        assert np.array_equal(got[tb + 32 * ng:tb + 36 * ng].view(np.float32), ws[16 * nfull + t])


# ----------------------------------------------------------------- GEMV

# expert (512 x 2048 gate/up, 2048 x 512 down), dense, ragged tails (N % 16),
# partial stages (K / 64 % 8 != 0), few slabs (split-K) and many
SHAPES = [(512, 2048), (2048, 512), (2048, 2048), (1536, 8960), (17, 576), (1, 64), (300, 1024), (33, 11008),
          (4099, 1536)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_gs64_matches_oracle(orc, N, K, T):
    wq, ws, W = packed(7 * N + K, N, K)
    x = synth.activations(3 * N + K + T, T, K)
    qd, sd = q.quantize_vec_i8(torch.from_numpy(x).to(DEV), T, K)
    wsp = q.new_workspace(q.gs64_workspace_bytes(N, K, T))
    y = q.gemv_gs64(W, qd, sd, N, K, T, wsp)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    qr, sr = orc.quantize_vec_i8(x)
    y64, S = orc.gemv_gs64(wq, ws, N, K, qr, sr)
    check_close(y.cpu().numpy(), y64, S, f"gs64 N={N} K={K} T={T}")


@pytest.mark.parametrize("N,K", [(2048, 512), (48, 8960), (4099, 1536)])
def test_gs64_bit_identical_across_T(orc, N, K):
    wq, ws, W = packed(11 * N + K, N, K)
    x = synth.activations(5 * N, 8, K)
    xd = torch.from_numpy(x).to(DEV)
    q8, s8 = q.quantize_vec_i8(xd, 8, K)
    y8 = q.gemv_gs64(W, q8, s8, N, K, 8, q.new_workspace(q.gs64_workspace_bytes(N, K, 8))).cpu()
    for t in range(8):
        q1, s1 = q.quantize_vec_i8(xd[t:t + 1].contiguous(), 1, K)
        y1 = q.gemv_gs64(W, q1, s1, N, K, 1, q.new_workspace(q.gs64_workspace_bytes(N, K, 1))).cpu()
        assert torch.equal(y1[0].view(torch.int32), y8[t].view(torch.int32)), t


@pytest.mark.parametrize("N,K", [(512, 2048), (2048, 512), (17, 576), (33, 11008), (4099, 1536), (1, 64)])
@pytest.mark.parametrize("T", [1, 3, 8])
@pytest.mark.parametrize("shift", [0, 1])
def test_gs64_f32_matches_two_launches(orc, N, K, T, shift):
    """fp32 activations quantised inside the GEMV launch: y bit-identical to
    the quantiser launch followed by the GEMV, and within the bound of the
    oracle; shift = 1 puts x at a 4-byte (not 16-byte) boundary."""
    wq, ws, W = packed(13 * N + K, N, K)
    x = synth.activations(17 * N + K + T, T, K)
    x[T - 1, K // 3] = -55.0                            # an extreme inside the last row
    buf = torch.zeros(T * K + 4, dtype=torch.float32, device=DEV)
    xd = buf[shift:shift + T * K].view(T, K)
    xd.copy_(torch.from_numpy(x))
    wsp = q.new_workspace(q.gs64_workspace_bytes(N, K, T))
    qd, sd = q.quantize_vec_i8(xd, T, K)
    y2 = q.gemv_gs64(W, qd, sd, N, K, T, wsp)
    y1 = q.gemv_gs64_f32(W, xd, N, K, T, wsp)
    y1b = q.gemv_gs64_f32(W, xd, N, K, T, wsp)          # the workspace left reusable
    torch.cuda.synchronize()
    assert q.device_status() == 0
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert torch.equal(y1b.view(torch.int32), y2.view(torch.int32))
    qr, sr = orc.quantize_vec_i8(x)
    y64, S = orc.gemv_gs64(wq, ws, N, K, qr, sr)
    check_close(y1.cpu().numpy(), y64, S, f"gs64 f32 N={N} K={K} T={T}")


def test_gs64_f32_edge_rows(orc):
    # a zero row (s = 0, all codes 0), a tiny one, exact halves, a huge value
    N, K = 40, 256
    wq, ws, W = packed(99, N, K)
    x = np.zeros((4, K), np.float32)
    x[1] = 1e-30
    x[2, :5] = [127.0, 2.5, -2.5, 0.5, -0.5]
    x[3, 7] = 3.0e38
    xd = torch.from_numpy(x).to(DEV)
    qd, sd = q.quantize_vec_i8(xd, 4, K)
    y2 = q.gemv_gs64(W, qd, sd, N, K, 4)
    y1 = q.gemv_gs64_f32(W, xd, N, K, 4)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert not y1[0].any()
    y64, S = orc.gemv_gs64(wq, ws, N, K, *orc.quantize_vec_i8(x))
    check_close(y1.cpu().numpy(), y64, S, "gs64 f32 edge rows")


def test_gs64_closed_forms(orc):
    # every nibble c, every scale s, every code q = 127 (x constant, s_x = x / 127):
    # y = s_x * (K / 64) * s * 64 * (c - 8) * 127, exact here
    N, K = 20, 1024
    for c in (0, 8, 15):
        wq = np.full((N, K // 64, 32), c * 0x11, np.uint8)
        ws = np.full((N, K // 64), 0.5, np.float32)
        W = q.pack_gs64(torch.from_numpy(wq).to(DEV), torch.from_numpy(ws).to(DEV), N, K)
        x = np.full((1, K), 127.0, np.float32)
        qd, sd = q.quantize_vec_i8(torch.from_numpy(x).to(DEV), 1, K)
        y = q.gemv_gs64(W, qd, sd, N, K, 1, q.new_workspace(q.gs64_workspace_bytes(N, K, 1))).cpu().numpy()
        want = np.float32(1.0) * (K // 64) * 0.5 * 64 * (c - 8) * 127
        assert np.all(y == want), (c, y[0, 0], want)
        y64, _ = orc.gemv_gs64(wq, ws, N, K, *orc.quantize_vec_i8(x))
        assert np.all(y64 == want)


def test_gs64_errors():
    N, K, T = 64, 512, 1
    W = torch.zeros(q.gs64_bytes(N, K), dtype=torch.uint8, device=DEV)
    qd = torch.zeros((T, K), dtype=torch.int8, device=DEV)
    sd = torch.zeros(T, dtype=torch.float32, device=DEV)
    with pytest.raises(q.QgemvError, match="INVALID_ARG"):
        q.gemv_gs64(W, qd, sd, N, 96, T)                  # K % 64 != 0
    with pytest.raises(q.QgemvError, match="UNSUPPORTED"):
        big = 1 << 19                                      # codes beyond shared memory
        q.gemv_gs64(torch.zeros(q.gs64_bytes(16, big), dtype=torch.uint8, device=DEV),
                    torch.zeros((8, big), dtype=torch.int8, device=DEV), torch.zeros(8, device=DEV), 16, big, 8)
    buf = torch.zeros(T * N + T * K, dtype=torch.float32, device=DEV)
    with pytest.raises(q.QgemvError, match="INVALID_ARG"):         # y over x
        q.gemv_gs64_f32(W, buf[:T * K].view(T, K), N, K, T, y=buf[8:8 + T * N].view(T, N))
    assert q.device_status() == 0

"""Sequences with the output epilogue y = W.x + bias + residual through the
C ABI.  Bit-exact: against the plain sequence's y followed by the two fp32
adds (torch's elementwise adds, IEEE round to nearest), on the balanced path
(long lists, small groups at T >= 5), the split-K path (short lists), fp32
and Q8_0 inputs, and a residual that is y itself.  Within the bound: against
the oracle's fp64 W.x + bias + residual."""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

DEV = "cuda"

LONG = [(2048, 2048), (256, 2048), (2048, 11008), (1536, 8960)] * 6   # 2208 slabs: balanced mode
SHORT = [(256, 1536), (40, 544), (17, 96)]


@pytest.fixture(scope="module")
def orc():
    from quantized_q4_weight_gb300 import _build
    _build.build()
    oracle.build()
    q.lib()
    torch.cuda.init()
    return oracle.load()


def build(shapes, T, seed):
    rng = np.random.default_rng(seed)
    items = []
    for i, (N, K) in enumerate(shapes):
        Wg = synth.q4_0_weights(seed + i, N, K)
        W = q.pack_q4_0(to_dev(Wg), N, K)
        x = synth.activations(seed + 100 + i, T, K)
        bias = rng.standard_normal(N).astype(np.float32) * 4 if i % 3 != 1 else None
        res = rng.standard_normal((T, N)).astype(np.float32) if i % 3 != 2 else None
        items.append(dict(N=N, K=K, Wg=Wg, W=W, x=x, bias=bias, res=res, inplace=(i % 4 == 0 and res is not None)))
    return items


@pytest.mark.parametrize("shapes", [LONG, SHORT], ids=["long", "short"])
@pytest.mark.parametrize("T", [1, 5, 8])
@pytest.mark.parametrize("x_f32", [False, True], ids=["q8", "f32"])
def test_seq_epilogue(orc, shapes, T, x_f32):
    its = build(shapes, T, 5000 + T + len(shapes))
    xs, ys, ys_plain, bs, rs, ep = [], [], [], [], [], []
    for it in its:
        xd = torch.from_numpy(it["x"]).to(DEV)
        xs.append(xd if x_f32 else q.quantize_q8_0(xd, T, it["K"]))
        ys_plain.append(torch.empty((T, it["N"]), dtype=torch.float32, device=DEV))
        b = None if it["bias"] is None else torch.from_numpy(it["bias"]).to(DEV)
        r = None if it["res"] is None else torch.from_numpy(it["res"]).to(DEV)
        y = r.clone() if it["inplace"] else torch.full((T, it["N"]), float("nan"), device=DEV)
        bs.append(b)
        rs.append(r)
        ys.append(y)
        ep.append((it["W"], xs[-1], y, it["N"], it["K"], b, y if it["inplace"] else r))
    plain = [(it["W"], xs[i], ys_plain[i], it["N"], it["K"]) for i, it in enumerate(its)]
    if x_f32:
        pi = q.seq_f32_items(plain)
        q.gemv_seq_f32(pi, q.W_PACKED, T, q.new_workspace(q.seq_f32_workspace_bytes(pi, T)))
    else:
        pi = q.seq_items(plain)
        q.gemv_seq(pi, q.W_PACKED, T, q.new_workspace(q.seq_workspace_bytes(pi, T)))
    items = q.seq_ep_items(ep)
    q.gemv_seq_ep(items, q.W_PACKED, T, q.new_workspace(q.seq_ep_workspace_bytes(items, T, x_f32)), x_f32=x_f32)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    for i, it in enumerate(its):
        want = ys_plain[i]
        if bs[i] is not None:
            want = want + bs[i][None, :]
        if rs[i] is not None:
            want = want + rs[i]
        assert torch.equal(ys[i].view(torch.int32), want.view(torch.int32)), (i, it["N"], it["K"])
        y64, S = orc.gemv_ep(it["Wg"], it["N"], it["K"], orc.quantize(it["x"]), T, it["bias"], it["res"])
        err = np.abs(ys[i].cpu().numpy().astype(np.float64) - y64)
        assert np.all(err <= oracle.tolerance(S)), (i, float(np.max(err - oracle.tolerance(S))))


def test_seq_epilogue_errors():
    N, K, T = 64, 256, 2
    W = torch.zeros(q.q4_0_bytes(N, K), dtype=torch.uint8, device=DEV)
    xq = torch.zeros(q.xq_bytes(T, K), dtype=torch.uint8, device=DEV)
    # y and its shifted residual are slices of one buffer, so that even an
    # accepted call would stay inside an allocation
    yy = torch.zeros(T * N + 1, device=DEV)
    y = yy[:T * N].view(T, N)
    y2 = torch.zeros((T, N), device=DEV)
    buf = torch.zeros(4 * N + 4, device=DEV)
    ws = q.new_workspace(1 << 20)
    L = q.lib()

    def call(items, x_f32=0):
        return L.qgemv_q4_0_seq_ep(items, len(items), q.W_PACKED, T, x_f32, q._ptr(ws), ws.numel(), None)

    ok = q.seq_ep_items([(W, xq, y, N, K, None, None)])
    assert call(ok, 2) == 1                                               # x_f32 must be 0 or 1
    bad_b = q.seq_ep_items([(W, xq, y, N, K, buf[1:1 + N], None)])
    bad_b[0].bias = buf.data_ptr() + 2                                    # misaligned bias
    assert call(bad_b) == 2
    part = q.seq_ep_items([(W, xq, y, N, K, None, y)])
    part[0].residual = yy.data_ptr() + 4                                  # residual shifted over y
    assert call(part) == 1
    other = q.seq_ep_items([(W, xq, y, N, K, None, y2), (W, xq, y2, N, K, None, None)])
    assert call(other) == 1                                               # residual over another output
    assert q.device_status() == 0

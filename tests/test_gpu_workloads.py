"""The benchmark's workloads at full size, in the launch configuration that
bench.py times, checked against the CPU oracle: every output where the
oracle finishes in seconds, sampled rows of every GEMV otherwise."""
import numpy as np
import pytest
import torch

import bench
import oracle
import quantized_q4_weight_gb300 as q
from tests.gpu_util import check_close, rank_vs_fp64, report_near_ties

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def orc():
    from quantized_q4_weight_gb300 import _build
    _build.build()
    oracle.build()
    return oracle.load()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("name,T", [("qwen2.5-1.5b_layerset", 1), ("qwen2.5-3b_verify", 8),
                                    ("qwen2.5-3b_verify", 5), ("qwen2.5-3b_verify", 4),
                                    ("qwen2.5-3b_verify", 2), ("qwen2.5-3b_verify", 1)])
def test_layer_sets_sampled(orc, name, T):
    wl = bench.build_workload(name, DEV, T=T, keep_host=True)
    wl.step()                                   # fp32 inputs, one quantiser + one GEMV launch
    torch.cuda.synchronize()
    assert q.device_status() == 0
    y_step = [host(y).copy() for y in wl.y]
    wl.kernel()                                 # pre-quantised inputs, the GEMV launch alone
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for i, (nm, N, K) in enumerate(wl.mats):
        assert np.array_equal(y_step[i].view(np.int32), host(wl.y[i]).view(np.int32)), nm
        x = host(wl.x[i])
        xq = orc.quantize(x)
        if i < 5:   # activation bytes of the first layer, bit-exact
            got = host(wl.xq[i])
            assert np.array_equal(got[:T * K].reshape(T, K // 32, 32), xq[:, :, 2:])
            assert np.array_equal(got[T * K:T * K + 2 * T * (K // 32)].reshape(T, K // 32, 2), xq[:, :, :2])
        rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 6)]))
        y64, S = orc.gemv_rows(wl.host[i], N, K, xq, T, rows)
        check_close(y_step[i][:, rows], y64, S, f"{name} {nm}")


def test_layer_set_epilogue_full(orc):
    """The 28-layer set with its epilogues (qkv bias, o and down residuals) as
    bench.py times it: every GEMV's y equals the plain sequence's y plus the
    bias and the residual (torch's fp32 adds), and the first layer's outputs
    are within the bound of the oracle's fp64 W.x + bias + residual."""
    wl = bench.build_workload("qwen2.5-1.5b_layerset_ep", DEV, keep_host=True)
    wl.step()
    torch.cuda.synchronize()
    assert q.device_status() == 0
    y_ep = [host(y).copy() for y in wl.y]
    plain = q.seq_f32_items([(wl.W[i], wl.x[i], wl.y[i], N, K) for i, (_, N, K) in enumerate(wl.mats)])
    q.gemv_seq_f32(plain, q.W_PACKED, wl.T, q.new_workspace(q.seq_f32_workspace_bytes(plain, wl.T)))
    torch.cuda.synchronize()
    for i, (nm, N, K) in enumerate(wl.mats):
        want = wl.y[i]
        if wl.bias[i] is not None:
            want = want + wl.bias[i][None, :]
        if wl.res[i] is not None:
            want = want + wl.res[i]
        assert np.array_equal(y_ep[i].view(np.int32), host(want).view(np.int32)), nm
        if i < 5:
            b = None if wl.bias[i] is None else host(wl.bias[i])
            r = None if wl.res[i] is None else host(wl.res[i])
            y64, S = orc.gemv_ep(wl.host[i], N, K, orc.quantize(host(wl.x[i])), wl.T, b, r)
            check_close(y_ep[i], y64, S, f"epilogue {nm}")


def test_lm_head_argmax_full(orc):
    wl = bench.build_workload("lm_head_argmax", DEV, keep_host=True)
    y = torch.empty((wl.T, wl.N), dtype=torch.float32, device=DEV)
    ties = tokens = 0
    for c in range(len(wl.W)):
        wl.copy = c
        wl.step()
        idx = host(wl.idx).copy()
        q.gemv(wl.W[c], q.W_PACKED, wl.xqb, wl.N, wl.K, wl.T, wl.ws, y=y)
        yh = host(y)
        xq = orc.quantize(host(wl.x))
        y64, S = orc.gemv(wl.host[c], wl.N, wl.K, xq, wl.T)
        check_close(yh, y64, S, "lm_head")
        for t in range(wl.T):
            assert idx[t] == orc.argmax_f32(yh[t])
        ties += rank_vs_fp64(idx, [orc.argmax_f64(y64[t]) for t in range(wl.T)], y64, S, f"lm_head copy {c}",
                             log=False)
        tokens += wl.T
    report_near_ties("lm_head 151936 x 1536, every copy", ties, tokens)


def test_single_full(orc):
    wl = bench.build_workload("single_1536", DEV, keep_host=True)
    wl.step()
    torch.cuda.synchronize()
    xq = orc.quantize(host(wl.x))
    y64, S = orc.gemv(wl.host[0], wl.N, wl.K, xq, wl.T)
    check_close(host(wl.y), y64, S, "single")


def test_moe_full(orc):
    wl = bench.build_workload("moe_top8_shared", DEV, keep_host=True)
    wl.tok = 0
    wl.step()            # token 0, expert set 0
    torch.cuda.synchronize()
    assert q.device_status() == 0
    ids = host(wl.ids[0])
    xin = orc.quantize(host(wl.x_in))
    xdn = host(wl.x_dn)
    outs = [host(wl.yg), host(wl.yu), host(wl.yd)]
    shapes = [(512, 2048), (512, 2048), (2048, 512)]
    for m, (N, K) in enumerate(shapes):
        for s, e in enumerate(ids):
            xq = xin if m < 2 else orc.quantize(xdn[s:s + 1])
            y64, S = orc.gemv(wl.host[(m, int(e))], N, K, xq, 1)
            check_close(outs[m][s], y64, S, f"moe m={m} slot={s}")


def test_gs64_lm_head_full(orc):
    """The gs64 workload as bench.py times it (quantiser launch, then the
    GEMV), every output of each weight copy against the oracle."""
    wl = bench.build_workload("gs64_lm_head", DEV, keep_host=True)
    for c in range(len(wl.W)):
        wl.copy = c
        wl.step()
        torch.cuda.synchronize()
        assert q.device_status() == 0
        qr, sr = orc.quantize_vec_i8(host(wl.x))
        assert np.array_equal(host(wl.qx), qr) and np.array_equal(host(wl.sx).view(np.int32), sr.view(np.int32))
        wq, ws = wl.host[c]
        y64, S = orc.gemv_gs64(wq, ws, wl.N, wl.K, qr, sr)
        check_close(host(wl.y), y64, S, f"gs64 lm_head copy {c}")

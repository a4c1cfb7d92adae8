"""The tcgen05 tensor-core kernel of packed few-token sequences (switched
on here; it is off by default) against the other paths and the CPU oracle,
through the C ABI (minfer README M16: the
multi-token path forms the same per-block integer sums as the one-token
path, so the logits do not depend on the step size).

Bit-exact: y of every sequence on the tcgen05 kernel equals y of the same
sequence with it switched off (the mma.sync and dp4a kernels), which the
other tests pin to the oracle; the fp32-input sequences (quantised first)
equal the quantised-input ones.  Within |y - y64| <= 1e-5 * S + 1e-6:
sampled outputs against the fp64 reference.  The shapes cut tiles between
warp groups and CTAs (few units per group), end in partial 128-row tiles
and in half segments (K = 11008: 344 blocks), and mix items in one launch.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests.gpu_util import check_close, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def orc():
    from quantized_q4_weight_gb300 import _build
    _build.build()
    oracle.build()
    yield oracle.load()
    q.set_tc_min_T(0)


def make(seed, shapes, T):
    ents = []
    for i, (N, K) in enumerate(shapes):
        Wg = synth.q4_0_weights(seed + i, N, K)
        W = q.pack_q4_0(to_dev(Wg), N, K)
        x = synth.activations(seed + 100 + i, T, K)
        xd = torch.from_numpy(x).to(DEV)
        ents.append(dict(Wg=Wg, W=W, x=x, xd=xd, xq=q.quantize_q8_0(xd, T, K), N=N, K=K))
    return ents


def run_seq(ents, T, f32=False):
    ys = [torch.full((T, e["N"]), float("nan"), dtype=torch.float32, device=DEV) for e in ents]
    if f32:
        items = q.seq_f32_items([(e["W"], e["xd"], y, e["N"], e["K"]) for e, y in zip(ents, ys)])
        ws = q.new_workspace(q.seq_f32_workspace_bytes(items, T))
        q.gemv_seq_f32(items, q.W_PACKED, T, ws)
    else:
        items = q.seq_items([(e["W"], e["xq"], y, e["N"], e["K"]) for e, y in zip(ents, ys)])
        ws = q.new_workspace(q.seq_workspace_bytes(items, T))
        q.gemv_seq(items, q.W_PACKED, T, ws)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    return [y.cpu().numpy() for y in ys]


# one item split over every warp group, items of a few units, a partial last
# tile (N % 128 != 0), half last segments (K = 11008, 8960), a mixed list
CASES = [
    [(2048, 11008)],
    [(16, 256)],
    [(4000, 1536)],
    [(48, 8960), (2560, 2048), (176, 256)],
    [(2560, 2048), (2048, 2048), (11008, 2048), (11008, 2048), (2048, 11008)],
]


@pytest.mark.parametrize("T", [5, 6, 7, 8])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_tc_bit_identical_to_other_paths_and_within_bound(orc, case, T):
    shapes = CASES[case]
    ents = make(900 + 10 * case + T, shapes, T)
    q.set_tc_min_T(1)
    y_tc = run_seq(ents, T)
    q.set_tc_min_T(9)
    y_ref = run_seq(ents, T)
    q.set_tc_min_T(0)
    rng = np.random.default_rng(case * 10 + T)
    for e, a, b in zip(ents, y_tc, y_ref):
        assert not np.isnan(a).any()
        assert np.array_equal(a.view(np.int32), b.view(np.int32)), (e["N"], e["K"])
        rows = np.unique(np.concatenate([[0, e["N"] - 1], rng.integers(0, e["N"], 40)]))
        y64, S = orc.gemv_rows(e["Wg"], e["N"], e["K"], orc.quantize(e["x"]), T, rows)
        check_close(a[:, rows], y64, S, f"tc N={e['N']} K={e['K']} T={T}")


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_tc_kernel_at_few_tokens(orc, T):
    # the kernel itself covers every T (forced on below its default)
    ents = make(700 + T, [(2560, 2048), (2048, 11008)], T)
    q.set_tc_min_T(1)
    y_tc = run_seq(ents, T)
    q.set_tc_min_T(9)
    y_ref = run_seq(ents, T)
    q.set_tc_min_T(0)
    for a, b in zip(y_tc, y_ref):
        assert np.array_equal(a.view(np.int32), b.view(np.int32))


@pytest.mark.parametrize("T", [5, 8])
def test_tc_fp32_inputs(orc, T):
    ents = make(800 + T, [(2560, 2048), (2048, 11008), (11008, 2048)], T)
    q.set_tc_min_T(1)
    y_q = run_seq(ents, T)
    y_f = run_seq(ents, T, f32=True)
    q.set_tc_min_T(9)
    y_old = run_seq(ents, T, f32=True)
    q.set_tc_min_T(0)
    for a, b, c in zip(y_q, y_f, y_old):
        assert np.array_equal(a.view(np.int32), b.view(np.int32))
        assert np.array_equal(b.view(np.int32), c.view(np.int32))


def test_tc_repeated_calls_share_a_workspace(orc):
    # the counters are left at zero: the same workspace serves the next call
    T = 8
    q.set_tc_min_T(1)
    ents = make(950, [(2048, 11008), (2560, 2048)], T)
    ys = [torch.empty((T, e["N"]), dtype=torch.float32, device=DEV) for e in ents]
    items = q.seq_items([(e["W"], e["xq"], y, e["N"], e["K"]) for e, y in zip(ents, ys)])
    ws = q.new_workspace(q.seq_workspace_bytes(items, T))
    outs = []
    for _ in range(3):
        q.gemv_seq(items, q.W_PACKED, T, ws)
        torch.cuda.synchronize()
        outs.append([y.cpu().numpy().copy() for y in ys])
    q.set_tc_min_T(0)
    assert q.device_status() == 0
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a.view(np.int32), b.view(np.int32))
    assert int(ws[:16384].count_nonzero()) == 0

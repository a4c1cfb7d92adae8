"""Top-2 rows per token and the verify-commit rule, through the C ABI,
against the CPU oracle.

Bit-exact: the two rows (against the oracle's top-2 of the GPU's own y, the
same y the plain GEMV writes), their values (y's, with -0 returned as +0),
the argmax calls' index (the first row), and the committed count of the
verify rule.  Against the fp64 reference the rows may differ only on a
near-tie within the output bound.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests.gpu_util import rank_vs_fp64, to_dev

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


def ws_for(N, K, T):
    return q.new_workspace(q.workspace_bytes(N, K, T))


def setup(seed, N, K, T, layout=q.W_PACKED):
    Wg = synth.q4_0_weights(seed, N, K)
    Wd = to_dev(Wg)
    W = q.pack_q4_0(Wd, N, K) if layout == q.W_PACKED else Wd
    x = synth.activations(seed + 1, T, K)
    xd = torch.from_numpy(x).to(DEV)
    return Wg, W, x, xd, q.quantize_q8_0(xd, T, K)


def check_top2_against_own_y(orc, idx2, val2, y):
    T, N = y.shape
    for t in range(T):
        i0, i1 = orc.top2_f32(y[t])
        assert (int(idx2[t, 0]), int(idx2[t, 1])) == (i0, i1)
        assert val2[t, 0].view(np.int32) == (y[t, i0] + np.float32(0)).view(np.int32)   # -0 comes back as +0
        if i1 >= 0:
            assert val2[t, 1].view(np.int32) == (y[t, i1] + np.float32(0)).view(np.int32)
        else:
            assert N == 1 and val2[t, 1] == -np.inf


# dp4a (T <= 4) and tensor-core (T >= 5) kernels; split-K (few slabs, several
# segments) and balanced (many slabs) modes; one and two rows
SHAPES = [(1, 32, 1), (2, 64, 2), (4099, 1536, 1), (1000, 544, 3), (40000, 512, 3), (20000, 256, 8),
          (48, 8960, 5), (40000, 512, 6), (3000, 2048, 7)]


@pytest.mark.parametrize("N,K,T", SHAPES)
def test_top2(orc, N, K, T):
    Wg, W, x, xd, xq = setup(31 * N + K + T, N, K, T)
    ws = ws_for(N, K, T)
    yw = torch.empty((T, N), dtype=torch.float32, device=DEV)
    idx2, val2 = q.gemv_top2(W, q.W_PACKED, xq, N, K, T, ws, y=yw)
    idx = q.gemv_argmax(W, q.W_PACKED, xq, N, K, T, ws).cpu().numpy()
    y = q.gemv(W, q.W_PACKED, xq, N, K, T, ws).cpu().numpy()
    idx2, val2 = idx2.cpu().numpy(), val2.cpu().numpy()
    assert np.array_equal(yw.cpu().numpy().view(np.int32), y.view(np.int32))
    assert np.array_equal(idx2[:, 0], idx)
    check_top2_against_own_y(orc, idx2, val2, y)
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    # against the fp64 top-2: equal, except on a counted near tie
    rank_vs_fp64(idx2, [orc.top2_f64(y64[t]) for t in range(T)], y64, S, f"top2 N={N} K={K} T={T}")
    assert q.device_status() == 0


@pytest.mark.parametrize("T", [1, 4, 8])
def test_top2_f32_and_ggml(orc, T):
    N, K = 6000, 1536
    Wg, W, x, xd, xq = setup(400 + T, N, K, T)
    ws = ws_for(N, K, T)
    a_i, a_v = q.gemv_top2(W, q.W_PACKED, xq, N, K, T, ws)
    b_i, b_v = q.gemv_top2_f32(W, q.W_PACKED, xd, N, K, T, ws)
    c_i, c_v = q.gemv_top2(to_dev(Wg), q.W_GGML, xq, N, K, T, ws)
    for i, v in ((b_i, b_v), (c_i, c_v)):
        assert torch.equal(i.cpu(), a_i.cpu())
        assert torch.equal(v.cpu().view(torch.int32), a_v.cpu().view(torch.int32))


def test_top2_ties_and_zero_rows(orc):
    N, K, T = 5000, 256, 2
    Wg = synth.q4_0_weights(41, N, K)
    blk = Wg.reshape(N, K // 32, 18).copy()
    for r in (4000, 4999):
        blk[r] = blk[1234]                                   # identical rows
    for r in (1234, 4000, 4999):
        blk[r, :, 0:2] = np.array([0x00, 0x7A], np.uint8)    # d = 49152: far above the rest
    Wg = blk.reshape(Wg.shape)
    x = synth.activations(42, T, K)
    xd = torch.from_numpy(x).to(DEV)
    xq = q.quantize_q8_0(xd, T, K)
    Wp = q.pack_q4_0(to_dev(Wg), N, K)
    ws = ws_for(N, K, T)
    idx2, val2 = (a.cpu().numpy() for a in q.gemv_top2(Wp, q.W_PACKED, xq, N, K, T, ws))
    y = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws).cpu().numpy()
    check_top2_against_own_y(orc, idx2, val2, y)
    for t in range(T):
        if y[t, 1234] == y[t].max():
            assert tuple(idx2[t]) == (1234, 4000) and val2[t, 0] == val2[t, 1]
    for bits in (0x0000, 0x8000):   # all outputs +0, or -0 that ties with +0
        Wz = q.pack_q4_0(to_dev(synth.with_scales(Wg, K, bits)), N, K)
        i2, v2 = (a.cpu().numpy() for a in q.gemv_top2(Wz, q.W_PACKED, xq, N, K, T, ws))
        assert np.all(i2 == np.array([0, 1])) and np.all(v2.view(np.int32) == 0)


def test_top2_argument_checks():
    import ctypes
    N, K, T = 64, 64, 2
    W = torch.zeros(q.q4_0_bytes(N, K), dtype=torch.uint8, device=DEV)
    xq = torch.zeros(q.xq_bytes(T, K), dtype=torch.uint8, device=DEV)
    ws = ws_for(N, K, T)
    buf = torch.zeros(64, dtype=torch.int64, device=DEV)
    base = buf.data_ptr()
    L = q.lib()

    def top2(idx_ptr, val_ptr):
        return L.qgemv_q4_0_top2(q._ptr(W), q.W_PACKED, q._ptr(xq), None, ctypes.c_void_p(idx_ptr),
                                 ctypes.c_void_p(val_ptr), N, K, T, q._ptr(ws), ws.numel(), q._stream())

    assert top2(base, base + 16 * T) == 0                  # disjoint and aligned: accepted
    torch.cuda.synchronize()
    assert top2(base, base + 8) == 1                       # val2 overlaps idx2
    assert top2(base + 4, base + 256) == 2                 # idx2 not 8-byte aligned
    assert top2(base, base + 256 + 2) == 2                 # val2 not 4-byte aligned
    assert top2(0, base + 256) == 1                        # no idx2
    n = base + 400
    def vc(tok, pred, stride, T):
        return L.qgemv_verify_commit(ctypes.c_void_p(tok), ctypes.c_void_p(pred), stride, T, ctypes.c_void_p(n),
                                     q._stream())

    assert vc(base, base, 1, 0) == 1 and vc(base, base, 1, 33) == 1 and vc(base, base, 0, 4) == 1
    assert vc(base + 4, base, 1, 4) == 2
    assert q.device_status() == 0


def test_verify_commit_against_oracle(orc):
    rng = np.random.default_rng(71)
    cases = [([5, 7, 9, 11], [7, 9, 11, 4]), ([5, 8, 9, 11], [7, 9, 11, 4]), ([5, 7, 10, 11], [7, 9, 11, 4]),
             ([5, 7, 0, 11], [7, 9, 11, 4]), ([5], [7])]
    for _ in range(200):
        T = int(rng.integers(1, 33))
        pred = rng.integers(0, 4, T)
        tokens = np.concatenate([[9], np.where(rng.random(T - 1) < 0.8, pred[:-1], rng.integers(0, 4, T - 1))])
        cases.append((tokens.tolist(), pred.tolist()))
    n = torch.empty(1, dtype=torch.int32, device=DEV)
    for tokens, pred in cases:
        tk = torch.tensor(tokens, dtype=torch.int64, device=DEV)
        pr = torch.tensor(pred, dtype=torch.int64, device=DEV)
        q.verify_commit(tk, pr, n_commit=n)
        assert int(n.item()) == orc.verify_commit(tokens, pred)


def test_verify_step_on_the_lm_head(orc):
    """A verify step end to end: T positions through the fp32 top-2 lm_head,
    then the commit rule on its first rows.  Drafts taken from the step's own
    predictions commit all T; a draft at position k + 1 that disagrees with
    pred[k] commits k + 1."""
    N, K, T = 151936 // 8, 1536, 8
    Wg, W, x, xd, xq = setup(77, N, K, T)
    ws = ws_for(N, K, T)
    idx2, val2 = q.gemv_top2_f32(W, q.W_PACKED, xd, N, K, T, ws)
    pred = idx2[:, 0]                       # a strided view: pred_stride 2
    n = torch.empty(1, dtype=torch.int32, device=DEV)
    for k in range(T):
        tokens = torch.cat([torch.tensor([3], dtype=torch.int64, device=DEV), pred[:-1].contiguous()])
        if k + 1 < T:
            tokens[k + 1] = (pred[k] + 1) % N     # the draft at position k+1 disagrees with pred[k]
        q.verify_commit(tokens, pred, n_commit=n)
        assert int(n.item()) == (k + 1 if k + 1 < T else T)
        assert int(n.item()) == orc.verify_commit(tokens.cpu().numpy(), pred.cpu().numpy())
    assert torch.all(val2[:, 0] >= val2[:, 1])


@pytest.mark.parametrize("T", [1, 3, 8])
def test_verify_in_one_launch(orc, T):
    """qgemv_q4_0_verify_f32 (top-2 and the rule in one launch) gives the
    rows, values and committed count of top2_f32 followed by verify_commit."""
    N, K = 20000, 1536
    Wg, W, x, xd, xq = setup(90 + T, N, K, T)
    ws = ws_for(N, K, T)
    i_ref, v_ref = q.gemv_top2_f32(W, q.W_PACKED, xd, N, K, T, ws)
    pred = i_ref[:, 0].contiguous()
    n_ref = torch.empty(1, dtype=torch.int32, device=DEV)
    for k in range(T):
        tokens = torch.cat([torch.tensor([5], dtype=torch.int64, device=DEV), pred[:-1]])
        if k + 1 < T:
            tokens[k + 1] = (pred[k] + 7) % N            # the draft after position k disagrees
        i2, v2, n = q.verify_f32(W, q.W_PACKED, xd, tokens, N, K, T, ws)
        q.verify_commit(tokens, pred, n_commit=n_ref)
        assert torch.equal(i2.cpu(), i_ref.cpu())
        assert torch.equal(v2.cpu().view(torch.int32), v_ref.cpu().view(torch.int32))
        assert int(n.item()) == int(n_ref.item()) == orc.verify_commit(tokens.cpu().numpy(), pred.cpu().numpy())
    assert q.device_status() == 0

"""CUDA path against the CPU oracle, through the C ABI, on small and ragged
shapes that span several slabs, segments and quads.

Bit-exact: Q8_0 activation bytes, per-block int32 sums, pack/unpack bytes,
argmax indices (against the argmax of the GPU's own y), and y across T,
layouts, split-K and entry points (the library's order depends on K only).
Within |y - y64| <= 1e-5 * S + 1e-6: every fp32 output against the fp64
reference.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests import oracle_pins as P
from tests.gpu_util import blocks_to_planar, check_close, planar_to_blocks, rank_vs_fp64, to_dev

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


def weights(seed, N, K, layout):
    Wg = synth.q4_0_weights(seed, N, K)
    Wd = to_dev(Wg)
    return Wg, (q.pack_q4_0(Wd, N, K) if layout == q.W_PACKED else Wd)


def quantized(seed, T, K):
    x = synth.activations(seed, T, K)
    xd = torch.from_numpy(x).to(DEV)
    return x, xd, q.quantize_q8_0(xd, T, K)


def ws_for(N, K, T):
    return q.new_workspace(q.workspace_bytes(N, K, T))


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("R,K,batch", [(1, 32, 1), (1, 1536, 1), (3, 96, 2), (8, 11008, 1), (9, 512, 3),
                                       (5, 8960, 1), (2, 64, 7)])
def test_quantize_bit_exact(orc, R, K, batch):
    x = synth.activations(100 + R + K + batch, batch * R, K)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), R, K, batch).cpu().numpy()
    n = q.xq_bytes(R, K)
    assert xq.size == n * batch
    for b in range(batch):
        ref = orc.quantize(x[b * R:(b + 1) * R])
        assert np.array_equal(xq[b * n:(b + 1) * n], blocks_to_planar(ref, n))


def test_quantize_hand_blocks_and_edges(orc):
    xs = [P._x_block(e) for e in P.golden()["q8_0"]]
    rng = np.random.default_rng(3)
    xs += [np.full(32, -3.0, np.float32), np.full(32, 1e-30, np.float32),            # tiny amax
           (rng.standard_normal(32) * 1e4).astype(np.float32),
           np.where(np.arange(32) % 2 == 0, 0.5, -0.5).astype(np.float32) * 127 / 63.5]
    x = np.stack(xs).reshape(1, -1).astype(np.float32)
    K = x.shape[1]
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), 1, K).cpu().numpy()
    assert np.array_equal(xq, blocks_to_planar(orc.quantize(x), q.xq_bytes(1, K)))
    for i, e in enumerate(P.golden()["q8_0"]):
        blk = planar_to_blocks(xq, 1, K)[0, i]
        assert int(blk[0]) | (int(blk[1]) << 8) == int(e["d_bits"], 16)
        assert np.array_equal(blk[2:].view(np.int8), P._q_block(e))


# ----------------------------------------------------------------- pack

@pytest.mark.parametrize("N,K", [(1, 32), (15, 64), (16, 128), (17, 96), (33, 160), (100, 544), (48, 2080)])
def test_pack_roundtrip_and_layout(orc, N, K):
    Wg = synth.q4_0_weights(N * K, N, K)
    Wd = to_dev(Wg)
    Wp = q.pack_q4_0(Wd, N, K)
    assert torch.equal(q.unpack_q4_0(Wp, N, K), Wd)
    # the layout as include/qgemv.h states it
    got = Wp.cpu().numpy()
    nb = K // 32
    blk = Wg.reshape(N, nb, 18)
    nfull = N // 16
    for s in range(nfull):
        base = s * 288 * nb
        for qd in range((nb + 3) // 4):
            nbq = min(4, nb - 4 * qd)
            qb = base + 1152 * qd
            for r in range(16):
                for jq in range(nbq):
                    b = 4 * qd + jq
                    c = ((jq + (r >> 1)) & 3) if nbq == 4 else jq     # full quads rotate by r // 2
                    o = qb + (r * nbq + c) * 16
                    assert np.array_equal(got[o:o + 16], blk[16 * s + r, b, 2:])
                    so = qb + 256 * nbq + ((r % 8) * nbq + jq) * 4 + (r // 8) * 2
                    assert np.array_equal(got[so:so + 2], blk[16 * s + r, b, :2])
    tail = nfull * 16 * nb * 18
    assert np.array_equal(got[tail:], Wg.reshape(-1)[tail:])


# ----------------------------------------------------------------- block sums

@pytest.mark.parametrize("layout", [q.W_PACKED, q.W_GGML])
@pytest.mark.parametrize("N,K,T", [(16, 32, 1), (17, 544, 3), (40, 1536, 8), (5, 96, 2)])
def test_block_isums_bit_exact(orc, layout, N, K, T):
    Wg, W = weights(11 * N + K, N, K, layout)
    x, xd, xq = quantized(13 * N + T, T, K)
    got = q.block_isums(W, layout, xq, N, K, T).cpu().numpy()
    ref = orc.block_isums(Wg, N, K, orc.quantize(x), T)
    assert np.array_equal(got, ref)


def test_block_isums_range_extremes(orc):
    K, N = 64, 16
    W = synth.with_scales(synth.with_nibbles(synth.q4_0_weights(1, N, K), K, 0), K, 0x3C00)
    x = np.full((1, K), -127.0, np.float32)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), 1, K)
    got = q.block_isums(q.pack_q4_0(to_dev(W), N, K), q.W_PACKED, xq, N, K, 1).cpu().numpy()
    assert np.all(got == 32512)


# The tensor-core path's own block sums (its MMAs over the subnormal nibble
# operands, both activation operand forms), bit-exact against the oracle.
@pytest.mark.parametrize("f16_image", [True, False])
@pytest.mark.parametrize("layout", [q.W_PACKED, q.W_GGML])
@pytest.mark.parametrize("N,K,T", [(16, 32, 5), (17, 544, 6), (40, 1536, 8), (35, 96, 7), (33, 2080, 2),
                                   (48, 8960, 4), (1, 64, 1), (100, 160, 3)])
def test_block_isums_tensor_core_bit_exact(orc, f16_image, layout, N, K, T):
    Wg, W = weights(11 * N + K + 1, N, K, layout)
    x, xd, xq = quantized(13 * N + T + 1, T, K)
    got = q.block_isums_tc(W, layout, xq, N, K, T, f16_image).cpu().numpy()
    ref = orc.block_isums(Wg, N, K, orc.quantize(x), T)
    assert np.array_equal(got, ref)
    assert np.array_equal(got, q.block_isums(W, layout, xq, N, K, T).cpu().numpy())


@pytest.mark.parametrize("f16_image", [True, False])
def test_block_isums_tensor_core_extremes(orc, f16_image):
    # nibbles all 0 or all 15 against codes all -127 or +127 (per token), and
    # one block of each nibble value 0..15 against a ramp: the range ends
    # +-32512 and every nibble value through both MMAs
    K, N, T = 64, 32, 8
    W0 = synth.with_nibbles(synth.q4_0_weights(2, 16, K), K, 0)
    W15 = synth.with_nibbles(synth.q4_0_weights(3, 16, K), K, 15)
    Wg = np.concatenate([W0, W15])
    x = np.empty((T, K), np.float32)
    for t in range(T):
        x[t] = 127.0 if t % 2 == 0 else -127.0
    x[7] = np.linspace(-127, 127, K).astype(np.float32)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), T, K)
    for layout in (q.W_PACKED, q.W_GGML):
        W = q.pack_q4_0(to_dev(Wg), N, K) if layout == q.W_PACKED else to_dev(Wg)
        got = q.block_isums_tc(W, layout, xq, N, K, T, f16_image).cpu().numpy()
        ref = orc.block_isums(Wg, N, K, orc.quantize(x), T)
        assert np.array_equal(got, ref)
        assert got[0, 0, 0] == -32512 and got[1, 0, 0] == 32512 and got[0, 16, 0] == 7 * 32 * 127
    # every nibble value: row r of a slab holds nibble r in every position
    rows = [synth.with_nibbles(synth.q4_0_weights(10 + r, 1, K), K, r) for r in range(16)]
    Wn = np.concatenate(rows)
    W = q.pack_q4_0(to_dev(Wn), 16, K)
    got = q.block_isums_tc(W, q.W_PACKED, xq, 16, K, T, f16_image).cpu().numpy()
    assert np.array_equal(got, orc.block_isums(Wn, 16, K, orc.quantize(x), T))


# ----------------------------------------------------------------- GEMV vs oracle

SHAPES = [(1, 32), (15, 64), (16, 512), (17, 544), (64, 1536), (100, 2080), (48, 8960), (300, 1024), (33, 11008)]


@pytest.mark.parametrize("layout", [q.W_PACKED, q.W_GGML])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemv_matches_oracle(orc, layout, N, K, T):
    Wg, W = weights(7 * N + K, N, K, layout)
    x, xd, xq = quantized(3 * N + K + T, T, K)
    y = q.gemv(W, layout, xq, N, K, T, ws_for(N, K, T))
    torch.cuda.synchronize()
    assert q.device_status() == 0
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    check_close(y.cpu().numpy(), y64, S, f"N={N} K={K} T={T}")


def test_closed_forms_on_gpu(orc):
    for e in P.golden()["closed_forms"]:
        K, N = e["K"], 20
        Wg = synth.with_scales(synth.with_nibbles(synth.q4_0_weights(1, N, K), K, e["nibble"]), K,
                               int(e["w_d_bits"], 16))
        x = np.full((1, K), e["x_value"], np.float32)
        xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), 1, K)
        for layout in (q.W_PACKED, q.W_GGML):
            W = q.pack_q4_0(to_dev(Wg), N, K) if layout == q.W_PACKED else to_dev(Wg)
            y = q.gemv(W, layout, xq, N, K, 1, ws_for(N, K, 1)).cpu().numpy()
            assert np.all(y == e["y"]), (e["name"], y)


def test_hand_block_on_gpu(orc):
    for e in P.golden()["q4_0"]:
        w = P._wq_bytes(int(e["w_d_bits"], 16), e["w_qs"])
        xe = [g for g in P.golden()["q8_0"] if g["name"] == e["x_block"]][0]
        x = P._x_block(xe).reshape(1, 32)
        W = to_dev(np.tile(w, 16))                        # 16 identical rows = one slab
        xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), 1, 32)
        for layout, Wl in ((q.W_GGML, W), (q.W_PACKED, q.pack_q4_0(W, 16, 32))):
            assert np.all(q.block_isums(Wl, layout, xq, 16, 32, 1).cpu().numpy() == e["isum"])
            assert np.all(q.gemv(Wl, layout, xq, 16, 32, 1, ws_for(16, 32, 1)).cpu().numpy() == e["y"])


# ----------------------------------------------------------------- bit identity

@pytest.mark.parametrize("N,K", [(50, 8960), (40, 1536), (7, 544), (300, 2048)])
def test_bit_identical_across_T_layouts_and_paths(orc, N, K):
    Wg, Wp = weights(5 * N + K, N, K, q.W_PACKED)
    Wd = to_dev(Wg)
    x, xd, xq8 = quantized(9 * N, 8, K)
    y8 = q.gemv(Wp, q.W_PACKED, xq8, N, K, 8, ws_for(N, K, 8)).cpu()
    y8g = q.gemv(Wd, q.W_GGML, xq8, N, K, 8, ws_for(N, K, 8)).cpu()
    assert torch.equal(y8.view(torch.int32), y8g.view(torch.int32))
    for t in range(8):
        xq1 = q.quantize_q8_0(xd[t:t + 1].contiguous(), 1, K)
        y1 = q.gemv(Wp, q.W_PACKED, xq1, N, K, 1, ws_for(N, K, 1)).cpu()
        assert torch.equal(y1[0].view(torch.int32), y8[t].view(torch.int32)), t
    # fp32-input entry point == quantise + GEMV
    yf = q.gemv_f32(Wp, q.W_PACKED, xd, N, K, 8, ws_for(N, K, 8)).cpu()
    assert torch.equal(yf.view(torch.int32), y8.view(torch.int32))
    # a long sequence launch (no split-K) gives the same bits as the single call (split-K when K > 512)
    reps = 160
    ys = [torch.empty((8, N), dtype=torch.float32, device=DEV) for _ in range(reps)]
    items = q.seq_items([(Wp, xq8, ys[i], N, K) for i in range(reps)])
    ws = q.new_workspace(q.seq_workspace_bytes(items, 8))
    q.gemv_seq(items, q.W_PACKED, 8, ws)
    for i in (0, reps // 2, reps - 1):
        assert torch.equal(ys[i].cpu().view(torch.int32), y8.view(torch.int32))


# ----------------------------------------------------------------- argmax

@pytest.mark.parametrize("layout", [q.W_PACKED, q.W_GGML])
@pytest.mark.parametrize("N,K,T", [(1, 32, 1), (4099, 1536, 1), (1000, 544, 3), (20000, 256, 8), (48, 8960, 2)])
def test_argmax(orc, layout, N, K, T):
    Wg, W = weights(17 * N + K, N, K, layout)
    x, xd, xq = quantized(19 * N + T, T, K)
    ws = ws_for(N, K, T)
    y = torch.empty((T, N), dtype=torch.float32, device=DEV)
    idx = q.gemv_argmax(W, layout, xq, N, K, T, ws, y=y).cpu().numpy()
    idx2 = q.gemv_argmax(W, layout, xq, N, K, T, ws).cpu().numpy()        # y not written
    yref = q.gemv(W, layout, xq, N, K, T, ws).cpu().numpy()
    assert np.array_equal(y.cpu().numpy().view(np.int32), yref.view(np.int32))
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    for t in range(T):
        assert idx[t] == idx2[t] == orc.argmax_f32(yref[t])
    # against the fp64 argmax: equal, except on a counted near tie
    rank_vs_fp64(idx, [orc.argmax_f64(y64[t]) for t in range(T)], y64, S, f"argmax N={N} K={K} T={T}")


def test_argmax_ties_and_zero_rows(orc):
    N, K, T = 5000, 256, 2
    Wg = synth.q4_0_weights(23, N, K)
    Wg[4000] = Wg[1234]          # identical rows
    Wg[4999] = Wg[1234]
    x, xd, xq = quantized(24, T, K)
    Wp = q.pack_q4_0(to_dev(Wg), N, K)
    y = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu().numpy()
    # make row 1234 the maximum for token 0 by construction: scale it up
    blk = Wg.reshape(N, K // 32, 18).copy()
    for r in (1234, 4000, 4999):
        blk[r, :, 0:2] = np.array([0x00, 0x7A], np.uint8)     # d = 49152 on every block
    Wg2 = blk.reshape(Wg.shape)
    Wp2 = q.pack_q4_0(to_dev(Wg2), N, K)
    y2 = q.gemv(Wp2, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu().numpy()
    idx = q.gemv_argmax(Wp2, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu().numpy()
    for t in range(T):
        assert idx[t] == orc.argmax_f32(y2[t])
        if y2[t, 1234] == y2[t].max():
            assert idx[t] == 1234
    # all-zero scales: every output is +-0 and the answer is row 0
    Wz = q.pack_q4_0(to_dev(synth.with_scales(Wg, K, 0x0000)), N, K)
    assert np.all(q.gemv_argmax(Wz, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu().numpy() == 0)
    # negative-zero scales give -0 outputs that tie with +0
    Wn = q.pack_q4_0(to_dev(synth.with_scales(Wg, K, 0x8000)), N, K)
    assert np.all(q.gemv_argmax(Wn, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu().numpy() == 0)
    del y


# ----------------------------------------------------------------- sequence and gather

def test_seq_matches_single_calls(orc):
    shapes = [(2048, 1536), (1536, 1536), (96, 8960), (17, 544), (64, 32), (300, 2048)]
    T = 3
    entries, refs = [], []
    for i, (N, K) in enumerate(shapes):
        Wg, Wp = weights(40 + i, N, K, q.W_PACKED)
        x, xd, xq = quantized(60 + i, T, K)
        y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
        entries.append((Wp, xq, y, N, K))
        refs.append((Wg, x, q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu()))
    items = q.seq_items(entries)
    ws = q.new_workspace(q.seq_workspace_bytes(items, T))
    q.gemv_seq(items, q.W_PACKED, T, ws)
    torch.cuda.synchronize()
    for (Wp, xq, y, N, K), (Wg, x, yref) in zip(entries, refs):
        assert torch.equal(y.cpu().view(torch.int32), yref.view(torch.int32)), (N, K)
        y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
        check_close(y.cpu().numpy(), y64, S, f"seq N={N} K={K}")


@pytest.mark.parametrize("layout", [q.W_PACKED, q.W_GGML])
def test_gather_matches_single_calls(orc, layout):
    n_experts, d_model, d_ff, T = 12, 512, 160, 1
    shapes = [("gate", d_ff, d_model), ("up", d_ff, d_model), ("down", d_model, d_ff)]
    ids_np = np.array([3, 7, 3, 11, 0], np.int32)          # repeats allowed
    n_ids = ids_np.size
    mats, checks = [], []
    for m, (name, N, K) in enumerate(shapes):
        per = q.q4_0_bytes(N, K)
        Wg_all = [synth.q4_0_weights(500 + 10 * m + e, N, K) for e in range(n_experts)]
        Wd = torch.cat([to_dev(w) for w in Wg_all])
        W = torch.cat([q.pack_q4_0(to_dev(w), N, K) for w in Wg_all]) if layout == q.W_PACKED else Wd
        shared = name != "down"
        xs = synth.activations(700 + m, 1 if shared else n_ids, K)
        xqb = q.xq_bytes(T, K)
        xq = q.quantize_q8_0(torch.from_numpy(xs).to(DEV), T, K, batch=xs.shape[0])
        y = torch.full((n_ids, T, N), float("nan"), dtype=torch.float32, device=DEV)
        mats.append((W, per, xq, 0 if shared else xqb, y, T * N, N, K))
        checks.append((Wg_all, W, per, xs, xq, xqb, y, N, K, shared))
    gm = q.gather_mats(mats)
    ws = q.new_workspace(q.gather_workspace_bytes(gm, n_ids, T))
    ids = torch.from_numpy(ids_np).to(DEV)
    q.gemv_gather(gm, ids, n_experts, layout, T, ws)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    for Wg_all, W, per, xs, xq, xqb, y, N, K, shared in checks:
        for s in range(n_ids):
            e = int(ids_np[s])
            xqs = xq[(0 if shared else s) * xqb:((0 if shared else s) + 1) * xqb]
            Ws = W[e * per:(e + 1) * per]
            yref = q.gemv(Ws, layout, xqs, N, K, T, ws_for(N, K, T)).cpu()
            assert torch.equal(y[s].cpu().view(torch.int32), yref.view(torch.int32))
            y64, S = orc.gemv(Wg_all[e], N, K, orc.quantize(xs[0 if shared else s][None]), T)
            check_close(y[s].cpu().numpy(), y64, S, "gather")
    # an expert id out of range: nothing read for that slot, status recorded
    bad = torch.tensor([1, 99], dtype=torch.int32, device=DEV)
    for W, _, xq, _, y, _, N, K in mats:
        y.fill_(-1.0)
    q.gemv_gather(gm, bad, n_experts, layout, T, ws)
    torch.cuda.synchronize()
    assert q.device_status() == 7                         # QGEMV_ERR_BAD_ID
    for W, _, xq, _, y, _, N, K in mats:
        assert torch.all(y[1] == -1.0) and not torch.all(y[0] == -1.0)
    assert q.device_status() == 0


@pytest.mark.parametrize("T", [3, 6])
def test_gather_several_tokens_and_bad_ids(orc, T):
    """Gathers at several tokens (dp4a at T = 3, the tensor cores at T = 6),
    many slots over a grid of CTAs, repeated ids: each slot bit-identical to
    a single call on its expert and within the bound of the oracle; then one
    slot with an id out of range (nothing read for it, its output untouched,
    the status word set) while the others stay bit-identical."""
    n_experts, N, K = 10, 1024, 2048
    per = q.q4_0_bytes(N, K)
    Wg_all = [synth.q4_0_weights(2100 + e, N, K) for e in range(n_experts)]
    W = torch.cat([q.pack_q4_0(to_dev(w), N, K) for w in Wg_all])
    ids_np = np.array([4, 9, 4, 0, 7, 2, 9, 5], np.int32)
    n_ids = ids_np.size
    xs = synth.activations(2200 + T, n_ids * T, K)
    xqb = q.xq_bytes(T, K)
    xq = q.quantize_q8_0(torch.from_numpy(xs).to(DEV), T, K, batch=n_ids)
    y = torch.full((n_ids, T, N), float("nan"), dtype=torch.float32, device=DEV)
    gm = q.gather_mats([(W, per, xq, xqb, y, T * N, N, K)])
    ws = q.new_workspace(q.gather_workspace_bytes(gm, n_ids, T))
    q.gemv_gather(gm, torch.from_numpy(ids_np).to(DEV), n_experts, q.W_PACKED, T, ws)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    ref = []
    for s_ in range(n_ids):
        e = int(ids_np[s_])
        yref = q.gemv(W[e * per:(e + 1) * per], q.W_PACKED, xq[s_ * xqb:(s_ + 1) * xqb], N, K, T,
                      ws_for(N, K, T)).cpu()
        ref.append(yref)
        assert torch.equal(y[s_].cpu().view(torch.int32), yref.view(torch.int32)), s_
        y64, S = orc.gemv(Wg_all[e], N, K, orc.quantize(xs[s_ * T:(s_ + 1) * T]), T)
        check_close(y[s_].cpu().numpy(), y64, S, f"gather T={T} slot {s_}")
    bad_np = ids_np.copy()
    bad_np[5] = n_experts                                   # out of range
    y.fill_(-1.0)
    q.gemv_gather(gm, torch.from_numpy(bad_np).to(DEV), n_experts, q.W_PACKED, T, ws)
    torch.cuda.synchronize()
    assert q.device_status() == 7                           # QGEMV_ERR_BAD_ID
    assert torch.all(y[5] == -1.0)
    for s_ in range(n_ids):
        if s_ != 5:
            assert torch.equal(y[s_].cpu().view(torch.int32), ref[s_].view(torch.int32)), s_
    assert q.device_status() == 0


# ----------------------------------------------------------------- workspace contract

def test_workspace_left_zeroed_and_reusable(orc):
    N, K, T = 96, 8960, 4            # few slabs: split-K with counters
    Wg, Wp = weights(77, N, K, q.W_PACKED)
    x, xd, xq = quantized(78, T, K)
    ws = ws_for(N, K, T)
    y1 = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws).cpu()
    idx = q.gemv_argmax(Wp, q.W_PACKED, xq, N, K, T, ws).cpu()
    y2 = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws).cpu()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32)[0]) == 0           # argmax arrival counter
    assert idx.shape == (T,)


@pytest.mark.parametrize("layout", [q.W_PACKED, q.W_GGML])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_seq_balanced_mode_bit_identical(orc, layout, T):
    """Lists with 608 slabs or more run unsplit, with CTAs balanced by
    16-block stages (slabs cut between warps); the bits must equal the single
    calls (which split K) and stay within the bound of the oracle."""
    shapes = [(2048, 1536), (1000, 2080), (1536, 8960), (17, 544), (301, 1024), (64, 11008), (8960, 1536)] * 3
    entries, refs = [], []
    cache = {}
    for i, (N, K) in enumerate(shapes):
        if (N, K) not in cache:
            Wg, W = weights(300 + N + K, N, K, layout)
            x, xd, xq = quantized(400 + N + K + T, T, K)
            yref = q.gemv(W, layout, xq, N, K, T, ws_for(N, K, T)).cpu()
            cache[(N, K)] = (Wg, W, x, xq, yref)
        Wg, W, x, xq, yref = cache[(N, K)]
        y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
        entries.append((W, xq, y, N, K))
        refs.append(((N, K), yref))
    items = q.seq_items(entries)
    ws = q.new_workspace(q.seq_workspace_bytes(items, T))
    for rep in range(2):
        for e in entries:
            e[2].fill_(float("nan"))
        q.gemv_seq(items, layout, T, ws)
        torch.cuda.synchronize()
        assert q.device_status() == 0
        for (W, xq, y, N, K), (key, yref) in zip(entries, refs):
            assert torch.equal(y.cpu().view(torch.int32), yref.view(torch.int32)), (key, rep)
    rng = np.random.default_rng(T)
    for (N, K), (Wg, W, x, xq, yref) in cache.items():
        rows = np.unique(rng.integers(0, N, 12))
        y64, S = orc.gemv_rows(Wg, N, K, orc.quantize(x), T, rows)
        check_close(yref.numpy()[:, rows], y64, S, f"balanced N={N} K={K}")


@pytest.mark.parametrize("T", [5, 6, 8])
def test_seq_small_groups_bit_identical(orc, T):
    """Layer lists whose long-row projections need the activation area alone
    leave CTAs with groups of a few slabs, which all warps of a tensor-core
    launch share when the workspace holds the CTAs' segment-sum regions.  The bits must equal the
    single calls with the full workspace, with regions for a third of the
    CTAs, and with none."""
    shapes = [(2048, 2048), (256, 2048), (2048, 11008), (11008, 2048), (2048, 11008), (1536, 8960)] * 4
    entries, refs, cache = [], [], {}
    for N, K in shapes:
        if (N, K) not in cache:
            Wg, W = weights(700 + N + K, N, K, q.W_PACKED)
            x, xd, xq = quantized(800 + N + K + T, T, K)
            yref = q.gemv(W, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu()
            cache[(N, K)] = (Wg, W, x, xq, yref)
        Wg, W, x, xq, yref = cache[(N, K)]
        entries.append((W, xq, torch.empty((T, N), dtype=torch.float32, device=DEV), N, K))
        refs.append(((N, K), yref))
    items = q.seq_items(entries)
    full = q.seq_workspace_bytes(items, T)
    base = 16384                                   # the counter area: all an unsplit list needs
    assert full > base
    for size in (full, base + (full - base) // 3, base):
        ws = q.new_workspace(size)
        for e in entries:
            e[2].fill_(float("nan"))
        q.gemv_seq(items, q.W_PACKED, T, ws)
        torch.cuda.synchronize()
        assert q.device_status() == 0
        for (W, xq, y, N, K), (key, yref) in zip(entries, refs):
            assert torch.equal(y.cpu().view(torch.int32), yref.view(torch.int32)), (key, size)
    rng = np.random.default_rng(70 + T)
    for (N, K), (Wg, W, x, xq, yref) in cache.items():
        rows = np.unique(rng.integers(0, N, 8))
        y64, S = orc.gemv_rows(Wg, N, K, orc.quantize(x), T, rows)
        check_close(yref.numpy()[:, rows], y64, S, f"small groups N={N} K={K}")


def test_seq_f32_equals_quantize_then_seq(orc):
    shapes = [(2048, 1536), (17, 544), (1536, 8960), (100, 2080)] * 40
    T = 2
    entries_f, entries_q, ys_f, ys_q = [], [], [], []
    for i, (N, K) in enumerate(shapes):
        Wg, Wp = weights(900 + N + K, N, K, q.W_PACKED) if i < 4 else (None, entries_f[i % 4][0])
        x = torch.from_numpy(synth.activations(950 + i, T, K)).to(DEV)
        yf = torch.empty((T, N), dtype=torch.float32, device=DEV)
        yq = torch.empty((T, N), dtype=torch.float32, device=DEV)
        entries_f.append((Wp, x, yf, N, K))
        entries_q.append((Wp, q.quantize_q8_0(x, T, K), yq, N, K))
        ys_f.append(yf)
        ys_q.append(yq)
    itf = q.seq_f32_items(entries_f)
    itq = q.seq_items(entries_q)
    q.gemv_seq_f32(itf, q.W_PACKED, T, q.new_workspace(q.seq_f32_workspace_bytes(itf, T)))
    q.gemv_seq(itq, q.W_PACKED, T, q.new_workspace(q.seq_workspace_bytes(itq, T)))
    torch.cuda.synchronize()
    assert q.device_status() == 0
    for a, b in zip(ys_f, ys_q):
        assert torch.equal(a.cpu().view(torch.int32), b.cpu().view(torch.int32))


@pytest.mark.parametrize("N,K", [(40, 1536), (17, 544), (300, 2080), (33, 8960)])
@pytest.mark.parametrize("T", [2, 3, 8])
def test_dp4a_and_tensor_core_paths_bit_identical(orc, N, K, T):
    """T > 1 runs on the int8 tensor-core path or on dp4a (a tuning choice);
    both must give the same bits, and the split / unsplit launches too."""
    Wg, Wp = weights(600 + N + K, N, K, q.W_PACKED)
    x, xd, xq = quantized(650 + N + T, T, K)
    outs = []
    try:
        for mma_min in (9, 2):
            q.set_tuning(0, 0, mma_min)
            outs.append(q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu())
            ys = [torch.empty((T, N), dtype=torch.float32, device=DEV) for _ in range(48)]
            items = q.seq_items([(Wp, xq, y, N, K) for y in ys])
            q.gemv_seq(items, q.W_PACKED, T, q.new_workspace(q.seq_workspace_bytes(items, T)))
            outs += [y.cpu() for y in ys[::16]]
    finally:
        q.set_tuning(0, 0, 0)
    assert q.device_status() == 0
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int32), o.view(torch.int32))
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    check_close(outs[-1].numpy(), y64, S, f"paths N={N} K={K} T={T}")


@pytest.mark.parametrize("T", [2, 8])
def test_paths_at_extreme_magnitudes(orc, T):
    """Nibbles all 0 or all 15 and activations all +-127 (same sign across a
    block): the largest block sums and folded constants either path meets."""
    N, K = 48, 1024
    nb = K // 32
    rng = np.random.default_rng(77)
    Wg = np.zeros((N, nb, 18), np.uint8)
    d = rng.uniform(1e-3, 1e-2, (N, nb)).astype(np.float16)
    Wg[:, :, :2] = d.view(np.uint8).reshape(N, nb, 2)
    Wg[:, :, 2:] = rng.choice(np.array([0x00, 0xFF, 0x0F, 0xF0], np.uint8), (N, nb))[:, :, None]
    Wg = Wg.reshape(-1)
    sign = rng.choice(np.array([-1.0, 1.0], np.float32), (T, nb))
    x = np.repeat(sign, 32, axis=1).astype(np.float32)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), T, K)
    Wp = q.pack_q4_0(to_dev(Wg), N, K)
    outs = []
    try:
        for mma_min in (9, 2):
            q.set_tuning(0, 0, mma_min)
            for W, lay in ((Wp, q.W_PACKED), (to_dev(Wg), q.W_GGML)):
                outs.append(q.gemv(W, lay, xq, N, K, T, ws_for(N, K, T)).cpu())
    finally:
        q.set_tuning(0, 0, 0)
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int32), o.view(torch.int32))
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    check_close(outs[0].numpy(), y64, S, f"extremes T={T}")


@pytest.mark.parametrize("ring_depth", [1, 3, 6])
def test_ring_depth_leaves_results_unchanged(orc, ring_depth):
    """The weight-stage depth per warp is a tuning knob only: same bits."""
    N, K, T = 300, 2080, 1
    Wg, Wp = weights(900 + ring_depth, N, K, q.W_PACKED)
    x, xd, xq = quantized(901, T, K)
    ref = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu()
    ys = [torch.empty((T, N), dtype=torch.float32, device=DEV) for _ in range(40)]
    items = q.seq_items([(Wp, xq, y, N, K) for y in ys])
    try:
        q.set_tuning(0, 0, 0, ring_depth)
        got = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu()
        q.gemv_seq(items, q.W_PACKED, T, q.new_workspace(q.seq_workspace_bytes(items, T)))
        torch.cuda.synchronize()
    finally:
        q.set_tuning(0, 0, 0, 0)
    assert q.device_status() == 0
    for o in [got] + [y.cpu() for y in ys[::13]]:
        assert torch.equal(ref.view(torch.int32), o.view(torch.int32))


@pytest.mark.parametrize("T,K", [(1, 1536), (3, 544), (8, 1536), (8, 8960)])
@pytest.mark.parametrize("offset", [0, 1])
def test_fp32_entry_points_quantise_in_kernel(orc, T, K, offset):
    """The fp32 calls quantise inside the GEMV kernel: the same bits as the
    standalone quantiser followed by the quantised-input call, with x
    16-byte aligned (offset 0) or only 4-byte aligned (offset 1 float).
    T = 8 covers the tensor-core path with an f16 (K = 1536) and an int8
    (K = 8960) activation image."""
    N = 200
    Wg, Wp = weights(1000 + T + K, N, K, q.W_PACKED)
    x = synth.activations(1100 + T + K, T, K)
    buf = torch.zeros(T * K + 4, dtype=torch.float32, device=DEV)
    xd = buf[offset:offset + T * K].view(T, K)
    xd.copy_(torch.from_numpy(x))
    xq = q.quantize_q8_0(xd.contiguous(), T, K)
    ref = q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu()
    got = q.gemv_f32(Wp, q.W_PACKED, xd, N, K, T, ws_for(N, K, T)).cpu()
    ys = [torch.empty((T, N), dtype=torch.float32, device=DEV) for _ in range(3)]
    items = q.seq_f32_items([(Wp, xd, y, N, K) for y in ys])
    q.gemv_seq_f32(items, q.W_PACKED, T, q.new_workspace(q.seq_f32_workspace_bytes(items, T)))
    torch.cuda.synchronize()
    assert q.device_status() == 0
    for o in [got] + [y.cpu() for y in ys]:
        assert torch.equal(ref.view(torch.int32), o.view(torch.int32))
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    check_close(got.numpy(), y64, S, f"fp32 in-kernel quantise T={T} K={K}")


@pytest.mark.parametrize("T", [1, 8])
def test_argmax_f32_matches_quantised_argmax(orc, T):
    """The fp32-input argmax quantises in the kernel: same index and same y
    bits as quantising first."""
    N, K = 5000, 1536
    Wg, Wp = weights(1200 + T, N, K, q.W_PACKED)
    x = synth.activations(1201 + T, T, K)
    xd = torch.from_numpy(x).to(DEV)
    xq = q.quantize_q8_0(xd, T, K)
    y0 = torch.empty((T, N), dtype=torch.float32, device=DEV)
    y1 = torch.empty((T, N), dtype=torch.float32, device=DEV)
    i0 = q.gemv_argmax(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T), y=y0).cpu()
    i1 = q.gemv_argmax_f32(Wp, q.W_PACKED, xd, N, K, T, ws_for(N, K, T), y=y1).cpu()
    assert q.device_status() == 0
    assert torch.equal(i0, i1)
    assert torch.equal(y0.cpu().view(torch.int32), y1.cpu().view(torch.int32))
    for t in range(T):
        assert int(i1[t]) == orc.argmax_f32(y1[t].cpu().numpy())


def test_gather_f32_matches_quantised_gather(orc):
    """The fp32 gather quantises inside the kernel: same bits as quantising
    the shared input and the per-slot inputs first."""
    T, n_exp, n_ids = 1, 6, 4
    N1, K1, N2, K2 = 96, 512, 512, 256
    shapes = [(N1, K1), (N2, K2)]
    W = []
    for m, (N, K) in enumerate(shapes):
        per = q.q4_0_bytes(N, K)
        buf = torch.empty(n_exp * per, dtype=torch.uint8, device=DEV)
        for e in range(n_exp):
            buf[e * per:(e + 1) * per] = q.pack_q4_0(to_dev(synth.q4_0_weights(1300 + m, N, K, stream=(e,))), N, K)
        W.append(buf)
    x1 = torch.from_numpy(synth.activations(1310, T, K1)).to(DEV)
    x2 = torch.from_numpy(synth.activations(1311, n_ids * T, K2)).to(DEV)
    xq1 = q.quantize_q8_0(x1, T, K1)
    xq2 = q.quantize_q8_0(x2, T, K2, batch=n_ids)
    ids = torch.tensor([3, 0, 5, 3], dtype=torch.int32, device=DEV)
    outs = []
    for f32 in (False, True):
        y1 = torch.empty((n_ids, T, N1), dtype=torch.float32, device=DEV)
        y2 = torch.empty((n_ids, T, N2), dtype=torch.float32, device=DEV)
        if f32:
            mats = q.gather_f32_mats([(W[0], q.q4_0_bytes(N1, K1), x1, 0, y1, T * N1, N1, K1),
                                      (W[1], q.q4_0_bytes(N2, K2), x2, 4 * T * K2, y2, T * N2, N2, K2)])
            q.gemv_gather_f32(mats, ids, n_exp, q.W_PACKED, T, q.new_workspace(q.gather_f32_workspace_bytes(mats, n_ids, T)))
        else:
            mats = q.gather_mats([(W[0], q.q4_0_bytes(N1, K1), xq1, 0, y1, T * N1, N1, K1),
                                  (W[1], q.q4_0_bytes(N2, K2), xq2, q.xq_bytes(T, K2), y2, T * N2, N2, K2)])
            q.gemv_gather(mats, ids, n_exp, q.W_PACKED, T, q.new_workspace(q.gather_workspace_bytes(mats, n_ids, T)))
        torch.cuda.synchronize()
        outs.append((y1.cpu(), y2.cpu()))
    assert q.device_status() == 0
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("f32", [False, True])
def test_seq_longer_than_one_launch(orc, f32):
    """More items than one launch takes (200): the library splits the list;
    every item equals its single call, bit for bit."""
    n, T = 230, 2
    shapes = [(16 + (i % 5), 32 * (1 + i % 4)) for i in range(n)]
    Ws, xs, xqs, ys, refs = [], [], [], [], []
    for i, (N, K) in enumerate(shapes):
        Wg, Wp = weights(2000 + i, N, K, q.W_PACKED)
        x = torch.from_numpy(synth.activations(3000 + i, T, K)).to(DEV)
        xq = q.quantize_q8_0(x, T, K)
        Ws.append(Wp)
        xs.append(x)
        xqs.append(xq)
        ys.append(torch.empty((T, N), dtype=torch.float32, device=DEV))
        refs.append(q.gemv(Wp, q.W_PACKED, xq, N, K, T, ws_for(N, K, T)).cpu())
    if f32:
        items = q.seq_f32_items([(Ws[i], xs[i], ys[i], N, K) for i, (N, K) in enumerate(shapes)])
        q.gemv_seq_f32(items, q.W_PACKED, T, q.new_workspace(q.seq_f32_workspace_bytes(items, T)))
    else:
        items = q.seq_items([(Ws[i], xqs[i], ys[i], N, K) for i, (N, K) in enumerate(shapes)])
        q.gemv_seq(items, q.W_PACKED, T, q.new_workspace(q.seq_workspace_bytes(items, T)))
    torch.cuda.synchronize()
    assert q.device_status() == 0
    for i in range(n):
        assert torch.equal(refs[i].view(torch.int32), ys[i].cpu().view(torch.int32)), i

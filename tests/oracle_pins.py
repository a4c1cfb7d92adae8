"""Pins that tie the CPU oracle to facts outside itself.

Each pin takes a loaded oracle and raises AssertionError on a mismatch.  The
sources are: hand-worked blocks (tests/golden/hand_blocks.json), closed
forms, invariants of the definitions, numpy's binary16 cast (an independent
library implementation of IEEE 754 rounding), and an fp64 dequantise-then-dot
brute force on tiny shapes.  test_oracle_pins.py runs them against the
oracle; it also builds planted-mistake variants of the oracle and checks
that every one of them fails at least one pin.
"""
from __future__ import annotations

import json
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_blocks.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _x_block(entry) -> np.ndarray:
    x = np.zeros(32, np.float32)
    for k, v in entry["x_nonzero"].items():
        x[int(k)] = v
    return x


def _q_block(entry) -> np.ndarray:
    q = np.zeros(32, np.int8)
    for k, v in entry["q_nonzero"].items():
        q[int(k)] = v
    return q


def _xq_bytes(d_bits: int, q: np.ndarray) -> np.ndarray:
    return np.concatenate([np.array([d_bits & 0xFF, d_bits >> 8], np.uint8), q.view(np.uint8)])


def _wq_bytes(d_bits: int, qs) -> np.ndarray:
    return np.concatenate([np.array([d_bits & 0xFF, d_bits >> 8], np.uint8), np.array(qs, np.uint8)])


# ------------------------------------------------------------------ binary16

def pin_half_decode_all(o):
    """Every binary16 pattern decodes like numpy's float16 -> float32 cast."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([o.half_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_half_encode_against_numpy(o):
    """float32 -> binary16 RN-even matches numpy's cast on halfway points,
    neighbours of halfway points, the overflow threshold, subnormals and a
    random sweep (numpy's cast is an independent IEEE implementation)."""
    finite = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (finite[:-1] + finite[1:]) / 2.0          # exact halfway points (fit in fp32)
    cand = np.concatenate([finite, mids]).astype(np.float32)
    up = np.nextafter(cand, np.float32(np.inf))
    dn = np.nextafter(cand, np.float32(0))
    rng = np.random.default_rng(7)
    rand = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000))).astype(np.float32)
    extra = np.array([65519.99, 65520.0, 65536.0, 1e9, 2.0 ** -25, 2.0 ** -24 * 1.5, 5.96e-8], np.float32)
    vals = np.concatenate([cand, up, dn, rand, extra])
    vals = np.concatenate([vals, -vals])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    sample = np.random.default_rng(8).choice(vals.size, size=min(vals.size, 60000), replace=False)
    for i in sample:
        assert o.float_to_half(float(vals[i])) == int(ref[i]), (vals[i], hex(ref[i]))


def pin_half_round_trip(o):
    """encode(decode(h)) == h for every finite binary16, -0 included."""
    for h in list(range(0, 0x7C00)) + list(range(0x8000, 0xFC00)):
        assert o.float_to_half(o.half_to_float(h)) == h, hex(h)


# ------------------------------------------------------------------ Q8_0

def pin_q8_hand_blocks(o):
    for e in golden()["q8_0"]:
        d, q = o.quantize_block(_x_block(e))
        assert d == int(e["d_bits"], 16), (e["name"], hex(d))
        assert np.array_equal(q, _q_block(e)), (e["name"], q)


def pin_q8_constant_block(o):
    """x == c on a whole block gives q == 127 everywhere and d = fp16(c/127)."""
    for c in (1.0, 0.3, 7.25, 1000.0, 1e-3):
        d, q = o.quantize_block(np.full(32, c, np.float32))
        assert np.all(q == 127), (c, q)
        assert d == int(np.float16(np.float32(c) / np.float32(127.0)).view(np.uint16)), c


def pin_q8_symmetry_and_range(o):
    """q(-x) == -q(x) with the same d; |q| <= 127; the amax element maps to +-127."""
    rng = np.random.default_rng(11)
    for _ in range(300):
        x = synth.activations(int(rng.integers(1 << 30)), 1, 32)[0]
        d1, q1 = o.quantize_block(x)
        d2, q2 = o.quantize_block(-x)
        assert d1 == d2 and np.array_equal(q2, -q1)
        assert np.abs(q1.astype(np.int32)).max() == 127
        k = int(np.argmax(np.abs(x)))
        assert abs(int(q1[k])) == 127
    assert o.range_violations() == 0


def pin_q8_power_of_two_scaling(o):
    """Scaling a block by 2^k leaves q unchanged and scales d by 2^k exactly
    while fp16(d) stays a normal number."""
    rng = np.random.default_rng(12)
    for _ in range(100):
        x = (rng.standard_normal(32) * 3).astype(np.float32)
        d0, q0 = o.quantize_block(x)
        for k in (-3, 1, 4):
            d1, q1 = o.quantize_block((x * np.float32(2.0 ** k)).astype(np.float32))
            assert np.array_equal(q0, q1)
            f0 = np.uint16(d0).view(np.float16).astype(np.float64)
            f1 = np.uint16(d1).view(np.float16).astype(np.float64)
            assert f1 == f0 * 2.0 ** k


def pin_q8_layout(o):
    """The T x K quantiser lays blocks out as [t][b] with fp16 d then 32 int8."""
    x = synth.activations(5, 3, 96)
    xq = o.quantize(x)
    assert xq.shape == (3, 3, 34)
    for t in range(3):
        for b in range(3):
            d, q = o.quantize_block(x[t, 32 * b: 32 * b + 32])
            assert int(xq[t, b, 0]) | (int(xq[t, b, 1]) << 8) == d
            assert np.array_equal(xq[t, b, 2:].view(np.int8), q)


# ------------------------------------------------------------------ Q4_0 sums / GEMV

def _hand_xq(name):
    e = [e for e in golden()["q8_0"] if e["name"] == name][0]
    return _xq_bytes(int(e["d_bits"], 16), _q_block(e))


def pin_q4_hand_block(o):
    for e in golden()["q4_0"]:
        w = _wq_bytes(int(e["w_d_bits"], 16), e["w_qs"])
        xq = _hand_xq(e["x_block"])
        assert o.block_isum(w, xq) == e["isum"]
        y, S = o.gemv(w.reshape(1, 18), 1, 32, xq.reshape(1, 1, 34), 1)
        assert y[0, 0] == e["y"]
        assert S[0, 0] == abs(e["y"])


def pin_closed_forms(o):
    for e in golden()["closed_forms"]:
        K = e["K"]
        W = synth.with_nibbles(synth.q4_0_weights(1, 4, K), K, e["nibble"])
        W = synth.with_scales(W, K, int(e["w_d_bits"], 16))
        x = np.full((1, K), e["x_value"], np.float32)
        xq = o.quantize(x)
        y, S = o.gemv(W, 4, K, xq, 1)
        assert np.all(y == e["y"]), (e["name"], y)
        if "isum" in e:
            assert np.all(o.block_isums(W, 4, K, xq, 1) == e["isum"])


def pin_zero_scale(o):
    """A zero weight scale gives y == 0 (and argmax 0 on an all-zero output)."""
    K = 128
    W = synth.with_scales(synth.q4_0_weights(2, 8, K), K, 0x0000)
    xq = o.quantize(synth.activations(3, 2, K))
    y, S = o.gemv(W, 8, K, xq, 2)
    assert np.all(y == 0.0) and np.all(S == 0.0)
    assert o.argmax_f32(y[0].astype(np.float32)) == 0


def pin_nibble_complement(o):
    """Replacing every nibble n by 15-n maps isum to -isum - sum(q) (from
    (15-n-8) = -(n-8) - 1)."""
    K = 256
    W = synth.q4_0_weights(4, 6, K)
    Wc = W.copy().reshape(6, K // 32, 18)
    Wc[:, :, 2:] = 0xFF - Wc[:, :, 2:]
    Wc = Wc.reshape(W.shape)
    xq = o.quantize(synth.activations(5, 2, K))
    i1 = o.block_isums(W, 6, K, xq, 2).astype(np.int64)
    i2 = o.block_isums(Wc, 6, K, xq, 2).astype(np.int64)
    qsum = xq[:, :, 2:].view(np.int8).astype(np.int64).sum(axis=2)      # [T, nb]
    assert np.array_equal(i2, -i1 - qsum[:, None, :])


def _dequant_f64(W, N, K):
    """Brute force: every weight as (n - 8) * d in fp64, [N, K]."""
    nb = K // 32
    blk = W.reshape(N, nb, 18)
    d = blk[:, :, 0:2].copy().view("<f2").astype(np.float64)[:, :, 0]
    qs = blk[:, :, 2:]
    n = np.concatenate([qs & 0x0F, qs >> 4], axis=2).astype(np.float64)  # elements 0..15, 16..31
    return ((n - 8.0) * d[:, :, None]).reshape(N, K)


def _dequant_x_f64(xq, T, K):
    nb = K // 32
    d = xq[:, :, 0:2].copy().view("<f2").astype(np.float64)[:, :, 0]
    q = xq[:, :, 2:].view(np.int8).astype(np.float64)
    return (q * d[:, :, None]).reshape(T, K)


def pin_bruteforce_dequant_dot(o):
    """Dequantise both operands to fp64 and take numpy's dot: equals y64."""
    rng = np.random.default_rng(13)
    for trial in range(24):
        N = int(rng.integers(1, 48))
        K = 32 * int(rng.integers(1, 9))
        T = int(rng.integers(1, 9))
        W = synth.q4_0_weights(100 + trial, N, K)
        x = synth.activations(200 + trial, T, K)
        xq = o.quantize(x)
        y, S = o.gemv(W, N, K, xq, T)
        ref = _dequant_x_f64(xq, T, K) @ _dequant_f64(W, N, K).T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * max(1.0, float(np.abs(ref).max())))
        assert np.all(S >= np.abs(y) - 1e-9)


def pin_row_permutation(o):
    K, N, T = 192, 20, 3
    W = synth.q4_0_weights(21, N, K)
    xq = o.quantize(synth.activations(22, T, K))
    perm = np.random.default_rng(23).permutation(N)
    y, _ = o.gemv(W, N, K, xq, T)
    yp, _ = o.gemv(np.ascontiguousarray(W[perm]), N, K, xq, T)
    assert np.array_equal(yp, y[:, perm])


def pin_token_columns_independent(o):
    """Column t of a T-token GEMV equals the 1-token GEMV of that column."""
    K, N, T = 160, 24, 5
    W = synth.q4_0_weights(31, N, K)
    xq = o.quantize(synth.activations(32, T, K))
    y, S = o.gemv(W, N, K, xq, T)
    for t in range(T):
        y1, S1 = o.gemv(W, N, K, np.ascontiguousarray(xq[t:t + 1]), 1)
        assert np.array_equal(y1[0], y[t]) and np.array_equal(S1[0], S[t])


def pin_rows_subset(o):
    K, N, T = 96, 30, 2
    W = synth.q4_0_weights(41, N, K)
    xq = o.quantize(synth.activations(42, T, K))
    y, S = o.gemv(W, N, K, xq, T)
    rows = np.array([0, 7, 29, 3])
    yr, Sr = o.gemv_rows(W, N, K, xq, T, rows)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(Sr, S[:, rows])


def pin_scale_linearity(o):
    """Doubling every weight scale (exact in fp16) doubles y64 exactly."""
    K, N = 128, 10
    W = synth.q4_0_weights(51, N, K)
    W2 = W.copy().reshape(N, K // 32, 18)
    d = W2[:, :, 0:2].copy().view("<f2")[:, :, 0]
    W2[:, :, 0:2] = (d.astype(np.float32) * 2).astype("<f2").view(np.uint8).reshape(N, K // 32, 2)
    W2 = W2.reshape(W.shape)
    xq = o.quantize(synth.activations(52, 1, K))
    y1, _ = o.gemv(W, N, K, xq, 1)
    y2, _ = o.gemv(W2, N, K, xq, 1)
    assert np.array_equal(y2, 2 * y1)


# ------------------------------------------------------------------ argmax

def pin_argmax_rules(o):
    assert o.argmax_f32(np.array([1, 3, 3, 2], np.float32)) == 1
    assert o.argmax_f32(np.array([-0.0, 0.0, -1.0], np.float32)) == 0
    assert o.argmax_f32(np.array([-1.0, 0.0, -0.0], np.float32)) == 1
    assert o.argmax_f32(np.zeros(9, np.float32)) == 0
    assert o.argmax_f32(np.array([-5.0, -2.0, -2.0, -7.0], np.float32)) == 1
    y = np.random.default_rng(61).standard_normal(1000).astype(np.float32)
    y[[100, 400, 900]] = y.max() + 1
    assert o.argmax_f32(y) == 100
    assert o.argmax_f64(np.array([2.0, 5.0, 5.0], np.float64)) == 1


# ------------------------------------------------------------------ Q8_0 weights

def _q8w_bytes(d_bits: int, w) -> np.ndarray:
    """One 34-byte Q8_0 weight block: fp16 d (little-endian), then 32 int8."""
    return np.concatenate([np.array([d_bits & 0xFF, d_bits >> 8], np.uint8),
                           np.asarray(w, np.int8).view(np.uint8)])


def pin_q8w_hand_block(o):
    # weights: w0 = 3, w1 = -2, w31 = 127, rest 0; activations q0 = 10, q1 = 7,
    # q31 = -127, rest 0: isum = 30 - 14 - 16129 = -16113 (worked by hand)
    w = np.zeros(32, np.int8); w[0], w[1], w[31] = 3, -2, 127
    qx = np.zeros(32, np.int8); qx[0], qx[1], qx[31] = 10, 7, -127
    wb, xb = _q8w_bytes(0x3800, w), _xq_bytes(0x3C00, qx)          # d_w = 0.5, d_x = 1
    assert o.block_isum_q8(wb, xb) == -16113
    y, S = o.gemv_q8(wb, 1, 32, xb, 1)
    assert y[0, 0] == -8056.5 and S[0, 0] == 8056.5


def pin_q8w_closed_forms_and_range(o):
    K, nb = 1536, 48
    for c in (-128, -127, -1, 0, 1, 127):
        W = np.tile(_q8w_bytes(0x3C00, np.full(32, c, np.int8)), nb)   # d_w = 1
        x = np.full((1, K), 127.0, np.float32)                         # every q = 127, d_x = 1
        xq = o.quantize(x)
        y, _ = o.gemv_q8(W, 1, K, xq, 1)
        assert y[0, 0] == nb * 32 * 127 * c
        assert o.block_isum_q8(W[:34], xq.reshape(-1, 34)[0]) == 32 * 127 * c
    # the range extreme: -128 * -127 * 32
    xb = _xq_bytes(0x3C00, np.full(32, -127, np.int8))
    assert o.block_isum_q8(_q8w_bytes(0x3C00, np.full(32, -128, np.int8)), xb) == 520192


def pin_q8w_from_q4_blocks(o):
    """A Q4_0 block rewritten as Q8_0 weights (w = n - 8, same d) gives the
    same integer sums and outputs as the Q4_0 path (pinned separately)."""
    N, K, T = 7, 256, 3
    import synth
    W4 = synth.q4_0_weights(81, N, K).reshape(N, K // 32, 18)
    lo, hi = W4[:, :, 2:] & 0x0F, W4[:, :, 2:] >> 4
    n = np.concatenate([lo, hi], axis=2).astype(np.int16)            # elements 0..15, 16..31
    W8 = np.empty((N, K // 32, 34), np.uint8)
    W8[:, :, :2] = W4[:, :, :2]
    W8[:, :, 2:] = (n - 8).astype(np.int8).view(np.uint8)
    xq = o.quantize(synth.activations(82, T, K))
    assert np.array_equal(o.block_isums_q8(W8.reshape(N, -1), N, K, xq, T),
                          o.block_isums(W4.reshape(N, -1), N, K, xq, T))
    y8, S8 = o.gemv_q8(W8.reshape(N, -1), N, K, xq, T)
    y4, S4 = o.gemv(W4.reshape(N, -1), N, K, xq, T)
    assert np.array_equal(y8, y4) and np.array_equal(S8, S4)


def pin_q8w_bruteforce_dequant_dot(o):
    import synth
    rng = np.random.default_rng(83)
    for _ in range(10):
        N, K, T = int(rng.integers(1, 40)), 32 * int(rng.integers(1, 9)), int(rng.integers(1, 9))
        W = synth.q8_0_weights(int(rng.integers(1 << 30)), N, K)
        x = synth.activations(int(rng.integers(1 << 30)), T, K)
        xq = o.quantize(x)
        blk = W.reshape(N, K // 32, 34)
        dw = blk[:, :, :2].copy().view("<f2").astype(np.float64)[:, :, 0]
        wf = blk[:, :, 2:].view(np.int8).astype(np.float64) * dw[:, :, None]
        xf = _dequant_x_f64(xq, T, K)
        ref = xf @ wf.reshape(N, K).T
        y, S = o.gemv_q8(W, N, K, xq, T)
        assert np.all(np.abs(y - ref) <= 1e-12 * np.maximum(S, 1e-30))


# ------------------------------------------------------------------ FFN chain

def pin_exp_against_libm(o):
    """Cody-Waite exp against numpy's fp64 exp: within 2 ulp over [-87, 88]."""
    x = np.linspace(-87.0, 88.0, 400001).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 1e-8, -1e-8, 0.5, -0.5], np.float32)])
    e = o.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(e - ref) <= 2 * ulp)
    assert o.exp_f32(np.array([0.0], np.float32))[0] == 1.0
    assert np.all(np.diff(o.exp_f32(np.sort(x))) >= 0)        # monotone


def pin_silu_identities(o):
    g = np.linspace(-40.0, 40.0, 100001).astype(np.float32)
    s, sm = o.silu_f32(g).astype(np.float64), o.silu_f32(-g).astype(np.float64)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    assert np.all(np.abs(s - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32)) + 1e-30)
    # silu(g) - silu(-g) = g
    assert np.all(np.abs((s - sm) - g) <= 8 * np.spacing(np.abs(g)) + 1e-30)
    assert o.silu_f32(np.array([0.0], np.float32))[0] == 0.0


def pin_silu_mul_quantize_against_fp64(o):
    """Dequantised codes of SiLU(g) * u within half a quantisation step (plus
    the fp32 rounding of h) of the fp64 value; token-major blocks."""
    rng = np.random.default_rng(91)
    T, F = 3, 512
    g = (rng.standard_normal((T, F)) * 3).astype(np.float32)
    u = rng.standard_normal((T, F)).astype(np.float32)
    hq, h = o.silu_mul_quantize(g, u)
    h64 = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64))) * u
    assert np.all(np.abs(h - h64) <= 8 * np.spacing(np.abs(h64).astype(np.float32)) + 1e-30)
    d = hq[:, :, 0:2].copy().view("<f2").astype(np.float64)          # [T, F/32, 1]
    q = hq[:, :, 2:].view(np.int8).astype(np.float64)
    deq = (q * d).reshape(T, F)
    step = np.repeat(d[:, :, 0], 32, axis=1)
    assert np.all(np.abs(deq - h64) <= 0.5 * step * (1 + 1e-3) + 1e-3 * np.abs(h64) + 1e-12)
    assert np.array_equal(hq, o.quantize(h))                          # the quantiser of x, applied to h


# ------------------------------------------------------------------ top-2

def _top2_by_sort(y):
    """The first two rows in (larger value, lower index) order, by a library
    sort; Python compares -0.0 == 0.0, so the tie rule is IEEE equality."""
    order = sorted(range(len(y)), key=lambda i: (-float(y[i]), i))
    return order[0], (order[1] if len(order) > 1 else -1)


def pin_top2_rules(o):
    assert o.top2_f32(np.array([1, 3, 3, 2], np.float32)) == (1, 2)
    assert o.top2_f32(np.array([4, 1, 3, 3], np.float32)) == (0, 2)
    assert o.top2_f32(np.array([-0.0, 0.0, -1.0], np.float32)) == (0, 1)
    assert o.top2_f32(np.array([0.0, -1.0, -0.0], np.float32)) == (0, 2)
    assert o.top2_f32(np.array([2.5], np.float32)) == (0, -1)
    assert o.top2_f32(np.zeros(9, np.float32)) == (0, 1)
    assert o.top2_f32(np.array([-5.0, -2.0, -9.0, -2.0], np.float32)) == (1, 3)
    assert o.top2_f64(np.array([2.0, 5.0, 5.0, 7.0], np.float64)) == (3, 1)


def pin_top2_against_sort(o):
    rng = np.random.default_rng(62)
    for n in (2, 3, 17, 1000):
        for _ in range(20):
            # few distinct values, so ties are frequent; some zeros of both signs
            y = rng.integers(-3, 4, n).astype(np.float32)
            y[rng.random(n) < 0.2] = -0.0
            assert o.top2_f32(y) == _top2_by_sort(y)
            y64 = y.astype(np.float64) * 0.5
            assert o.top2_f64(y64) == _top2_by_sort(y64)


# ------------------------------------------------------------------ verify-commit

def pin_verify_commit_hand_cases(o):
    # tokens = [current, draft1, draft2, draft3]; pred[t] follows tokens[0..t]
    pred = [7, 9, 11, 4]
    assert o.verify_commit([5, 7, 9, 11], pred) == 4    # every draft right: all four commit
    assert o.verify_commit([5, 8, 9, 11], pred) == 1    # first draft wrong: pred[0] only
    assert o.verify_commit([5, 7, 10, 11], pred) == 2   # second wrong: pred[0], pred[1]
    assert o.verify_commit([5, 7, 0, 11], pred) == 2    # a later match after a miss does not count
    assert o.verify_commit([5], [7]) == 1               # plain decode step


def pin_verify_commit_is_lossless(o):
    """The committed tokens are exactly what plain greedy decoding emits, and
    as many as the drafts allow (a toy deterministic model stands in for the
    lm_head: next token = a hash of the whole prefix)."""
    def nxt(prefix):
        h = 1469598103934665603
        for tok in prefix:
            h = ((h ^ tok) * 1099511628211) % (1 << 61)
        return h % 13

    rng = np.random.default_rng(63)
    for _ in range(300):
        prefix = [int(v) for v in rng.integers(0, 13, rng.integers(1, 6))]
        greedy = []
        for _ in range(8):
            greedy.append(nxt(prefix + greedy))
        T = int(rng.integers(1, 9))
        # drafts: the greedy continuation with some tokens replaced
        drafts = [g if rng.random() < 0.7 else int(rng.integers(0, 13)) for g in greedy[:T - 1]]
        tokens = [prefix[-1]] + drafts
        pred = [nxt(prefix + drafts[:t]) for t in range(T)]
        n = o.verify_commit(tokens, pred)
        assert pred[:n] == greedy[:n]
        right = 0
        while right < T - 1 and drafts[right] == greedy[right]:
            right += 1
        assert n == right + 1


# --------------------------------------------- Q4_0 requantisation at load
# The encoder (reading: the GGML q4_0 encoder; minfer README M14 and M18
# requantise heads to q4_0 at load) must invert the block format's decoder
# on every block it can represent, keep its error within half a step, place
# the block's extreme at code 0, and commute with power-of-two scaling.

def _q4_decode(blk: np.ndarray) -> np.ndarray:
    """fp64 values of one 18-byte Q4_0 block, from the format's definition."""
    d = float(blk[:2].view(np.float16)[0])
    n = np.concatenate([blk[2:] & 0x0F, blk[2:] >> 4]).astype(np.float64)
    return (n - 8.0) * d, n.astype(int), d


def _q4_block(d_bits: int, n) -> np.ndarray:
    n = np.asarray(n, np.uint8)
    return np.concatenate([np.array([d_bits & 0xFF, d_bits >> 8], np.uint8), (n[:16] | (n[16:] << 4)).astype(np.uint8)])


def pin_q4enc_hand_blocks(o):
    # Worked by hand.  A: the first element of largest magnitude is x[3] = 8,
    # so d = 8 / -8 = -1 (fp16 0xBC00) and 1/d = -1; codes floor(-x + 8.5):
    # 8 -> 0, -8 -> 16 -> clamped 15, -4 -> 12, 2 -> 6, 3.75 -> 4, 0 -> 8.
    x = np.zeros(32, np.float32)
    x[[0, 1, 2, 3, 9]] = [-4.0, 2.0, 3.75, 8.0, -8.0]
    n = [8] * 32
    n[0], n[1], n[2], n[3], n[9] = 12, 6, 4, 0, 15
    assert np.array_equal(o.quantize_block_q4_0(x), _q4_block(0xBC00, n))
    # B: the tie goes the other way (x[3] = -8 first), so d = 1 (0x3C00):
    # codes floor(x + 8.5): -8 -> 0, 8 -> 15, -4 -> 4, 2 -> 10, 3.75 -> 12.
    x[3], x[9] = -8.0, 8.0
    n[0], n[1], n[2], n[3], n[9] = 4, 10, 12, 0, 15
    assert np.array_equal(o.quantize_block_q4_0(x), _q4_block(0x3C00, n))
    # C: m = -1.6e-39 (an fp32 subnormal), d = m / -8 about 2e-40, whose
    # reciprocal (5e39) overflows to +inf; x * inf + 8.5 is -inf for x < 0
    # (code 0), +inf for x > 0 (code 15) and NaN for x = 0 (code 0); d
    # underflows to fp16 +0.
    x = np.zeros(32, np.float32)
    x[0], x[1] = np.float32(-1.6e-39), np.float32(1e-40)
    n = [0] * 32
    n[1] = 15
    assert np.array_equal(o.quantize_block_q4_0(x), _q4_block(0x0000, n))


def pin_q4enc_round_trip(o):
    """Every block holding code 0 (its unique extreme value -8d) decodes to
    fp32 values that encode back to the same 18 bytes."""
    rng = np.random.default_rng(1410)
    for i in range(600):
        mag = rng.choice([rng.uniform(1e-3, 4.0), rng.uniform(6e-8, 6e-5), rng.uniform(1.0, 8000.0)])
        d16 = np.float16(mag * rng.choice([-1.0, 1.0]))
        if d16 == 0:
            continue
        n = rng.integers(0, 16, 32)
        n[rng.integers(0, 32, rng.integers(1, 4))] = 0
        blk = _q4_block(int(np.array([d16]).view(np.uint16)[0]), n)
        vals, _, _ = _q4_decode(blk)
        x = vals.astype(np.float32)
        assert np.array_equal(x.astype(np.float64), vals)          # exact in fp32
        assert np.array_equal(o.quantize_block_q4_0(x), blk), i


def pin_q4enc_error_and_extreme(o):
    rng = np.random.default_rng(1411)
    for i in range(400):
        x = (rng.standard_normal(32) * rng.choice([1e-3, 0.05, 1.0, 30.0])).astype(np.float32)
        if i % 3 == 0:
            x[rng.integers(0, 32)] *= 6.0                              # an outlier
        if i % 5 == 0:
            x[rng.integers(0, 32)] = -x[np.argmax(np.abs(x))]          # the extreme's opposite
        vals, n, d = _q4_decode(o.quantize_block_q4_0(x))
        x64 = x.astype(np.float64)
        first = int(np.argmax(np.abs(x64)))                            # first of the largest magnitude
        assert n[first] == 0
        assert abs(d - (-x64[first] / 8.0)) <= 2.0 ** -11 * abs(x64[first] / 8.0)
        err = np.abs(x64 - vals)
        step = abs(d) * (1.0 + 2.0 ** -10)
        assert np.all(err[n < 15] <= 0.5045 * step), i
        assert np.all(err[n == 15] <= 1.0045 * step), i


def pin_q4enc_zero_and_power_of_two_scaling(o):
    vals, n, d = _q4_decode(o.quantize_block_q4_0(np.zeros(32, np.float32)))
    assert d == 0.0 and np.all(n == 8) and np.all(vals == 0.0)
    rng = np.random.default_rng(1412)
    for i in range(100):
        x = rng.standard_normal(32).astype(np.float32)
        base = o.quantize_block_q4_0(x)
        for k in (-6, -1, 3, 9):
            sc = o.quantize_block_q4_0((x * np.float32(2.0 ** k)).astype(np.float32))
            assert np.array_equal(sc[2:], base[2:]), (i, k)
            d0 = float(base[:2].view(np.float16)[0])
            assert float(sc[:2].view(np.float16)[0]) == d0 * 2.0 ** k


def pin_q8_to_q4_exact_blocks(o):
    """Q8_0 blocks whose codes are (n - 8) * s for an integer s requantise to
    Q4_0 codes n with d = s * d8 (exact in fp32), stored as numpy's fp16."""
    rng = np.random.default_rng(1413)
    N, K = 3, 256
    nb = K // 32
    q8 = np.empty((N, nb, 34), np.uint8)
    expect = np.empty((N, nb, 18), np.uint8)
    for r in range(N):
        for b in range(nb):
            n = rng.integers(0, 16, 32)
            n[rng.integers(0, 32)] = 0
            s = int(rng.integers(1, 16))
            d8 = np.float16(rng.uniform(1e-4, 0.5) * rng.choice([-1.0, 1.0]))
            q8[r, b, :2] = np.array([d8]).view(np.uint8)
            q8[r, b, 2:] = ((n - 8) * s).astype(np.int8).view(np.uint8)
            dq = np.float16(np.float32(s) * np.float32(d8))
            expect[r, b] = _q4_block(int(np.array([dq]).view(np.uint16)[0]), n)
    got = o.requant_q8_0_q4_0(q8.reshape(N, -1), N, K)
    assert np.array_equal(got.reshape(N, nb, 18), expect)
    # and the fp32 entry point agrees block for block on the decoded values
    x = (q8[:, :, 2:].view(np.int8).astype(np.float32) *
         q8[:, :, :2].copy().view(np.float16).astype(np.float32)).reshape(N, K)
    assert np.array_equal(o.requant_f32_q4_0(x, N, K), got)


# ---------------------------------------------------- sequence epilogue
# y = W.x + bias + residual (minfer README M19: bias and residual adds in the
# GEMVs' epilogues).  Zero-scale weight blocks make W.x exactly 0, so the
# output is the bias plus the residual, exactly (both fp32, their fp64 sum
# exact); without the terms the output is the plain GEMV's.

def pin_epilogue_closed_forms(o):
    rng = np.random.default_rng(1500)
    N, K, T = 40, 96, 3
    W = synth.q4_0_weights(1501, N, K).reshape(N, K // 32, 18).copy()
    W[:, :, 0:2] = 0                                            # d = +0: every weight is 0
    x = rng.standard_normal((T, K)).astype(np.float32)
    xq = o.quantize(x)
    bias = rng.standard_normal(N).astype(np.float32)
    res = rng.standard_normal((T, N)).astype(np.float32)
    y, S = o.gemv_ep(W.reshape(N, -1), N, K, xq, T, bias, res)
    assert np.array_equal(y, bias.astype(np.float64)[None, :] + res.astype(np.float64))
    assert np.array_equal(S, np.abs(bias.astype(np.float64))[None, :] + np.abs(res.astype(np.float64)))
    yb, _ = o.gemv_ep(W.reshape(N, -1), N, K, xq, T, bias, None)
    assert np.array_equal(yb, np.broadcast_to(bias.astype(np.float64), (T, N)))
    Wr = synth.q4_0_weights(1502, N, K)
    y0, S0 = o.gemv(Wr, N, K, xq, T)
    y1, S1 = o.gemv_ep(Wr, N, K, xq, T, None, None)
    assert np.array_equal(y0, y1) and np.array_equal(S0, S1)


# ------------------------------------ gs64 planar int4, per-vector int8
# (colibri qwen36 docs: 64-weight groups with one scale, repacked so that one
# AND and one shift give a group's two halves in order; activations
# quantised once per vector with amax / 127.)

def _gs64_decode_f64(Wq, Ws, N, K):
    """fp64 weights [N][K] from the layout's definition: byte j of a group
    holds element j (low nibble) and element j + 32 (high nibble)."""
    g = Wq.reshape(N, K // 64, 32)
    n = np.concatenate([g & 0x0F, g >> 4], axis=2).astype(np.float64)     # [N][G][64]
    return ((n - 8.0) * Ws.reshape(N, K // 64, 1).astype(np.float64)).reshape(N, K)


def pin_gs64_hand_group(o):
    # one group: every code 8 (weight 0) except element 33 = 15 (weight 7 s);
    # element 33 is the high nibble of byte 1.  q = 1 everywhere but q[33] = 5:
    # isum = 7 * 5 = 35, y = s_w * s_x * 35 exactly.
    Wq = np.full((1, 32), 0x88, np.uint8)
    Wq[0, 1] = 0xF8
    Ws = np.array([[0.375]], np.float32)
    q = np.ones((1, 64), np.int8)
    q[0, 33] = 5
    y, S = o.gemv_gs64(Wq, Ws, 1, 64, q, np.array([2.0], np.float32))
    assert y[0, 0] == 0.375 * 2.0 * 35 and S[0, 0] == abs(y[0, 0])


def pin_gs64_bruteforce(o):
    rng = np.random.default_rng(1600)
    for N, K, T in [(3, 64, 1), (5, 256, 3), (2, 640, 2)]:
        Wq = rng.integers(0, 256, (N, K // 64 * 32)).astype(np.uint8)
        Ws = rng.uniform(-0.02, 0.02, (N, K // 64)).astype(np.float32)
        q = rng.integers(-127, 128, (T, K)).astype(np.int8)
        s = rng.uniform(1e-3, 1e-1, T).astype(np.float32)
        y, _ = o.gemv_gs64(Wq, Ws, N, K, q, s)
        ref = (q.astype(np.float64) * s.astype(np.float64)[:, None]) @ _gs64_decode_f64(Wq, Ws, N, K).T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-15), (N, K, T)


def pin_vec_i8_quantiser(o):
    rng = np.random.default_rng(1601)
    x = (rng.standard_normal((4, 1000)) * np.array([[1e-3], [1.0], [50.0], [3.0]])).astype(np.float32)
    x[3, 500] = -40.0                                   # the extreme late in the vector
    q, s = o.quantize_vec_i8(x)
    for t in range(4):
        a = int(np.argmax(np.abs(x[t])))
        assert abs(int(q[t, a])) == 127 and np.sign(q[t, a]) == np.sign(x[t, a])
        assert s[t] == np.float32(np.max(np.abs(x[t])) / np.float32(127.0))
        err = np.abs(x[t].astype(np.float64) - q[t].astype(np.float64) * float(s[t]))
        assert np.all(err <= 0.5 * float(s[t]) * (1 + 1e-5)), t
    q2, s2 = o.quantize_vec_i8(-x)
    assert np.array_equal(q2, -q) and np.array_equal(s2, s)
    q3, s3 = o.quantize_vec_i8((x * np.float32(2.0 ** -5)).astype(np.float32))
    assert np.array_equal(q3, q) and np.array_equal(s3, (s * np.float32(2.0 ** -5)).astype(np.float32))
    qz, sz = o.quantize_vec_i8(np.zeros((1, 64), np.float32))
    assert sz[0] == 0.0 and not qz.any()


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

"""Seeded synthetic inputs for the Q4_0 x Q8_0 decode GEMV.

This module only draws random numbers and lays them out as bytes. It holds
none of the method's arithmetic (no quantisation, no dot products), so both
the CPU oracle's tests and the CUDA path's tests and benchmark can take their
inputs from here without sharing any of the computation.

Generator: numpy's ``Generator(PCG64)`` (O'Neill's PCG family, 128-bit LCG
with an XSL-RR output permutation), seeded through ``SeedSequence`` so that
every matrix / vector of a workload gets its own independent stream.

Value recipe (the same for every workload):
  * Q4_0 weights, GGML block layout: per block of 32 weights an fp16 scale
    ``d`` (little-endian) followed by 16 bytes of nibbles.  Every nibble is
    uniform on 0..15 (so every nibble byte is uniform on 0..255); ``d`` is
    uniform real on [1e-3, 4e-3], rounded once to binary16 (round to nearest
    even, numpy's cast).
  * Activations x: fp32, standard normal drawn in fp64 and cast once; each
    entry independently (Bernoulli p = 0.01) multiplied by 20 (outliers).
    Token columns are independent.
  * Expert ids: k distinct ids out of n_experts per token (uniform subset,
    drawn without replacement).
  * gs64 grouped int4 weights (64 weights per group in 32 nibble bytes, one
    fp32 scale): nibble bytes uniform on 0..255, scales uniform real on
    [1e-3, 4e-3] kept in fp32.
"""
from __future__ import annotations

import numpy as np

Q4_0_BLOCK_BYTES = 18      # fp16 scale + 16 nibble bytes
QK = 32                    # weights per block

SCALE_LO, SCALE_HI = 1e-3, 4e-3
OUTLIER_P, OUTLIER_MUL = 0.01, 20.0


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, stream)])))


def q4_0_weights(seed: int, N: int, K: int, stream: tuple = ()) -> np.ndarray:
    """Random Q4_0 matrix in GGML row-major block layout, uint8 [N, K/32*18]."""
    assert K % QK == 0 and N >= 0
    nb = K // QK
    rng = _rng(seed, 1, *stream)
    blocks = np.empty((N, nb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    scales = rng.uniform(SCALE_LO, SCALE_HI, size=(N, nb)).astype(np.float16)
    blocks[:, :, 0:2] = scales.astype("<f2").view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = rng.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    return blocks.reshape(N, nb * Q4_0_BLOCK_BYTES)


def q8_0_weights(seed: int, N: int, K: int, stream: tuple = ()) -> np.ndarray:
    """Random Q8_0 weight matrix in GGML row-major block layout, uint8 [N, K/32*34]:
    fp16 scales as for Q4_0, int8 values uniform on [-127, 127]."""
    assert K % QK == 0 and N >= 0
    nb = K // QK
    rng = _rng(seed, 4, *stream)
    blocks = np.empty((N, nb, 34), dtype=np.uint8)
    scales = rng.uniform(SCALE_LO, SCALE_HI, size=(N, nb)).astype(np.float16)
    blocks[:, :, 0:2] = scales.astype("<f2").view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:] = rng.integers(-127, 128, size=(N, nb, 32)).astype(np.int8).view(np.uint8)
    return blocks.reshape(N, nb * 34)


def gs64_weights(seed: int, N: int, K: int, stream: tuple = ()):
    """Random gs64 grouped int4 matrix as its two row planes: nibble bytes
    uint8 [N, K/64, 32] (every byte uniform on 0..255, so every nibble is
    uniform on 0..15) and fp32 group scales [N, K/64] uniform real on
    [1e-3, 4e-3] (drawn in fp64, cast once)."""
    assert K % 64 == 0 and N >= 0
    ng = K // 64
    rng = _rng(seed, 6, *stream)
    wq = rng.integers(0, 256, size=(N, ng, 32), dtype=np.uint8)
    ws = rng.uniform(SCALE_LO, SCALE_HI, size=(N, ng)).astype(np.float32)
    return wq, ws


def f32_weights(seed: int, N: int, K: int, stream: tuple = ()) -> np.ndarray:
    """fp32 weight matrix [N, K] before quantisation: N(0, s_r^2) per row r,
    s_r log-uniform on [0.005, 0.1], with 1 % of entries scaled by 20."""
    rng = _rng(seed, 5, *stream)
    s = np.exp(rng.uniform(np.log(0.005), np.log(0.1), size=(N, 1)))
    w = rng.standard_normal(size=(N, K)) * s
    mask = rng.random(size=(N, K)) < OUTLIER_P
    w[mask] *= OUTLIER_MUL
    return w.astype(np.float32)


def activations(seed: int, T: int, K: int, stream: tuple = ()) -> np.ndarray:
    """fp32 [T, K]: N(0,1) with 1 % of entries scaled by 20."""
    rng = _rng(seed, 2, *stream)
    x = rng.standard_normal(size=(T, K))
    mask = rng.random(size=(T, K)) < OUTLIER_P
    x[mask] *= OUTLIER_MUL
    return x.astype(np.float32)


def expert_ids(seed: int, n_tokens: int, n_experts: int, k: int, stream: tuple = ()) -> np.ndarray:
    """int32 [n_tokens, k]: per token k distinct expert ids."""
    rng = _rng(seed, 3, *stream)
    out = np.empty((n_tokens, k), dtype=np.int32)
    for t in range(n_tokens):
        out[t] = rng.choice(n_experts, size=k, replace=False)
    return out


def with_scales(W: np.ndarray, K: int, scale_bits: int) -> np.ndarray:
    """Copy of a GGML Q4_0 matrix with every block scale set to one fp16 bit pattern."""
    nb = K // QK
    out = W.copy().reshape(W.shape[0], nb, Q4_0_BLOCK_BYTES)
    out[:, :, 0] = scale_bits & 0xFF
    out[:, :, 1] = (scale_bits >> 8) & 0xFF
    return out.reshape(W.shape)


def with_nibbles(W: np.ndarray, K: int, nibble: int) -> np.ndarray:
    """Copy of a GGML Q4_0 matrix with every nibble set to one value 0..15."""
    nb = K // QK
    out = W.copy().reshape(W.shape[0], nb, Q4_0_BLOCK_BYTES)
    out[:, :, 2:] = (nibble & 0xF) * 0x11
    return out.reshape(W.shape)


# ---------------------------------------------------------------------------
# Workload shapes.  Each GEMV is (name, N rows, K inner).  Per-layer sets are
# the fused-QKV / O / gate / up / down projections of the named decoder sizes.
# ---------------------------------------------------------------------------

QWEN25_1P5B_LAYER = [("qkv", 2048, 1536), ("o", 1536, 1536), ("gate", 8960, 1536),
                     ("up", 8960, 1536), ("down", 1536, 8960)]
QWEN25_3B_LAYER = [("qkv", 2560, 2048), ("o", 2048, 2048), ("gate", 11008, 2048),
                   ("up", 11008, 2048), ("down", 2048, 11008)]

WORKLOADS = {
    # single 1536x1536 GEMV, T=1, activation quantisation included
    "single_1536": dict(kind="single", N=1536, K=1536, T=1, seed=0),
    # 28-layer Qwen2.5-1.5B-shaped layer set, T=1, in layer order
    "qwen2.5-1.5b_layerset": dict(kind="seq", layer=QWEN25_1P5B_LAYER, layers=28, T=1, seed=1000),
    # the same with the decode step's epilogues: bias on qkv, a residual added to o and down
    "qwen2.5-1.5b_layerset_ep": dict(kind="seq", layer=QWEN25_1P5B_LAYER, layers=28, T=1, seed=1000,
                                     epilogue=True),
    # lm_head 151936x1536 with fused argmax, 4 weight copies in rotation
    "lm_head_argmax": dict(kind="argmax", N=151936, K=1536, T=1, copies=4, seed=2000),
    # lm_head verify step: 8 positions (current token + 7 drafts), top-2 rows
    # per position, then the commit rule; 4 weight copies in rotation
    "lm_head_top2_verify": dict(kind="verify", N=151936, K=1536, T=8, copies=4, seed=2100),
    # the decode FFN of the 28 Qwen2.5-1.5B layers: gate and up 8960x1536 on
    # the same x, SiLU(gate) * up quantised to Q8_0, down 1536x8960; T=1
    "qwen2.5-1.5b_ffn": dict(kind="ffn", d_model=1536, d_ff=8960, layers=28, T=1, seed=5000),
    # the lm_head held as Q8_0 weights (248 MB per copy), T=1, 2 copies in rotation
    "q8_lm_head": dict(kind="q8", N=151936, K=1536, T=1, copies=2, seed=2200),
    # a dense matrix of the lm_head's shape in the gs64 grouped int4 format,
    # per-vector int8 activations, T=1, 4 copies in rotation
    "gs64_lm_head": dict(kind="gs64", N=151936, K=1536, T=1, copies=4, seed=2400),
    # load-time requantisation of that Q8_0 lm_head to Q4_0
    "lm_head_requant_q8": dict(kind="requant", N=151936, K=1536, T=1, copies=2, seed=2300),
    # 36-layer Qwen2.5-3B-shaped layer set, T in {1,2,4,8}
    "qwen2.5-3b_verify": dict(kind="seq", layer=QWEN25_3B_LAYER, layers=36, Ts=(1, 2, 4, 8), seed=3000),
    # MoE: 256 experts (gate/up 512x2048, down 2048x512), top-8 + 1 shared, T=1
    "moe_top8_shared": dict(kind="moe", n_experts=256, top_k=8, d_model=2048, d_ff=512,
                            sets=4, T=1, seed=4000),
}


def layer_set(layer: list, layers: int) -> list:
    """Flattened list of (name, N, K) for `layers` repetitions, in layer order."""
    return [(f"L{l}.{name}", N, K) for l in range(layers) for (name, N, K) in layer]

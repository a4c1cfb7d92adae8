"""Benchmark of the Q4_0 x Q8_0 decode GEMV path on one GB300.

Default workload: the 28-layer Qwen2.5-1.5B-shaped layer set at T = 1
(fused QKV 2048x1536, O 1536x1536, gate/up 8960x1536, down 1536x8960),
seeded synthetic weights and activations.  One step = one persistent
launch over the 140 GEMVs in layer order, which quantises every GEMV's fp32
activations as it loads them.  The weights (0.737 GB) exceed L2, so every
step streams them from HBM.

Metric: effective weight-stream GB/s = (Q4_0 weight bytes + fp32 activation
bytes + fp32 output bytes) / step time; also microseconds per GEMV.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun each rank runs an independent replica (the path does not
shard across GPUs); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "effective weight-stream GB/s (% of GB300 HBM peak) and us per q4_0 GEMV"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "qwen2.5-1.5b_layerset"
L2_FLUSH_BYTES = 256 << 20  # written before the timed region: twice the 126 MB L2


# ============================================================ workloads

class Workload:
    """A resident workload: device weights (packed), activations, outputs,
    and the launches of one step."""

    def __init__(self, name: str, T: int):
        self.name = name
        self.T = T
        self.w_bytes = 0          # Q4_0 weight bytes streamed per step
        self.x_bytes = 0          # fp32 activation bytes read per step
        self.y_bytes = 0          # output bytes written per step
        self.xq_bytes = 0         # quantised activation bytes the GEMV reads per step
        self.n_gemv = 0
        self.launches = 0         # kernels of ours per step
        self.host = {}            # optional host copies for parity checks
        self.kernel_name = "qgemv_stream_kernel"  # the step's streaming kernel
        self.config = {}
        self.rotation = 1         # steps after which the step's inputs repeat

    @property
    def step_bytes(self) -> int:
        return self.w_bytes + self.x_bytes + self.y_bytes

    @property
    def gemv_kernel_bytes(self) -> int:
        """Algorithmic bytes of the dominant (GEMV) launch of one step."""
        return self.w_bytes + self.xq_bytes + self.y_bytes


def _q():
    import quantized_q4_weight_gb300 as q
    return q


def _upload_packed(q, torch, Wg, N, K, dev):
    Wd = torch.from_numpy(Wg.reshape(-1)).to(dev)
    Wp = q.pack_q4_0(Wd, N, K)
    del Wd
    return Wp


def build_layerset(name, layer, layers, T, seed, dev, keep_host=False, epilogue=False, reuse_W=None):
    """Layer set in order.  One step = one fp32-input sequence call (one
    persistent launch that also quantises the activations).  epilogue: qkv
    adds a bias [N], o and down add a residual [T][N] (seeded inputs).
    reuse_W: the packed weights of an earlier build of the same set (another
    T), used instead of generating them again."""
    import torch
    q = _q()
    wl = Workload(name, T)
    mats = synth.layer_set(layer, layers)
    wl.n_gemv = len(mats)
    xs_off, ys_off, xo, yo = [], [], 0, 0
    for (_, N, K) in mats:
        xs_off.append(xo)
        ys_off.append(yo)
        xo += T * K
        yo += T * N
    x_all = np.empty(xo, np.float32)
    for i, (_, N, K) in enumerate(mats):
        x_all[xs_off[i]:xs_off[i] + T * K] = synth.activations(seed, T, K, stream=(i,)).reshape(-1)
    wl.x_all = torch.from_numpy(x_all).to(dev)
    wl.y_all = torch.empty(yo, dtype=torch.float32, device=dev)
    wl.x = [wl.x_all[xs_off[i]:xs_off[i] + T * K].view(T, K) for i, (_, N, K) in enumerate(mats)]
    wl.y = [wl.y_all[ys_off[i]:ys_off[i] + T * N].view(T, N) for i, (_, N, K) in enumerate(mats)]
    wl.W, wl.xq = [], []
    for i, (nm, N, K) in enumerate(mats):
        if reuse_W is not None:
            wl.W.append(reuse_W[i])
        else:
            Wg = synth.q4_0_weights(seed, N, K, stream=(i,))
            if keep_host:
                wl.host[i] = Wg
            wl.W.append(_upload_packed(q, torch, Wg, N, K, dev))
        wl.xq.append(q.quantize_q8_0(wl.x[i], T, K))
        wl.w_bytes += q.q4_0_bytes(N, K)
        wl.x_bytes += 4 * T * K
        wl.y_bytes += 4 * T * N
        wl.xq_bytes += q.xq_bytes(T, K)
    wl.mats = mats
    wl.launches = 1
    wl.inputs, wl.outputs = [wl.x_all], [wl.y_all]
    if not epilogue:
        wl.items_f32 = q.seq_f32_items([(wl.W[i], wl.x[i], wl.y[i], N, K) for i, (_, N, K) in enumerate(mats)])
        wl.items_xq = q.seq_items([(wl.W[i], wl.xq[i], wl.y[i], N, K) for i, (_, N, K) in enumerate(mats)])
        wl.ws = q.new_workspace(q.seq_f32_workspace_bytes(wl.items_f32, T), dev)
        wl.ws_xq = q.new_workspace(q.seq_workspace_bytes(wl.items_xq, T), dev)

        def step(stream=None):
            q.gemv_seq_f32(wl.items_f32, q.W_PACKED, T, wl.ws, stream=stream)

        def kernel(stream=None):
            q.gemv_seq(wl.items_xq, q.W_PACKED, T, wl.ws_xq, stream=stream)
    else:
        bias, res = [None] * len(mats), [None] * len(mats)
        for i, (nm, N, K) in enumerate(mats):
            rng = np.random.default_rng([seed, 7, i])
            if nm.endswith(".qkv"):
                bias[i] = torch.from_numpy(rng.standard_normal(N).astype(np.float32)).to(dev)
                wl.x_bytes += 4 * N
                wl.xq_bytes += 4 * N
            elif nm.endswith(".o") or nm.endswith(".down"):
                res[i] = torch.from_numpy(rng.standard_normal((T, N)).astype(np.float32)).to(dev)
                wl.x_bytes += 4 * T * N
                wl.xq_bytes += 4 * T * N
        wl.bias, wl.res = bias, res
        wl.items_f32 = q.seq_ep_items([(wl.W[i], wl.x[i], wl.y[i], N, K, bias[i], res[i])
                                       for i, (_, N, K) in enumerate(mats)])
        wl.items_xq = q.seq_ep_items([(wl.W[i], wl.xq[i], wl.y[i], N, K, bias[i], res[i])
                                      for i, (_, N, K) in enumerate(mats)])
        wl.ws = q.new_workspace(q.seq_ep_workspace_bytes(wl.items_f32, T, True), dev)
        wl.ws_xq = q.new_workspace(q.seq_ep_workspace_bytes(wl.items_xq, T, False), dev)
        wl.inputs = [wl.x_all] + [b for b in bias if b is not None] + [r for r in res if r is not None]

        def step(stream=None):
            q.gemv_seq_ep(wl.items_f32, q.W_PACKED, T, wl.ws, x_f32=True, stream=stream)

        def kernel(stream=None):
            q.gemv_seq_ep(wl.items_xq, q.W_PACKED, T, wl.ws_xq, x_f32=False, stream=stream)

    wl.step, wl.kernel = step, kernel
    wl.config = {"workload": name, "layers": layers, "gemvs": len(mats), "T": T,
                 "weight_bytes": wl.w_bytes,
                 "epilogue": "bias on qkv, residual on o and down (read as inputs)" if epilogue else None,
                 "l2_defeat": "weights larger than the 126 MB L2, each streamed once per step"}
    return wl


def build_lm_head(T, seed, dev, copies=4, keep_host=False, N=151936, K=1536):
    import torch
    q = _q()
    wl = Workload("lm_head_argmax", T)
    wl.W = []
    for c in range(copies):
        Wg = synth.q4_0_weights(seed, N, K, stream=(c,))
        if keep_host:
            wl.host[c] = Wg
        wl.W.append(_upload_packed(q, torch, Wg, N, K, dev))
    wl.x = torch.from_numpy(synth.activations(seed, T, K)).to(dev)
    wl.xqb = q.quantize_q8_0(wl.x, T, K)  # the kernel-only launches' input
    wl.idx = torch.empty(T, dtype=torch.int64, device=dev)
    wl.ws = q.new_workspace(q.workspace_bytes(N, K, T), dev)
    wl.w_bytes = q.q4_0_bytes(N, K)
    wl.x_bytes, wl.y_bytes, wl.xq_bytes = 4 * T * K, 8 * T, q.xq_bytes(T, K)
    wl.n_gemv, wl.launches = 1, 1
    wl.copy = 0
    wl.N, wl.K = N, K

    def kernel(stream=None):
        q.gemv_argmax(wl.W[wl.copy], q.W_PACKED, wl.xqb, N, K, T, wl.ws, idx=wl.idx, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    def step(stream=None):
        q.gemv_argmax_f32(wl.W[wl.copy], q.W_PACKED, wl.x, N, K, T, wl.ws, idx=wl.idx, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    wl.step, wl.kernel = step, kernel
    wl.rotation = copies
    wl.inputs, wl.outputs = [wl.x], [wl.idx]
    wl.config = {"workload": "lm_head_argmax", "N": N, "K": K, "T": T, "copies": copies,
                 "l2_defeat": f"{copies} weight copies in rotation ({copies * wl.w_bytes / 1e6:.0f} MB)"}
    return wl


def build_verify(T, seed, dev, copies=4, keep_host=False, N=151936, K=1536):
    """A speculative verify step on the lm_head: T positions (the current
    token and T-1 drafts) through the fp32-input top-2 GEMV, with the commit
    rule on the first rows applied by the same launch."""
    import torch
    q = _q()
    wl = build_lm_head(T, seed, dev, copies, keep_host, N, K)
    wl.name = "lm_head_top2_verify"
    wl.idx2 = torch.empty((T, 2), dtype=torch.int64, device=dev)
    wl.val2 = torch.empty((T, 2), dtype=torch.float32, device=dev)
    wl.n_commit = torch.empty(1, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(seed + 7)          # seeded synthetic drafts
    wl.tokens = torch.from_numpy(rng.integers(0, N, T).astype(np.int64)).to(dev)
    wl.y_bytes = 24 * T + 4                         # idx2, val2, committed count
    wl.launches = 1
    wl.copy = 0

    def kernel(stream=None):
        q.gemv_top2(wl.W[wl.copy], q.W_PACKED, wl.xqb, N, K, T, wl.ws, idx2=wl.idx2, val2=wl.val2, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    def step(stream=None):  # one launch: top-2 rows and the commit rule
        q.verify_f32(wl.W[wl.copy], q.W_PACKED, wl.x, wl.tokens, N, K, T, wl.ws, idx2=wl.idx2, val2=wl.val2,
                     n_commit=wl.n_commit, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    wl.step, wl.kernel = step, kernel
    wl.inputs, wl.outputs = [wl.x, wl.tokens], [wl.idx2, wl.val2, wl.n_commit]
    wl.config = {"workload": "lm_head_top2_verify", "N": N, "K": K, "T": T, "copies": copies,
                 "step": "top-2 lm_head GEMV on fp32 x (quantised in the kernel) and the commit rule, one launch",
                 "l2_defeat": f"{copies} weight copies in rotation ({copies * wl.w_bytes / 1e6:.0f} MB)"}
    return wl


def build_ffn(T, seed, dev, layers=28, d_model=1536, d_ff=8960, keep_host=False):
    """The decode FFN of every layer: per layer one qgemv_q4_0_ffn call (one
    fused launch for T <= 4; otherwise gate and up in one launch on the same
    fp32 x, the SiLU * up quantiser, down), each layer with its own seeded
    weights and x."""
    import torch
    q = _q()
    wl = Workload("qwen2.5-1.5b_ffn", T)
    wl.Wg, wl.Wu, wl.Wd, wl.xs, wl.ys = [], [], [], [], []
    for l in range(layers):
        for lst, (N, K, k) in zip((wl.Wg, wl.Wu, wl.Wd), ((d_ff, d_model, 0), (d_ff, d_model, 1), (d_model, d_ff, 2))):
            Wg = synth.q4_0_weights(seed, N, K, stream=(l, k))
            lst.append(_upload_packed(q, torch, Wg, N, K, dev))
            wl.w_bytes += Wg.nbytes
        wl.xs.append(torch.from_numpy(synth.activations(seed, T, d_model, stream=(l,))).to(dev))
        wl.ys.append(torch.empty((T, d_model), dtype=torch.float32, device=dev))
    wl.ws = q.new_workspace(q.ffn_workspace_bytes(d_model, d_ff, T), dev)
    wl.x_bytes = 4 * T * d_model * layers
    wl.y_bytes = 4 * T * d_model * layers
    wl.xq_bytes = (2 * q.xq_bytes(T, d_model) + q.xq_bytes(T, d_ff)) * layers
    fused = T <= 4  # one fused launch per layer; else gate/up, the SiLU step and down
    wl.n_gemv, wl.launches = 3 * layers, (1 if fused else 3) * layers

    def step(stream=None):
        for l in range(layers):
            q.ffn(wl.Wg[l], wl.Wu[l], wl.Wd[l], q.W_PACKED, wl.xs[l], d_model, d_ff, T, wl.ws, y=wl.ys[l],
                  stream=stream)

    wl.step, wl.kernel, wl.dominant = step, step, step
    wl.dominant_bytes = wl.w_bytes + wl.x_bytes + wl.y_bytes
    wl.other_launch = ("the whole step: per layer one fused launch (T <= 4), else the gate/up and down "
                       "streaming launches and the SiLU * up quantiser")
    wl.inputs, wl.outputs = list(wl.xs), list(wl.ys)
    wl.config = {"workload": "qwen2.5-1.5b_ffn", "layers": layers, "d_model": d_model, "d_ff": d_ff, "T": T,
                 "weight_bytes": wl.w_bytes, "step": ("per layer one qgemv_q4_0_ffn call: " +
                          ("one fused launch (gate+up, SiLU(gate)*up to Q8_0, down)" if fused else
                           "gate+up launch, SiLU(gate)*up to Q8_0, down launch")),
                 "l2_defeat": "weights larger than the 126 MB L2, each streamed once per step"}
    return wl


def build_q8(T, seed, dev, copies=2, keep_host=False, N=151936, K=1536):
    """The lm_head held as Q8_0 weights: one step quantises x and runs the
    Q8_0-weight GEMV (two launches); copies rotate so reads hit HBM."""
    import torch
    q = _q()
    wl = Workload("q8_lm_head", T)
    wl.W = []
    for c in range(copies):
        Wg = synth.q8_0_weights(seed, N, K, stream=(c,))
        if keep_host:
            wl.host[c] = Wg
        Wd = torch.from_numpy(Wg.reshape(-1)).to(dev)
        wl.W.append(q.pack_q8_0(Wd, N, K))
        del Wd
    wl.x = torch.from_numpy(synth.activations(seed, T, K)).to(dev)
    wl.xqb = q.quantize_q8_0(wl.x, T, K)
    wl.y = torch.empty((T, N), dtype=torch.float32, device=dev)
    wl.ws = q.new_workspace(q.q8_0_workspace_bytes(N, K, T), dev)
    wl.w_bytes = q.q8_0_bytes(N, K)
    wl.x_bytes, wl.y_bytes, wl.xq_bytes = 4 * T * K, 4 * T * N, q.xq_bytes(T, K)
    wl.n_gemv, wl.launches = 1, 2
    wl.copy = 0

    def kernel(stream=None):
        q.gemv_q8_0(wl.W[wl.copy], wl.xqb, N, K, T, wl.ws, y=wl.y, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    def step(stream=None):
        q.quantize_q8_0(wl.x, T, K, out=wl.xqb, stream=stream)
        kernel(stream)

    wl.step, wl.kernel, wl.dominant = step, kernel, kernel
    wl.dominant_bytes = wl.w_bytes + wl.xq_bytes + wl.y_bytes
    wl.other_launch = "the step's other launch is the activation quantiser"
    wl.kernel_name = "q8_gemv_kernel"
    wl.inputs, wl.outputs = [wl.x], [wl.y]
    wl.config = {"workload": "q8_lm_head", "N": N, "K": K, "T": T, "copies": copies, "weights": "Q8_0",
                 "step": "Q8_0 quantiser launch, then the Q8_0-weight GEMV launch",
                 "l2_defeat": f"{copies} weight copies in rotation ({copies * wl.w_bytes / 1e6:.0f} MB)"}
    return wl


def build_gs64(T, seed, dev, copies=4, keep_host=False, N=151936, K=1536):
    """A dense matrix of the lm_head's shape in the gs64 grouped int4 format
    (colibri qwen36 docs: the dense trunk stored as int4 in groups of 64 with
    one scale each): one step is one launch of the gs64 GEMV on fp32 x,
    quantised once per vector to int8 inside the launch; copies rotate so
    reads hit HBM."""
    import torch
    q = _q()
    wl = Workload("gs64_lm_head", T)
    wl.N, wl.K = N, K
    wl.W = []
    for c in range(copies):
        wq, ws = synth.gs64_weights(seed, N, K, stream=(c,))
        if keep_host:
            wl.host[c] = (wq, ws)
        wl.W.append(q.pack_gs64(torch.from_numpy(wq).to(dev), torch.from_numpy(ws).to(dev), N, K))
    wl.x = torch.from_numpy(synth.activations(seed, T, K)).to(dev)
    wl.qx, wl.sx = q.quantize_vec_i8(wl.x, T, K)
    wl.y = torch.empty((T, N), dtype=torch.float32, device=dev)
    wl.ws = q.new_workspace(q.gs64_workspace_bytes(N, K, T), dev)
    wl.w_bytes = q.gs64_bytes(N, K)
    wl.x_bytes, wl.y_bytes, wl.xq_bytes = 4 * T * K, 4 * T * N, T * K + 4 * T
    wl.n_gemv, wl.launches = 1, 1
    wl.copy = 0

    def kernel(stream=None):  # on pre-quantised activations
        q.gemv_gs64(wl.W[wl.copy], wl.qx, wl.sx, N, K, T, wl.ws, y=wl.y, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    def step(stream=None):  # fp32 x, quantised inside the one GEMV launch
        q.gemv_gs64_f32(wl.W[wl.copy], wl.x, N, K, T, wl.ws, y=wl.y, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    wl.step, wl.kernel = step, kernel
    wl.rotation = copies
    wl.kernel_name = "gs64_gemv_kernel"
    wl.dtype = "uint4 x int8 -> int32 group sums, fp32 accumulation"
    wl.data = ("synthetic (seeded; gs64 nibbles uniform, fp32 group scales U[1e-3,4e-3], "
               "x N(0,1) with 1% x20)")
    wl.inputs, wl.outputs = [wl.x], [wl.y]
    wl.config = {"workload": "gs64_lm_head", "N": N, "K": K, "T": T, "copies": copies,
                 "weights": "gs64 (64-weight groups, fp32 scale)",
                 "step": "one gs64 GEMV launch on fp32 x (per-vector int8 quantisation inside it)",
                 "l2_defeat": f"{copies} weight copies in rotation ({copies * wl.w_bytes / 1e6:.0f} MB)"}
    return wl


def build_requant(T, seed, dev, copies=2, keep_host=False, N=151936, K=1536):
    """Load-time requantisation of the Q8_0 lm_head to Q4_0 blocks (one
    launch per step); two source copies rotate so reads hit HBM."""
    import torch
    q = _q()
    wl = Workload("lm_head_requant_q8", T)
    wl.W = []
    for c in range(copies):
        Wg = synth.q8_0_weights(seed, N, K, stream=(c,))
        if keep_host:
            wl.host[c] = Wg
        wl.W.append(torch.from_numpy(Wg.reshape(-1)).to(dev))
    wl.out = torch.empty(q.q4_0_bytes(N, K), dtype=torch.uint8, device=dev)
    wl.w_bytes, wl.y_bytes = q.q8_0_bytes(N, K), q.q4_0_bytes(N, K)   # read, written
    wl.n_gemv, wl.launches = 1, 1
    wl.copy = 0

    def step(stream=None):
        q.requant_q8_0_q4_0(wl.W[wl.copy], N, K, out=wl.out, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    wl.step, wl.kernel = step, step
    wl.kernel_name = "requant_q4_0_staged_q8"
    wl.dtype = "fp32 encoder arithmetic (Q8_0 in, Q4_0 out)"
    wl.data = "synthetic (seeded; Q8_0 codes uniform on [-127, 127], fp16 scales U[1e-3,4e-3])"
    wl.inputs, wl.outputs = [wl.W[0]], [wl.out]
    wl.config = {"workload": "lm_head_requant_q8", "N": N, "K": K, "copies": copies,
                 "bytes": "Q8_0 read + Q4_0 written per step; us_per_gemv is us per requantisation",
                 "l2_defeat": f"{copies} source copies in rotation ({copies * wl.w_bytes / 1e6:.0f} MB)"}
    return wl


def build_single(T, seed, dev, copies=400, N=1536, K=1536, keep_host=False):
    import torch
    q = _q()
    wl = Workload("single_1536", T)
    Wg0 = synth.q4_0_weights(seed, N, K)
    if keep_host:
        wl.host[0] = Wg0
    W0 = _upload_packed(q, torch, Wg0, N, K, dev)
    wl.W = [W0] + [W0.clone() for _ in range(copies - 1)]     # distinct copies defeat L2
    wl.x = torch.from_numpy(synth.activations(seed, T, K)).to(dev)
    wl.y = torch.empty((T, N), dtype=torch.float32, device=dev)
    wl.ws = q.new_workspace(q.workspace_bytes(N, K, T), dev)
    wl.w_bytes, wl.x_bytes, wl.y_bytes = q.q4_0_bytes(N, K), 4 * T * K, 4 * T * N
    wl.xq_bytes = q.xq_bytes(T, K)
    wl.n_gemv, wl.launches, wl.copy = 1, 1, 0
    wl.N, wl.K = N, K

    wl.xqb = q.quantize_q8_0(wl.x, T, K)

    def step(stream=None):
        q.gemv_f32(wl.W[wl.copy], q.W_PACKED, wl.x, N, K, T, wl.ws, y=wl.y, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    def kernel(stream=None):
        q.gemv(wl.W[wl.copy], q.W_PACKED, wl.xqb, N, K, T, wl.ws, y=wl.y, stream=stream)
        wl.copy = (wl.copy + 1) % copies

    wl.step, wl.kernel = step, kernel
    wl.rotation = copies
    wl.inputs, wl.outputs = [wl.x], [wl.y]
    wl.config = {"workload": "single_1536", "N": N, "K": K, "T": T, "copies": copies,
                 "l2_defeat": f"{copies} weight copies in rotation"}
    return wl


def build_moe(T, seed, dev, sets=4, n_experts=256, top_k=8, d_model=2048, d_ff=512, keep_host=False):
    """Routed experts: per set 256 experts + 1 shared (stored as expert 256)."""
    import torch
    q = _q()
    wl = Workload("moe_top8_shared", T)
    shapes = [("gate", d_ff, d_model), ("up", d_ff, d_model), ("down", d_model, d_ff)]
    ne = n_experts + 1
    wl.sets = []
    for s in range(sets):
        mats = []
        for m, (nm, N, K) in enumerate(shapes):
            per = q.q4_0_bytes(N, K)
            W = torch.empty(ne * per, dtype=torch.uint8, device=dev)
            for e in range(ne):
                Wg = synth.q4_0_weights(seed, N, K, stream=(s, m, e))
                if keep_host and s == 0:
                    wl.host[(m, e)] = Wg
                W[e * per:(e + 1) * per] = _upload_packed(q, torch, Wg, N, K, dev)
            mats.append(W)
        wl.sets.append(mats)
    n_ids = top_k + 1
    ids = synth.expert_ids(seed, 64, n_experts, top_k)
    wl.ids = [torch.from_numpy(np.concatenate([ids[i], [n_experts]]).astype(np.int32)).to(dev) for i in range(64)]
    wl.x_in = torch.from_numpy(synth.activations(seed, T, d_model)).to(dev)
    wl.x_dn = torch.from_numpy(synth.activations(seed + 1, n_ids * T, d_ff)).to(dev)
    xg, xd = q.xq_bytes(T, d_model), q.xq_bytes(T, d_ff)
    wl.xq_in = torch.empty(xg, dtype=torch.uint8, device=dev)
    wl.xq_dn = torch.empty(n_ids * xd, dtype=torch.uint8, device=dev)
    wl.yg = torch.empty((n_ids, T, d_ff), dtype=torch.float32, device=dev)
    wl.yu = torch.empty((n_ids, T, d_ff), dtype=torch.float32, device=dev)
    wl.yd = torch.empty((n_ids, T, d_model), dtype=torch.float32, device=dev)
    wl.gm, wl.gf = [], []
    for s in range(sets):
        Wgt, Wup, Wdn = wl.sets[s]
        wl.gm.append(q.gather_mats([
            (Wgt, q.q4_0_bytes(d_ff, d_model), wl.xq_in, 0, wl.yg, T * d_ff, d_ff, d_model),
            (Wup, q.q4_0_bytes(d_ff, d_model), wl.xq_in, 0, wl.yu, T * d_ff, d_ff, d_model),
            (Wdn, q.q4_0_bytes(d_model, d_ff), wl.xq_dn, xd, wl.yd, T * d_model, d_model, d_ff)]))
        wl.gf.append(q.gather_f32_mats([
            (Wgt, q.q4_0_bytes(d_ff, d_model), wl.x_in, 0, wl.yg, T * d_ff, d_ff, d_model),
            (Wup, q.q4_0_bytes(d_ff, d_model), wl.x_in, 0, wl.yu, T * d_ff, d_ff, d_model),
            (Wdn, q.q4_0_bytes(d_model, d_ff), wl.x_dn, 4 * T * d_ff, wl.yd, T * d_model, d_model, d_ff)]))
    wl.ws = q.new_workspace(max(q.gather_workspace_bytes(wl.gm[0], n_ids, T),
                                q.gather_f32_workspace_bytes(wl.gf[0], n_ids, T)), dev)
    per_tok = n_ids * (2 * q.q4_0_bytes(d_ff, d_model) + q.q4_0_bytes(d_model, d_ff))
    wl.w_bytes = per_tok
    wl.x_bytes = 4 * T * (d_model + n_ids * d_ff)
    wl.y_bytes = 4 * T * n_ids * (2 * d_ff + d_model)
    wl.xq_bytes = xg + n_ids * xd
    wl.n_gemv, wl.launches, wl.tok = 3 * n_ids, 1, 0
    wl.n_experts, wl.n_ids = ne, n_ids

    def quantize(stream=None):
        q.quantize_q8_0(wl.x_in, T, d_model, out=wl.xq_in, stream=stream)
        q.quantize_q8_0(wl.x_dn, T, d_ff, batch=n_ids, out=wl.xq_dn, stream=stream)

    def kernel(stream=None):
        s = wl.tok % sets
        q.gemv_gather(wl.gm[s], wl.ids[wl.tok % 64], ne, q.W_PACKED, T, wl.ws, stream=stream)
        wl.tok += 1

    def step(stream=None):  # fp32 inputs, quantised inside the one gather launch
        s = wl.tok % sets
        q.gemv_gather_f32(wl.gf[s], wl.ids[wl.tok % 64], ne, q.W_PACKED, T, wl.ws, stream=stream)
        wl.tok += 1

    quantize()  # the kernel-only launches' inputs
    wl.quantize = quantize
    wl.step, wl.kernel = step, kernel
    wl.rotation = 64  # the seeded tokens' expert ids cycle every 64 steps (the 4 sets every 4)
    wl.inputs, wl.outputs = [wl.x_in, wl.x_dn], [wl.yg, wl.yu, wl.yd]
    wl.config = {"workload": "moe_top8_shared", "experts": n_experts, "top_k": top_k, "shared": 1, "T": T,
                 "sets": sets, "l2_defeat": f"{sets} expert sets in rotation ({sets * ne * 3 * q.q4_0_bytes(d_ff, d_model) / 1e9:.2f} GB)"}
    return wl


def build_workload(name: str, dev, T: int | None = None, keep_host: bool = False,
                   layers: int | None = None, reuse_W=None) -> Workload:
    spec = synth.WORKLOADS[name]
    if spec["kind"] == "seq":
        T = T or spec.get("T", 1)
        return build_layerset(name, spec["layer"], layers or spec["layers"], T, spec["seed"], dev, keep_host,
                              spec.get("epilogue", False), reuse_W)
    if spec["kind"] == "argmax":
        return build_lm_head(T or spec["T"], spec["seed"], dev, spec["copies"], keep_host, spec["N"], spec["K"])
    if spec["kind"] == "verify":
        return build_verify(T or spec["T"], spec["seed"], dev, spec["copies"], keep_host, spec["N"], spec["K"])
    if spec["kind"] == "ffn":
        return build_ffn(T or spec["T"], spec["seed"], dev, layers or spec["layers"], spec["d_model"], spec["d_ff"],
                         keep_host)
    if spec["kind"] == "q8":
        return build_q8(T or spec["T"], spec["seed"], dev, spec["copies"], keep_host, spec["N"], spec["K"])
    if spec["kind"] == "gs64":
        return build_gs64(T or spec["T"], spec["seed"], dev, spec["copies"], keep_host, spec["N"], spec["K"])
    if spec["kind"] == "requant":
        return build_requant(T or spec["T"], spec["seed"], dev, spec["copies"], keep_host, spec["N"], spec["K"])
    if spec["kind"] == "single":
        return build_single(T or spec["T"], spec["seed"], dev, keep_host=keep_host, N=spec["N"], K=spec["K"])
    if spec["kind"] == "moe":
        return build_moe(T or spec["T"], spec["seed"], dev, spec["sets"], spec["n_experts"], spec["top_k"],
                         spec["d_model"], spec["d_ff"], keep_host)
    raise KeyError(name)


# ============================================================ measurement helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources each measured kernel is built from, with the host planning
# code that sizes its launches: a traffic record stays valid while they do.
_COMMON_SOURCES = ["qgemv_internal.cuh", "qgemv_launch.h", "qgemv_api.cu"]
KERNEL_SOURCES = {
    "qgemv_stream_kernel": ["gemv_kernel.cuh", "launch_stream.cuh"] + [f"gemv_t{t}.cu" for t in range(1, 9)],
    "q8_gemv_kernel": ["q8_kernel.cu"],
    "requant_q4_0_staged_q8": ["kernels_misc.cu"],
    "gs64_gemv_kernel": ["gs64_kernel.cu"],
    "ffn_fused_kernel": ["ffn_fused.cu", "gemv_kernel.cuh"],
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of one kernel's sources (all of csrc when the kernel is unknown)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_q4_weight_gb300", "csrc")
    files = sorted(KERNEL_SOURCES[kernel] + _COMMON_SOURCES) if kernel in KERNEL_SOURCES else sorted(os.listdir(csrc))
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_record(workload: str, T: int):
    """DRAM bytes per GEMV launch from a committed ncu summary, if it was
    taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        r = rec.get(f"{workload}/T{T}")
        if r and r.get("kernel_hash") == kernel_source_hash(r.get("kernel")):
            return r.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            self.path = tempfile.mktemp(suffix=".csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, mem, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
                if len(parts) > 9:
                    try:
                        mem.append(float(parts[9]))
                    except ValueError:
                        pass
        os.unlink(self.path)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}
        if mem:
            out["mem_mhz"] = statistics.median(mem)
        return out


# ============================================================ CPU baseline (oracle)

_ORACLE_INPUTS = {}


def _oracle_inputs(workload: str):
    """Seeded inputs of one step of the workload (generated once, cached)."""
    if workload not in _ORACLE_INPUTS:
        spec = synth.WORKLOADS[workload]
        if spec["kind"] == "seq":
            T = 1
            mats = synth.layer_set(spec["layer"], spec["layers"])
        elif spec["kind"] in ("argmax", "single", "verify", "q8", "requant", "gs64"):
            T, mats = spec["T"], [("w", spec["N"], spec["K"])]
        elif spec["kind"] == "ffn":
            T = spec["T"]
            mats = [("gate", spec["d_ff"], spec["d_model"]), ("up", spec["d_ff"], spec["d_model"]),
                    ("down", spec["d_model"], spec["d_ff"])] * spec["layers"]
        else:
            T = 1
            mats = [("gate", spec["d_ff"], spec["d_model"]), ("up", spec["d_ff"], spec["d_model"]),
                    ("down", spec["d_model"], spec["d_ff"])] * (spec["top_k"] + 1)
        if spec["kind"] == "gs64":
            _ORACLE_INPUTS[workload] = (T, [(N, K, synth.gs64_weights(spec["seed"], N, K, stream=(i,)),
                                             synth.activations(spec["seed"], T, K, stream=(i,)))
                                            for i, (_, N, K) in enumerate(mats)])
            return _ORACLE_INPUTS[workload]
        gen = synth.q8_0_weights if spec["kind"] in ("q8", "requant") else synth.q4_0_weights
        data = [(N, K, gen(spec["seed"], N, K, stream=(i,)),
                 synth.activations(spec["seed"], T, K, stream=(i,))) for i, (_, N, K) in enumerate(mats)]
        _ORACLE_INPUTS[workload] = (T, data)
    return _ORACLE_INPUTS[workload]


def cpu_model() -> str:
    """The host CPU's model name, as /proc/cpuinfo or lscpu report it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_sample(workload: str, budget_s: float = 12.0, min_s: float = 3.0, threads: int | None = None):
    """Time the CPU oracle as it stands (Q8_0 quantisation, per-block int32
    sums, fp64 accumulation; OpenMP over rows) on a bounded sample of one step
    of the workload, on all cores or on `threads` threads.  Returns (GB/s
    under the GPU's byte accounting, threads, description of the sample)."""
    import oracle
    oracle.build()
    o = oracle.load()
    if threads:
        o.set_threads(threads)
    T, data = _oracle_inputs(workload)
    if synth.WORKLOADS[workload]["kind"] == "requant":
        return _oracle_requant_sample(o, data, budget_s, min_s)
    kind = synth.WORKLOADS[workload]["kind"]
    gemv = o.gemv_q8 if kind == "q8" else o.gemv
    done_bytes, t_total, n_done = 0, 0.0, 0
    while True:
        for N, K, Wg, x in data:
            t0 = time.perf_counter()
            if kind == "gs64":
                o.gemv_gs64(Wg[0], Wg[1], N, K, *o.quantize_vec_i8(x))
                wbytes = Wg[0].nbytes + Wg[1].nbytes
            else:
                xq = o.quantize(x)
                gemv(Wg, N, K, xq, T)
                wbytes = Wg.nbytes
            t_total += time.perf_counter() - t0
            done_bytes += wbytes + 4 * T * K + 4 * T * N
            n_done += 1
            if t_total >= budget_s:
                break
        if t_total >= min_s or t_total >= budget_s:
            break
    return (done_bytes / t_total / 1e9, o.num_threads(),
            f"{n_done} GEMVs ({n_done / len(data):.2f} steps of {len(data)} GEMVs, {done_bytes / 1e6:.0f} MB), "
            f"T={T}, {t_total:.1f} s of oracle time")


def _oracle_requant_sample(o, data, budget_s, min_s):
    """The oracle's Q8_0 -> Q4_0 requantisation (one thread: the oracle's
    encoder loop has no OpenMP) over row slices of the lm_head."""
    N, K, Wg, _ = data[0]
    rows = 8192
    done_bytes, t_total, n_done = 0, 0.0, 0
    while t_total < budget_s:
        r0 = (n_done * rows) % N
        r1 = min(N, r0 + rows)
        t0 = time.perf_counter()
        o.requant_q8_0_q4_0(Wg[r0:r1], r1 - r0, K)
        t_total += time.perf_counter() - t0
        done_bytes += (r1 - r0) * (K // 32) * (34 + 18)
        n_done += 1
        if t_total >= budget_s:
            break
    return (done_bytes / t_total / 1e9, 1,
            f"{n_done} slices of {rows} rows ({done_bytes / 1e6:.0f} MB read + written), {t_total:.1f} s of oracle time")


# ============================================================ main

def own_stream_gbs(dev, nbytes: int = 4 << 30) -> float:
    """The library's own read-only stream (TMA, 16 warps x 2 x 4608-byte
    stages per SM) over one 4 GiB buffer: the achievable HBM read rate of the
    GEMV's access pattern, measured in this run (best of 5 launches)."""
    import torch
    q = _q()
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        q.stream_read(buf, 0, 16, 2, 4608, sink)
    best = float("inf")
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q.stream_read(buf, 0, 16, 2, 4608, sink)
        b.record(stream)
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del buf
    torch.cuda.empty_cache()
    return nbytes / (best * 1e-3) / 1e9


def slowest_rank_ms(ms: float, world: int) -> float:
    """Replicas only: every rank runs the same workload; the job's step time
    is the slowest rank's (max over ranks)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t[0])


def job_value(step_bytes: int, ms: float, world: int) -> float:
    """Whole-job GB/s: the bytes all ranks processed / the slowest rank's time."""
    return step_bytes * world / (ms * 1e-3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    steps, warm = args.steps, args.warmup
    vals = []
    for i in range(warm + steps):
        v, cores, desc = oracle_sample(args.workload, budget_s=max(1.0, 60.0 / (warm + steps)),
                                        min_s=min(1.0, 60.0 / (warm + steps)))
        if i >= warm:
            vals.append(v)
    value = statistics.median(vals)
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32 block sums + f64 accumulation (CPU oracle)", "data": "synthetic (seeded)",
            "config": {"workload": args.workload},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers of a layer-set workload (smaller profiling captures only)")
    ap.add_argument("--tc-min-tokens", type=int, default=0,
                    help="token count from which packed sequences use the tcgen05 kernel (0 = library default, 9 = never)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations' records (the default workload at N=1 measures them)")
    args = ap.parse_args(argv)
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from quantized_q4_weight_gb300 import _build
    _build.build()
    q = _q()
    q.set_tc_min_T(args.tc_min_tokens)

    own_stream = own_stream_gbs(dev)
    spec = synth.WORKLOADS[args.workload]
    Ts = [args.T] if args.T else list(spec.get("Ts", [spec.get("T", 1)]))
    results = {}
    workloads = None
    for T in Ts:
        wl = build_workload(args.workload, dev, T=T, layers=args.layers)
        results[T] = measure(args, wl, dev, world, rank)
        if (T == Ts[0] and world == 1 and args.workload == DEFAULT_WORKLOAD and not args.no_workloads
                and args.layers is None):
            workloads = measure_workloads(dev, wl)
        del wl
        torch.cuda.empty_cache()
    head = results[Ts[0]]
    if workloads is not None:
        head["workloads"] = workloads
    for r in results.values():
        r["config"]["own_stream_gbs"] = round(own_stream, 1)
        r["config"]["pct_of_own_stream"] = round(100 * r["value"] / world / own_stream, 2)
        r["roofline"]["frac_of_own_stream"] = round(r["roofline"]["achieved"] / own_stream, 4)
    if rank == 0:
        if len(Ts) > 1:
            base = results[Ts[0]]["ms_per_step"]
            head["config"]["t_sweep"] = {f"T{T}": {"ms_per_step": r["ms_per_step"], "value": r["value"],
                                                   "cost_vs_T1": round(r["ms_per_step"] / base, 4)}
                                         for T, r in results.items()}
        if not args.no_cpu_baseline:
            v1, _, desc1 = oracle_sample(args.workload, budget_s=4.0, min_s=2.0, threads=1)
            v, cores, desc = oracle_sample(args.workload, min_s=10.0, threads=os.cpu_count() or 1)
            head["cpu_baseline"] = {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": desc, "single_thread_value": round(v1, 4),
                                    "single_thread_sample": desc1, "cpu": cpu_model()}
        print(json.dumps(head), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()
    return 0


# The other configurations of the metric, measured in the same run (one
# record each in the line's "workloads" list): the single 1536 x 1536 GEMV,
# the 28-layer Qwen2.5-1.5B set, the lm_head with argmax, the Qwen2.5-3B set
# at T = 1, 2, 4, 8 and the routed-expert step.
REPEAT_MIN_MS = 50.0   # each repeat times at least this much work
REPEATS = 7
GRAPH_CAP = 512        # steps captured in one graph (replayed as often as a repeat needs)


def repeat_timing(torch, dev, stream, wl):
    """Per-step device time of a workload: n steps captured once in a CUDA
    graph (n a multiple of the workload's rotation, so that every replay
    walks its weight copies in the same cyclic order and each copy comes
    back only after the whole rotation), replayed k times inside each of
    REPEATS timed repeats of at least REPEAT_MIN_MS.  Returns (median, min,
    max) microseconds per step and the steps per repeat."""
    for _ in range(3):
        wl.step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(max(8, wl.rotation)):
        wl.step()
    b.record(stream)
    torch.cuda.synchronize()
    est_ms = a.elapsed_time(b) / max(8, wl.rotation)
    rot = max(1, wl.rotation)
    n = min(GRAPH_CAP, max(1, int(REPEAT_MIN_MS / est_ms) + 1))
    n = max(rot, (n + rot - 1) // rot * rot)
    g = capture_steps(torch, dev, stream, wl.step, n)
    if g is None:
        raise RuntimeError(f"{wl.name}: graph capture failed")
    g.replay()
    torch.cuda.synchronize()
    k = max(1, int(REPEAT_MIN_MS / (n * est_ms)) + 1)
    per = []
    for _ in range(REPEATS):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) * 1e3 / (n * k))
    del g
    return statistics.median(per), min(per), max(per), n * k


def workload_record(torch, dev, stream, wl, label: str, peak: float, base_us: float | None = None):
    q = _q()
    med, lo, hi, steps = repeat_timing(torch, dev, stream, wl)
    assert q.device_status() == 0
    gbs = wl.step_bytes / (med * 1e-6) / 1e9
    rec = {"config": label, "workload": wl.name, "T": wl.T, "us_per_step": round(med, 3),
           "us_min": round(lo, 3), "us_max": round(hi, 3), "repeats": REPEATS, "steps_per_repeat": steps,
           "bytes_per_step": wl.step_bytes, "weight_bytes_per_step": wl.w_bytes,
           "value": round(gbs, 2), "unit": UNIT, "frac_of_peak": round(gbs / peak, 4), "peak": peak,
           "gemvs_per_step": wl.n_gemv, "us_per_gemv": round(med / wl.n_gemv, 3),
           "traffic": traffic_record(wl.name, wl.T),
           "l2_defeat": wl.config.get("l2_defeat")}
    if base_us is not None:
        rec["cost_vs_T1"] = round(med / base_us, 4)
    return rec


def measure_workloads(dev, head_wl):
    """One record per configuration of the metric (see REPEAT_MIN_MS)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peaks()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    recs = []
    wl = build_workload("single_1536", dev)
    recs.append(workload_record(torch, dev, stream, wl, "single 1536 x 1536, T=1, quantiser included", peak))
    del wl
    torch.cuda.empty_cache()
    recs.append(workload_record(torch, dev, stream, head_wl,
                                "Qwen2.5-1.5B 28-layer set, T=1 (the headline's workload)", peak))
    wl = build_workload("lm_head_argmax", dev)
    recs.append(workload_record(torch, dev, stream, wl, "lm_head 151936 x 1536 + argmax, T=1, 4 copies", peak))
    del wl
    torch.cuda.empty_cache()
    W3, base = None, None
    for T in (1, 2, 4, 8):
        wl = build_workload("qwen2.5-3b_verify", dev, T=T, reuse_W=W3)
        W3 = wl.W
        r = workload_record(torch, dev, stream, wl, f"Qwen2.5-3B 36-layer set, T={T}", peak, base)
        base = base or r["us_per_step"]
        r["cost_vs_T1"] = round(r["us_per_step"] / base, 4)
        recs.append(r)
        del wl
    del W3
    torch.cuda.empty_cache()
    wl = build_workload("moe_top8_shared", dev)
    recs.append(workload_record(torch, dev, stream, wl, "MoE top-8 + shared expert, T=1, 4 expert sets", peak))
    del wl
    torch.cuda.empty_cache()
    wl = build_workload("qwen2.5-1.5b_ffn", dev)
    recs.append(workload_record(torch, dev, stream, wl,
                                "decode FFN of 28 Qwen2.5-1.5B layers (one fused launch each), T=1", peak))
    del wl
    torch.cuda.empty_cache()
    wl = build_workload("gs64_lm_head", dev)
    recs.append(workload_record(torch, dev, stream, wl,
                                "gs64 grouped int4, 151936 x 1536, fp32 x quantised per vector in the launch, "
                                "T=1, 4 copies", peak))
    del wl
    torch.cuda.empty_cache()
    clk = clocks.stop()
    return {"records": recs, "peak_kind": peak_kind, "clocks": clk,
            "timed_as": f"{REPEATS} repeats, each >= {REPEAT_MIN_MS:.0f} ms of CUDA-graph replays of whole "
                        f"rotations of the workload's weight copies; median, min and max per step"}


def capture_steps(torch, dev, stream, fn, n: int):
    """n calls of fn captured, in order, in one CUDA graph; None if capture fails."""
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g):
                for _ in range(n):
                    fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        return g
    except Exception:
        torch.cuda.synchronize()
        return None


def measure(args, wl: Workload, dev, world, rank):
    import torch
    q = _q()
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    assert q.device_status() == 0

    # ---- timed region: K steps back to back, inputs resident in HBM.  The K
    # steps are issued as a decode loop issues them: captured once in a CUDA
    # graph, replayed once (direct calls if capture fails).  L2 is flushed
    # just before, so every weight byte of the K steps comes from HBM.
    K = args.steps
    g_steps = capture_steps(torch, dev, stream, wl.step, K)
    if g_steps is not None:
        g_steps.replay()  # untimed: the graph's first launch
    l2_flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    if world > 1:
        torch.distributed.barrier()
    clocks.start()
    time.sleep(0.3)
    # the flush is the last work before the timed steps, on the same stream:
    # no idle gap (and no clock ramp) between it and the first timed step
    l2_flush.fill_(1)
    t_start.record(stream)
    if g_steps is not None:
        g_steps.replay()
    else:
        for i in range(K):
            wl.step()
    t_end.record(stream)
    torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end) / K
    g_captured = g_steps is not None
    del g_steps, l2_flush
    # ---- the same K steps as direct calls through the API (context: host
    # launch rate bounds the smallest workloads here)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for i in range(K):
        wl.step()
    d1.record(stream)
    torch.cuda.synchronize()
    direct_ms = d0.elapsed_time(d1) / K
    # ---- the dominant (GEMV) launch alone: K launches back to back between
    # two events on the launching stream (average launch duration)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    for i in range(K):
        wl.kernel()
    k1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    gemv_ms = k0.elapsed_time(k1) / K
    # ---- the same kernel loop captured in a CUDA graph (median of 7 replays)
    graph_ms = None
    try:
        R = 20
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            wl.kernel()
            torch.cuda.synchronize()
            with torch.cuda.graph(g):
                for _ in range(R):
                    wl.kernel()
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            reps.append(a.elapsed_time(b) / R)
        graph_ms = statistics.median(reps)
        del g
    except Exception:
        graph_ms = None
    ms_local = ms  # this GPU's step time, for its roofline
    ms = slowest_rank_ms(ms, world)
    assert q.device_status() == 0

    # ---- end to end through the public API: pinned host inputs in, outputs out
    h_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x.cpu()) for x in wl.inputs]
    h_out = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in wl.outputs]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(y.numel() * y.element_size() for y in h_out)

    def e2e_step():
        for d, h in zip(wl.inputs, h_in):
            d.copy_(h, non_blocking=True)
        wl.step()
        for h, d in zip(h_out, wl.outputs):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps

    peak, peak_kind = peaks()
    gbs = job_value(wl.step_bytes, ms, world)
    if wl.launches == 1:
        # each step is exactly one launch of the streaming kernel, so the
        # kernel's average launch duration over the timed region is the step time
        dom_ms, dom_bytes = ms_local, wl.step_bytes
        dom_timing = "CUDA events around the K timed steps on the launching stream; one launch per step"
    else:
        # the step's streaming launch alone (the step's other launches are
        # tiny): K of them back to back between two events
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            wl.dominant()
        a.record(stream)
        for _ in range(K):
            wl.dominant()
        b.record(stream)
        torch.cuda.synchronize()
        dom_ms, dom_bytes = a.elapsed_time(b) / K, wl.dominant_bytes
        dom_timing = ("the step's GEMV launch alone, K launches back to back between two events on the "
                      "launching stream (" + wl.other_launch + ")")
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    achieved_preq = wl.gemv_kernel_bytes / (gemv_ms * 1e-3) / 1e9
    cfg = dict(wl.config)
    cfg.update({"timed_as": "one CUDA graph of the K steps replayed once after an L2 flush"
                            if g_captured else "K direct calls",
                "direct_calls_ms_per_step": round(direct_ms, 5),
                "l2_flush": f"{L2_FLUSH_BYTES >> 20} MB written just before the timed region",
                "us_per_gemv": round(ms * 1e3 / wl.n_gemv, 3), "gemv_kernel_ms": round(gemv_ms, 5),
                "gemv_kernel_graph_ms": None if graph_ms is None else round(graph_ms, 5),
                "pct_of_hbm_peak": round(100 * gbs / world / peak, 2), "peak_kind": peak_kind,
                "pct_of_8TBs": round(100 * gbs / world / 8000.0, 2), "step_bytes": wl.step_bytes})
    return {
        "metric": METRIC, "value": round(gbs, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": getattr(wl, "dtype", "int8 x uint4 -> int32 block sums, fp32 accumulation"),
        "data": getattr(wl, "data", "synthetic (seeded; Q4_0 nibbles uniform, fp16 scales U[1e-3,4e-3], "
                                    "x N(0,1) with 1% x20)"),
        "config": cfg,
        "e2e": {"value": round(wl.step_bytes / (e2e_ms * 1e-3) / 1e9 * world, 3), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic_record(wl.name, wl.T),
                     "kernel": wl.kernel_name, "algorithmic_bytes_per_launch": dom_bytes,
                     "ms_per_launch": round(dom_ms, 5), "timing": dom_timing,
                     "preq_input": {
                         "achieved": round(achieved_preq, 2), "frac": round(achieved_preq / peak, 4),
                         "ms_per_launch": round(gemv_ms, 5), "algorithmic_bytes_per_launch": wl.gemv_kernel_bytes,
                         "timing": "the same kernel on pre-quantised Q8_0 activations: K launches back to back "
                                   "after the timed region, between two events"}},
        "gpu_launches": wl.launches * K,
        "clocks": clk,
    }


if __name__ == "__main__":
    sys.exit(main())

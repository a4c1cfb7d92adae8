"""The C ABI without a GPU: the library loads, exports every function that
include/qgemv.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

import quantized_q4_weight_gb300 as q
from quantized_q4_weight_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "qgemv.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemv_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    # and the binding knows their signatures
    assert set(names) == set(q._SIGS), set(names) ^ set(q._SIGS)


def test_status_strings(L):
    for code, name in q.STATUS.items():
        assert L.qgemv_status_string(code).decode() == name
    assert L.qgemv_version() >= 100


def test_sizes(L):
    assert L.qgemv_q4_0_bytes(1536, 1536) == 1327104
    assert L.qgemv_q4_0_bytes(151936, 1536) == 131272704
    assert L.qgemv_q4_0_bytes(10, 33) == 0
    assert L.qgemv_q4_0_bytes(0, 32) == 0
    assert L.qgemv_xq_bytes(1, 1536) == 1536 + 96
    assert L.qgemv_xq_bytes(1, 32) == 32 + 16            # 2 scale bytes padded to 16
    assert L.qgemv_xq_bytes(8, 11008) == 8 * 11008 + 8 * 344 * 2
    assert L.qgemv_xq_bytes(0, 32) == 0


def test_layer_set_bytes_match_the_pages(L):
    # minfer README: 0.868 GB/token for Qwen2.5-1.5B (layers + q4 lm_head) and
    # 1.736 GB for 3B; the layer sets alone are 736,985,088 and 1,560,674,304 B.
    import synth
    l15 = sum(L.qgemv_q4_0_bytes(N, K) for _, N, K in synth.layer_set(synth.QWEN25_1P5B_LAYER, 28))
    l3 = sum(L.qgemv_q4_0_bytes(N, K) for _, N, K in synth.layer_set(synth.QWEN25_3B_LAYER, 36))
    assert l15 == 736985088 and l3 == 1560674304
    assert round((l15 + L.qgemv_q4_0_bytes(151936, 1536)) / 1e9, 3) == 0.868
    assert round((l3 + L.qgemv_q4_0_bytes(151936, 2048)) / 1e9, 3) == 1.736


def test_workspace_queries(L):
    # split-K only when a launch has few slabs: a long list needs no partials
    small = L.qgemv_workspace_bytes(1536, 8960, 1)
    assert small > 16384
    assert L.qgemv_workspace_bytes(1536, 8960, 8) > small
    assert L.qgemv_workspace_bytes(1536, 30, 1) == 0
    assert L.qgemv_workspace_bytes(1536, 64, 9) == 0
    items = (q.SeqItem * 2)(q.SeqItem(16, 4096, 8192, 40000, 1536), q.SeqItem(32, 4096, 8192, 1536, 8960))
    # the counter area; on the tensor-core path (T >= 5) a small-group region
    # of segment sums for each of the 152 CTAs (no device here):
    # 15 slabs x 18 segments (K = 8960) x T x 16 rows
    assert L.qgemv_seq_workspace_bytes(items, 2, 1) == 16384
    assert L.qgemv_seq_workspace_bytes(items, 2, 4) == 16384
    for T in (5, 8):
        assert L.qgemv_seq_workspace_bytes(items, 2, T) == 16384 + 152 * 15 * 18 * T * 16 * 4
    # with the tcgen05 kernel switched on, packed lists with N % 16 == 0 and
    # K % 256 == 0 may run on it: 16 KB of counters, then for each of the
    # 2 x 152 warp groups a slot of segment sums (18 segments x 8 x 128 rows)
    tc = 16384 + 2 * 152 * 18 * 8 * 128 * 4
    L.qgemv_set_tc_min_tokens(5)
    try:
        for T in (5, 8):
            assert L.qgemv_seq_workspace_bytes(items, 2, T) == max(16384 + 152 * 15 * 18 * T * 16 * 4, tc)
        assert L.qgemv_seq_workspace_bytes(items, 2, 4) == 16384
    finally:
        L.qgemv_set_tc_min_tokens(0)
    assert L.qgemv_set_tc_min_tokens(10) == 1
    assert L.qgemv_seq_workspace_bytes(items, 0, 1) == 0


FAKE = 1 << 40          # a plausible device address; never dereferenced on these paths


def test_gemv_rejects_bad_arguments(L):
    s = None
    ws = FAKE + (1 << 30)
    ok = dict(W=FAKE, layout=1, xq=FAKE + (1 << 28), y=FAKE + (1 << 29), N=64, K=128, T=1, ws=ws, nbytes=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return L.qgemv_q4_0(a["W"], a["layout"], a["xq"], a["y"], a["N"], a["K"], a["T"], a["ws"], a["nbytes"], s)

    assert call(T=0) == 1 and call(T=9) == 1
    assert call(K=100) == 1 and call(K=0) == 1 and call(N=0) == 1
    assert call(W=None) == 1 and call(xq=None) == 1 and call(y=None) == 1
    assert call(layout=7) == 1
    assert call(W=FAKE + 8) == 2                       # packed weights need 16-byte alignment
    assert call(xq=FAKE + (1 << 28) + 4) == 2
    assert call(y=FAKE + (1 << 29) + 2) == 2
    assert call(ws=None) == 4
    assert call(y=FAKE + 64) == 1                      # y overlaps W
    assert call(y=ws + 256) == 1                       # y overlaps the workspace


def test_other_calls_reject_bad_arguments(L):
    s = None
    assert L.qgemv_pack_q4_0(FAKE, FAKE + 96, 16, 64, s) == 1           # overlap
    assert L.qgemv_pack_q4_0(FAKE, FAKE + (1 << 30) + 8, 16, 64, s) == 2
    assert L.qgemv_quantize_q8_0(FAKE, FAKE + (1 << 30), 0, 64, 1, s) == 1
    assert L.qgemv_quantize_q8_0(FAKE, FAKE + (1 << 30) + 4, 1, 64, 1, s) == 2
    assert L.qgemv_q4_0_argmax(FAKE, 1, FAKE + (1 << 28), None, None, 64, 64, 1, FAKE + (1 << 30), 4096, s) == 1
    items = (q.SeqItem * 2)(q.SeqItem(FAKE, FAKE + (1 << 28), FAKE + (1 << 29), 64, 64),
                            q.SeqItem(FAKE + (1 << 27), FAKE + (1 << 28), FAKE + (1 << 29) + 64, 64, 64))
    assert L.qgemv_q4_0_seq(items, 2, 1, 1, FAKE + (1 << 30), 4096, s) == 1     # two outputs overlap
    assert L.qgemv_q4_0_seq(items, 0, 1, 1, FAKE + (1 << 30), 4096, s) == 1
    mats = (q.GatherMatrix * 1)(q.GatherMatrix(FAKE, 4608, FAKE + (1 << 28), 0, FAKE + (1 << 29), 10, 64, 128))
    assert L.qgemv_q4_0_gather(mats, 1, FAKE + (1 << 31), 2, 4, 1, 1, FAKE + (1 << 30), 4096, s) == 1  # y_stride < T*N
    assert L.qgemv_q4_0_gather(mats, 1, None, 1, 4, 1, 1, FAKE + (1 << 30), 4096, s) == 1
    assert L.qgemv_debug_block_isums(FAKE, 1, FAKE, None, 16, 64, 1, s) == 1
    # requantisation: shapes, null pointers, alignment, output over the input
    out = FAKE + (1 << 30)
    assert L.qgemv_requant_f32_q4_0(FAKE, out, 16, 48, s) == 1
    assert L.qgemv_requant_f32_q4_0(None, out, 16, 64, s) == 1
    assert L.qgemv_requant_f32_q4_0(FAKE + 2, out, 16, 64, s) == 2
    assert L.qgemv_requant_f32_q4_0(FAKE, out + 1, 16, 64, s) == 2
    assert L.qgemv_requant_f32_q4_0(FAKE, FAKE + 4 * 16 * 64 - 2, 16, 64, s) == 1
    assert L.qgemv_requant_q8_0_q4_0(FAKE + 1, out, 16, 64, s) == 2
    assert L.qgemv_requant_q8_0_q4_0(FAKE, FAKE + 34 * 16 * 2 - 18, 16, 64, s) == 1
    assert L.qgemv_requant_q8_0_q4_0(FAKE, out, 0, 64, s) == 1
    # sequences with the epilogue: x_f32 flag, misaligned bias, residual over another output
    ep = (q.SeqEpItem * 2)(q.SeqEpItem(FAKE, FAKE + (1 << 28), FAKE + (1 << 29), 64, 64, None, None),
                           q.SeqEpItem(FAKE, FAKE + (1 << 28), FAKE + (1 << 29) + 4096, 64, 64, None, None))
    ws = FAKE + (1 << 30)
    assert L.qgemv_q4_0_seq_ep(ep, 2, 1, 1, 2, ws, 1 << 20, s) == 1
    ep[0].bias = FAKE + (1 << 27) + 2
    assert L.qgemv_q4_0_seq_ep(ep, 2, 1, 1, 0, ws, 1 << 20, s) == 2
    ep[0].bias = None
    ep[0].residual = FAKE + (1 << 29) + 4096                          # item 1's output
    assert L.qgemv_q4_0_seq_ep(ep, 2, 1, 1, 0, ws, 1 << 20, s) == 1
    # the FFN chain with a residual: misaligned, or over the workspace
    need = L.qgemv_ffn_workspace_bytes(256, 512, 2)
    x, y = FAKE + (1 << 28), FAKE + (1 << 29)
    assert L.qgemv_q4_0_ffn_residual(FAKE, FAKE, FAKE, 1, x, None, y, 256, 512, 2, ws, need, s) == 1
    assert L.qgemv_q4_0_ffn_residual(FAKE, FAKE, FAKE, 1, x, y + 4098, y, 256, 512, 2, ws, need, s) == 2
    assert L.qgemv_q4_0_ffn_residual(FAKE, FAKE, FAKE, 1, x, ws + 256, y, 256, 512, 2, ws, need, s) == 1


def test_fp32_calls_reject_bad_arguments(L):
    """The fp32-input calls check their own input ranges: alignment (4 bytes),
    null pointers, and outputs that overlap the fp32 inputs or the workspace."""
    s = None
    ws = FAKE + (1 << 30)
    x = FAKE + (1 << 28)
    # argmax_f32: missing idx, misaligned x, y overlapping x
    assert L.qgemv_q4_0_argmax_f32(FAKE, 1, x, None, None, 64, 64, 1, ws, 4096, s) == 1
    assert L.qgemv_q4_0_argmax_f32(FAKE, 1, x + 2, None, FAKE + (1 << 29), 64, 64, 1, ws, 4096, s) == 2
    assert L.qgemv_q4_0_argmax_f32(FAKE, 1, x, x + 4, FAKE + (1 << 29), 64, 64, 1, ws, 4096, s) == 1
    # gemv_f32: x only needs 4-byte alignment, y overlapping the workspace is refused
    assert L.qgemv_q4_0_f32(FAKE, 1, x + 2, FAKE + (1 << 29), 64, 64, 1, ws, 1 << 20, s) == 2
    assert L.qgemv_q4_0_f32(FAKE, 1, x, ws + 256, 64, 64, 1, ws, 1 << 20, s) == 1
    # seq_f32: an output overlapping another item's fp32 input
    items = (q.SeqF32Item * 2)(q.SeqF32Item(FAKE, x, FAKE + (1 << 29), 64, 64),
                               q.SeqF32Item(FAKE, x + 4096, x, 64, 64))
    assert L.qgemv_q4_0_seq_f32(items, 2, 1, 1, ws, 1 << 20, s) == 1
    items2 = (q.SeqF32Item * 1)(q.SeqF32Item(FAKE, x + 2, FAKE + (1 << 29), 64, 64))
    assert L.qgemv_q4_0_seq_f32(items2, 1, 1, 1, ws, 1 << 20, s) == 2
    # gather_f32: misaligned x stride, y_stride below T * N
    mats = (q.GatherF32Matrix * 1)(q.GatherF32Matrix(FAKE, 4608, x, 6, FAKE + (1 << 29), 64, 64, 128))
    assert L.qgemv_q4_0_gather_f32(mats, 1, FAKE + (1 << 31), 2, 4, 1, 1, ws, 4096, s) == 2
    mats2 = (q.GatherF32Matrix * 1)(q.GatherF32Matrix(FAKE, 4608, x, 512, FAKE + (1 << 29), 10, 64, 128))
    assert L.qgemv_q4_0_gather_f32(mats2, 1, FAKE + (1 << 31), 2, 4, 1, 1, ws, 4096, s) == 1
    assert L.qgemv_gather_f32_workspace_bytes(mats2, 1, 2, 1) == 0
    assert L.qgemv_seq_f32_workspace_bytes(items, 2, 1) >= 16384


def test_noalloc_refusals_before_any_cuda_call(L):
    """The allocation-free argmax checks every argument on the host first:
    these refusals make no CUDA call (so they also pass without a GPU)."""
    s = None
    W, xq, idx = FAKE, FAKE + (1 << 28), FAKE + (1 << 29)
    f = L.qgemv_q4_0_argmax_noalloc
    assert f(W, 1, xq, None, idx, 64, 64, 0, s) == 1              # T out of range
    assert f(W, 1, xq, None, idx, 64, 64, 9, s) == 1
    assert f(W, 1, xq, None, idx, 64, 100, 1, s) == 1             # K % 32 != 0
    assert f(W, 1, xq, None, idx, 0, 64, 1, s) == 1
    # split-K partials of 600 slabs x 512 blocks x 8 tokens: 9.8 MB > 4 MiB
    assert f(None, 1, None, None, None, 9600, 16384, 8, s) == 3   # QGEMV_ERR_UNSUPPORTED
    assert L.qgemv_workspace_bytes(9600, 16384, 8) > 4 << 20
    assert f(None, 1, xq, None, idx, 64, 64, 1, s) == 1           # null weights
    assert f(W, 1, xq, None, None, 64, 64, 1, s) == 1             # null idx
    assert f(W, 1, xq + 4, None, idx, 64, 64, 1, s) == 2          # misaligned activations
    assert f(W + 8, 1, xq, None, idx, 64, 64, 1, s) == 2          # packed weights need 16 bytes
    assert f(W, 1, xq, idx - 8, idx, 64, 64, 1, s) == 1           # y over idx
    assert f(W, 1, xq, W + 64, idx, 64, 64, 1, s) == 1            # y over the weights


def test_tensor_core_isums_hook_rejects_bad_arguments(L):
    s = None
    assert L.qgemv_debug_block_isums_tc(FAKE, 1, FAKE, FAKE, 16, 64, 1, 2, s) == 1
    assert L.qgemv_debug_block_isums_tc(FAKE, 1, FAKE, None, 16, 64, 1, 0, s) == 1
    assert L.qgemv_debug_block_isums_tc(FAKE, 1, FAKE, FAKE, 16, 64, 9, 0, s) == 1
    assert L.qgemv_debug_block_isums_tc(FAKE + 8, 1, FAKE, FAKE, 16, 64, 1, 0, s) == 2


def test_gs64_calls_reject_bad_arguments(L):
    s = None
    assert L.qgemv_gs64_bytes(16, 96) == 0 and L.qgemv_gs64_bytes(16, 128) == 36 * 16 * 2
    assert L.qgemv_gs64_workspace_bytes(16, 96, 1) == 0
    W, qa, sa, y = FAKE, FAKE + (1 << 28), FAKE + (1 << 29), FAKE + (1 << 30)
    assert L.qgemv_gs64(W, qa, sa, y, 64, 96, 1, None, 0, s) == 1            # K % 64 != 0
    assert L.qgemv_gs64(W, qa, sa, y, 64, 128, 9, None, 0, s) == 1           # T out of range
    assert L.qgemv_gs64(W + 8, qa, sa, y, 64, 128, 1, None, 0, s) == 2       # packed weights: 16 bytes
    assert L.qgemv_gs64(W, qa + 4, sa, y, 64, 128, 1, None, 0, s) == 2       # codes: 16 bytes
    assert L.qgemv_gs64(W, qa, sa, W + 64, 64, 128, 1, None, 0, s) == 1      # y over the weights
    assert L.qgemv_gs64(W, qa, sa, qa + 16, 64, 128, 1, None, 0, s) == 1     # y over the codes
    assert L.qgemv_pack_gs64(W, sa, W + 64, 16, 128, s) == 1                 # output over the nibbles
    assert L.qgemv_pack_gs64(W, sa + 2, y, 16, 128, s) == 2
    assert L.qgemv_quantize_vec_i8(W, qa, sa, 0, 64, s) == 1
    assert L.qgemv_quantize_vec_i8(W, W + 16, sa, 1, 64, s) == 1             # codes over x
    assert L.qgemv_quantize_vec_i8(W + 2, qa, sa, 1, 64, s) == 2
    xa = FAKE + (1 << 31)
    assert L.qgemv_gs64_f32(W, xa, y, 64, 96, 1, None, 0, s) == 1             # K % 64 != 0
    assert L.qgemv_gs64_f32(W, xa, y, 64, 128, 0, None, 0, s) == 1            # T out of range
    assert L.qgemv_gs64_f32(W, None, y, 64, 128, 1, None, 0, s) == 1          # no x
    assert L.qgemv_gs64_f32(W, xa + 2, y, 64, 128, 1, None, 0, s) == 2        # x: 4 bytes
    assert L.qgemv_gs64_f32(W + 8, xa, y, 64, 128, 1, None, 0, s) == 2        # packed weights: 16 bytes
    assert L.qgemv_gs64_f32(W, xa, xa + 64, 64, 128, 1, None, 0, s) == 1      # y over x
    assert L.qgemv_gs64_f32(W, xa, W + 64, 64, 128, 1, None, 0, s) == 1       # y over the weights

"""The allocation-free lm_head argmax (qgemv_q4_0_argmax_noalloc) against
the workspace-taking entry point.

It serves callers that cannot allocate device memory where they run the
lm_head (a plugin handed only its tensors, a runtime with a fixed memory
budget): its scratch is a fixed array inside the library.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

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
    return oracle.load()


def noalloc(W, xq, y, idx, N, K, T):
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return q.lib().qgemv_q4_0_argmax_noalloc(ctypes.c_void_p(W.data_ptr()), q.W_PACKED,
                                             ctypes.c_void_p(xq.data_ptr()),
                                             ctypes.c_void_p(y.data_ptr()) if y is not None else None,
                                             ctypes.c_void_p(idx.data_ptr()), N, K, T, s)


# (20000, 1536, 3) splits K and so also uses the scratch for partial sums.
@pytest.mark.parametrize("N,K,T", [(151936, 1536, 1), (20000, 1536, 3), (4099, 544, 8)])
def test_noalloc_matches_workspace_entry_point(orc, N, K, T):
    Wg = synth.q4_0_weights(91 + N, N, K)
    W = q.pack_q4_0(to_dev(Wg), N, K)
    x = synth.activations(92 + N, T, K)
    xq = q.quantize_q8_0(torch.from_numpy(x).to(DEV), T, K)
    ws = q.new_workspace(q.workspace_bytes(N, K, T))
    y_ref = torch.empty((T, N), dtype=torch.float32, device=DEV)
    idx_ref = q.gemv_argmax(W, q.W_PACKED, xq, N, K, T, ws, y=y_ref).cpu().numpy()
    y_ref = y_ref.cpu().numpy()
    y64, S = orc.gemv(Wg, N, K, orc.quantize(x), T)
    for call in range(2):                    # two calls in a row share the scratch
        y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
        idx = torch.full((T,), -1, dtype=torch.int64, device=DEV)
        assert noalloc(W, xq, y, idx, N, K, T) == 0
        torch.cuda.synchronize()
        assert q.device_status() == 0
        yh = y.cpu().numpy()
        assert np.array_equal(idx.cpu().numpy(), idx_ref), call
        check_close(yh, y64, S, f"noalloc call {call}")
        assert np.array_equal(yh.view(np.int32), y_ref.view(np.int32)), call
    # the usual lm_head use: no logits, the index only
    idx = torch.full((T,), -1, dtype=torch.int64, device=DEV)
    assert noalloc(W, xq, None, idx, N, K, T) == 0
    torch.cuda.synchronize()
    assert q.device_status() == 0
    assert np.array_equal(idx.cpu().numpy(), idx_ref)


def test_noalloc_rejects_shapes_beyond_its_scratch(orc):
    # 600 slabs of 16 rows (split K) with K = 16384 at T = 8 need 9.8 MB of
    # partial sums, beyond the 4 MiB scratch.  Every buffer has its full size,
    # so that the call could run safely if it were accepted.
    N, K, T = 9600, 16384, 8
    W = torch.zeros(q.q4_0_bytes(N, K), dtype=torch.uint8, device=DEV)
    xq = torch.zeros(q.xq_bytes(T, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((T, N), dtype=torch.float32, device=DEV)
    idx = torch.empty(T, dtype=torch.int64, device=DEV)
    assert noalloc(W, xq, y, idx, N, K, T) == 3                    # QGEMV_ERR_UNSUPPORTED

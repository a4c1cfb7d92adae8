"""The decode FFN step through the C ABI against the CPU oracle.

Bit-exact: the Q8_0 codes of SiLU(g) * u against the oracle applied to the
same g, u (the GPU's own gate and up outputs in the chain); the chain's y
against the same down GEMV run alone on those codes.  Within the output
bound: y against the oracle's fp64 down projection of the oracle's codes.
The exponential both sides use is checked against CUDA's expf (torch.exp).
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_q4_weight_gb300 as q
import synth
from tests.gpu_util import blocks_to_planar, to_dev

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


def test_exp_against_cuda_expf(orc):
    """The FFN's exponential (Cody-Waite; the oracle's and the kernel's are the
    same fp32 operations) within 3 ulp of CUDA's expf over [-87, 88]."""
    x = np.linspace(-87.0, 88.0, 1000003).astype(np.float32)
    mine = orc.exp_f32(x)
    cuda = torch.exp(torch.from_numpy(x).to(DEV)).cpu().numpy()
    ulp = np.spacing(cuda)
    assert np.all(np.abs(mine.astype(np.float64) - cuda.astype(np.float64)) <= 3 * ulp)


@pytest.mark.parametrize("T,F", [(1, 32), (1, 8960), (3, 512), (8, 11008), (5, 2048)])
def test_silu_mul_q8_bit_exact(orc, T, F):
    rng = np.random.default_rng(700 + T + F)
    g = (rng.standard_normal((T, F)) * 4).astype(np.float32)
    u = rng.standard_normal((T, F)).astype(np.float32)
    # edges: the clamp range of exp, zeros of both signs, tiny values, a zero block
    g.flat[:8] = [100.0, -100.0, 88.5, -87.5, 0.0, -0.0, 1e-30, -1e-30]
    if F >= 64:
        u[0, 32:64] = 0.0
    hq = q.silu_mul_q8(torch.from_numpy(g).to(DEV), torch.from_numpy(u).to(DEV), T, F).cpu().numpy()
    ref, _ = orc.silu_mul_quantize(g, u)
    assert np.array_equal(hq, blocks_to_planar(ref, q.xq_bytes(T, F)))


@pytest.mark.parametrize("d_model,d_ff,T", [(1536, 8960, 1), (256, 512, 5), (2048, 11008, 8), (96, 160, 2)])
def test_ffn_chain(orc, d_model, d_ff, T):
    seed = 800 + d_model + T
    Wg_ggml = synth.q4_0_weights(seed, d_ff, d_model)
    Wu_ggml = synth.q4_0_weights(seed + 1, d_ff, d_model)
    Wd_ggml = synth.q4_0_weights(seed + 2, d_model, d_ff)
    Wg = q.pack_q4_0(to_dev(Wg_ggml), d_ff, d_model)
    Wu = q.pack_q4_0(to_dev(Wu_ggml), d_ff, d_model)
    Wd = q.pack_q4_0(to_dev(Wd_ggml), d_model, d_ff)
    x = synth.activations(seed + 3, T, d_model)
    xd = torch.from_numpy(x).to(DEV)
    ws = q.new_workspace(q.ffn_workspace_bytes(d_model, d_ff, T))
    y = q.ffn(Wg, Wu, Wd, q.W_PACKED, xd, d_model, d_ff, T, ws)
    # the pieces alone: gate and up, the SiLU * up codes, the down GEMV on them
    g = q.gemv_f32(Wg, q.W_PACKED, xd, d_ff, d_model, T, q.new_workspace(q.workspace_bytes(d_ff, d_model, T)))
    u = q.gemv_f32(Wu, q.W_PACKED, xd, d_ff, d_model, T, q.new_workspace(q.workspace_bytes(d_ff, d_model, T)))
    hq = q.silu_mul_q8(g, u, T, d_ff)
    y1 = q.gemv(Wd, q.W_PACKED, hq, d_model, d_ff, T, q.new_workspace(q.workspace_bytes(d_model, d_ff, T)))
    assert torch.equal(y.cpu().view(torch.int32), y1.cpu().view(torch.int32))
    # against the oracle: codes bit-exact from the GPU's own g, u; y within the bound
    ref_hq, _ = orc.silu_mul_quantize(g.cpu().numpy(), u.cpu().numpy())
    assert np.array_equal(hq.cpu().numpy(), blocks_to_planar(ref_hq, q.xq_bytes(T, d_ff)))
    y64, S = orc.gemv(Wd_ggml, d_model, d_ff, ref_hq, T)
    err = np.abs(y.cpu().numpy().astype(np.float64) - y64)
    assert np.all(err <= oracle.tolerance(S)), f"worst excess {np.max(err - oracle.tolerance(S))}"
    # the gate and up outputs themselves are within their own bound
    g64, Sg = orc.gemv(Wg_ggml, d_ff, d_model, orc.quantize(x), T)
    assert np.all(np.abs(g.cpu().numpy().astype(np.float64) - g64) <= oracle.tolerance(Sg))
    assert q.device_status() == 0


@pytest.mark.parametrize("d_model,d_ff,T", [(1536, 8960, 1), (2048, 11008, 8), (256, 512, 5)])
def test_ffn_residual(orc, d_model, d_ff, T):
    """The chain with a residual on down: y equals the plain chain's y plus
    the residual (one fp32 add), separate and in place; within the bound of
    the oracle's fp64 down projection plus the residual."""
    seed = 900 + d_model + T
    Wg_ggml = synth.q4_0_weights(seed, d_ff, d_model)
    Wd_ggml = synth.q4_0_weights(seed + 2, d_model, d_ff)
    Wg = q.pack_q4_0(to_dev(Wg_ggml), d_ff, d_model)
    Wu = q.pack_q4_0(to_dev(synth.q4_0_weights(seed + 1, d_ff, d_model)), d_ff, d_model)
    Wd = q.pack_q4_0(to_dev(Wd_ggml), d_model, d_ff)
    xd = torch.from_numpy(synth.activations(seed + 3, T, d_model)).to(DEV)
    r = torch.from_numpy(synth.activations(seed + 4, T, d_model)).to(DEV)
    ws = q.new_workspace(q.ffn_workspace_bytes(d_model, d_ff, T))
    y0 = q.ffn(Wg, Wu, Wd, q.W_PACKED, xd, d_model, d_ff, T, ws)
    y1 = q.ffn_residual(Wg, Wu, Wd, q.W_PACKED, xd, r, d_model, d_ff, T, ws)
    want = (y0 + r).cpu()
    assert torch.equal(y1.cpu().view(torch.int32), want.view(torch.int32))
    h = r.clone()                                                  # in place: h += FFN(x)
    q.ffn_residual(Wg, Wu, Wd, q.W_PACKED, xd, h, d_model, d_ff, T, ws, y=h)
    assert torch.equal(h.cpu().view(torch.int32), want.view(torch.int32))
    # against the oracle: the codes of the GPU's own gate and up, then fp64 down + residual
    g = q.gemv_f32(Wg, q.W_PACKED, xd, d_ff, d_model, T, q.new_workspace(q.workspace_bytes(d_ff, d_model, T)))
    u = q.gemv_f32(Wu, q.W_PACKED, xd, d_ff, d_model, T, q.new_workspace(q.workspace_bytes(d_ff, d_model, T)))
    ref_hq, _ = orc.silu_mul_quantize(g.cpu().numpy(), u.cpu().numpy())
    y64, S = orc.gemv_ep(Wd_ggml, d_model, d_ff, ref_hq, T, None, r.cpu().numpy())
    err = np.abs(y1.cpu().numpy().astype(np.float64) - y64)
    assert np.all(err <= oracle.tolerance(S))
    assert q.device_status() == 0


def test_ffn_errors():
    d_model, d_ff, T = 256, 512, 2
    W = torch.zeros(q.q4_0_bytes(d_ff, d_model), dtype=torch.uint8, device=DEV)
    x = torch.zeros((T, d_model), dtype=torch.float32, device=DEV)
    need = q.ffn_workspace_bytes(d_model, d_ff, T)
    assert need > 0 and q.ffn_workspace_bytes(d_model, 33, T) == 0
    with pytest.raises(q.QgemvError, match="WORKSPACE"):
        q.ffn(W, W, W, q.W_PACKED, x, d_model, d_ff, T, q.new_workspace(need)[: need - 256])
    ws = q.new_workspace(need)
    with pytest.raises(q.QgemvError, match="INVALID_ARG"):   # y inside the workspace
        q.ffn(W, W, W, q.W_PACKED, x, d_model, d_ff, T, ws, y=ws[:4 * T * d_model].view(torch.float32).view(T, d_model))
    assert q.device_status() == 0
    r = torch.zeros((T, d_model), dtype=torch.float32, device=DEV)
    y = torch.zeros((T, d_model), dtype=torch.float32, device=DEV)
    with pytest.raises(q.QgemvError, match="INVALID_ARG"):   # residual over the workspace
        q.ffn_residual(W, W, W, q.W_PACKED, x, ws[:4 * T * d_model].view(torch.float32).view(T, d_model), d_model,
                       d_ff, T, ws, y=y)
    with pytest.raises(q.QgemvError, match="INVALID_ARG"):   # residual shifted over y
        yy = torch.zeros(T * d_model + 1, dtype=torch.float32, device=DEV)
        q.ffn_residual(W, W, W, q.W_PACKED, x, yy[1:].view(T, d_model), d_model, d_ff, T, ws,
                       y=yy[:T * d_model].view(T, d_model))
    assert q.device_status() == 0


# the fused launch (T <= 4, packed) against the three launches: many h blocks
# per CTA and fewer h blocks than CTAs, partial segments in both projections
# (d_model = 96, d_ff = 8960 and 160), several rounds of h blocks (d_ff = 23 x
# 32 x 152 > 4 per CTA), with and without the residual, repeated calls
@pytest.mark.parametrize("d_model,d_ff,T", [(1536, 8960, 1), (1536, 8960, 4), (96, 160, 2), (2048, 11008, 3),
                                           (512, 32 * 152 * 5, 1), (4096, 1024, 2)])
def test_ffn_fused_matches_three_launches(orc, d_model, d_ff, T):
    seed = 1000 + d_model + d_ff + T
    Wg = q.pack_q4_0(to_dev(synth.q4_0_weights(seed, d_ff, d_model)), d_ff, d_model)
    Wu = q.pack_q4_0(to_dev(synth.q4_0_weights(seed + 1, d_ff, d_model)), d_ff, d_model)
    Wd = q.pack_q4_0(to_dev(synth.q4_0_weights(seed + 2, d_model, d_ff)), d_model, d_ff)
    xd = torch.from_numpy(synth.activations(seed + 3, T, d_model)).to(DEV)
    r = torch.from_numpy(synth.activations(seed + 4, T, d_model)).to(DEV)
    ws = q.new_workspace(q.ffn_workspace_bytes(d_model, d_ff, T))
    try:
        q.set_ffn_fused(False)
        y3 = q.ffn(Wg, Wu, Wd, q.W_PACKED, xd, d_model, d_ff, T, ws).cpu()
        y3r = q.ffn_residual(Wg, Wu, Wd, q.W_PACKED, xd, r, d_model, d_ff, T, ws).cpu()
        q.set_ffn_fused(True)
        for _ in range(2):                                    # the counters are left at zero
            y1 = q.ffn(Wg, Wu, Wd, q.W_PACKED, xd, d_model, d_ff, T, ws).cpu()
            assert torch.equal(y1.view(torch.int32), y3.view(torch.int32))
        y1r = q.ffn_residual(Wg, Wu, Wd, q.W_PACKED, xd, r, d_model, d_ff, T, ws).cpu()
        assert torch.equal(y1r.view(torch.int32), y3r.view(torch.int32))
        h = r.clone()                                         # in place: h += FFN(x)
        q.ffn_residual(Wg, Wu, Wd, q.W_PACKED, xd, h, d_model, d_ff, T, ws, y=h)
        assert torch.equal(h.cpu().view(torch.int32), y3r.view(torch.int32))
    finally:
        q.set_ffn_fused(True)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    assert int(ws[:16384].count_nonzero()) == 0

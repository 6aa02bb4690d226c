"""FC-norm on the GPU (normalisation kernel + tcgen05 GEMM) through the C ABI against
the float64 oracle, within the bound that bf16 rounding of the normalised
inputs and of the output implies: |gpu - ref| <= 2^-8 (sum_k |x_k||w_k| +
|ref|)."""

import numpy as np
import pytest
import torch

from oracle import fcnorm as ofc
from speculative_decoding_verification_73_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


def _f64(t):
    return t.to(torch.float64).numpy()


def _misaligned(t):
    """A copy of t on the GPU whose data starts 4 bytes past a 16-byte boundary."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    flat[1:] = t.reshape(-1).cuda()
    view = flat[1:].view(t.shape)
    assert view.data_ptr() % 16 != 0
    return view


def run_case(wl, norm, with_bias=True, with_beta=True, eps=1e-5, misalign_gamma=False):
    ctx = binding.SpecVerify(1, 1, 16, torch.float32)
    h = [x.cuda() for x in wl.h]
    gamma = None
    if norm != binding.SV_NORM_NONE:
        gamma = _misaligned(wl.gamma) if misalign_gamma else wl.gamma.cuda()
    beta = wl.beta.cuda() if (norm == binding.SV_NORM_LAYER and with_beta) else None
    bias = wl.bias.cuda() if with_bias else None
    out = binding.spec_verify_fc_norm(ctx.ctx, norm, *h, wl.weight.cuda(), gamma=gamma, beta=beta,
                                      bias=bias, eps=eps)
    code, bits = ctx.get_error()
    assert code == 0 and bits == 0
    got = out.float().cpu().numpy().astype(np.float64)
    hs = [_f64(x) for x in wl.h]
    g = _f64(wl.gamma) if gamma is not None else None
    b = _f64(wl.beta) if beta is not None else None
    ref = ofc.fc_norm(*hs, _f64(wl.weight), norm, g, b, _f64(wl.bias) if with_bias else None, eps)
    bound = ofc.abs_bound(*hs, _f64(wl.weight), norm, g, b, eps)
    err = np.abs(got - ref)
    tol = 2.0 ** -8 * (bound + np.abs(ref)) + 1e-6
    worst = float((err / tol).max())
    assert (err <= tol).all(), f"worst error / tolerance {worst:.3g}"
    ctx.close()
    return worst


CASES = [
    ("layer-bias", 200, 256, 384, binding.SV_NORM_LAYER, True, True),
    ("rms-ragged-out", 130, 64, 100, binding.SV_NORM_RMS, False, False),
    ("none-one-token", 1, 128, 256, binding.SV_NORM_NONE, True, False),
    ("layer-no-beta", 129, 192, 264, binding.SV_NORM_LAYER, False, False),
    ("layer-medium", 512, 1024, 1024, binding.SV_NORM_LAYER, True, True),
    ("layer-wide-row", 33, 4160, 96, binding.SV_NORM_LAYER, True, True),   # rows past the register form
    ("rms-widest-register-row", 40, 4096, 72, binding.SV_NORM_RMS, True, False),
    ("none-medium", 300, 512, 640, binding.SV_NORM_NONE, True, False),    # 3 x 8 K steps, ragged T
    ("rms-medium", 257, 1024, 512, binding.SV_NORM_RMS, False, False),
]


@pytest.mark.parametrize("name,T,d,d_out,norm,bias,beta", CASES)
def test_fc_norm_matches_oracle(name, T, d, d_out, norm, bias, beta):
    wl = workloads.make_fcnorm(T, d, d_out, gen_seed=sum(map(ord, name)))
    worst = run_case(wl, norm, bias, beta)
    print(f"{name}: worst error / tolerance {worst:.3f}")


def test_gamma_not_16_byte_aligned():
    """gamma off a 16-byte boundary: the one-warp-per-row normalisation
    (scalar gamma / beta loads) writes X before the GEMM."""
    wl = workloads.make_fcnorm(96, 256, 192, gen_seed=77)
    run_case(wl, binding.SV_NORM_LAYER, True, True, misalign_gamma=True)


def test_selector_weights_return_the_normalised_segment():
    """W = [0 I 0]: the output is the middle segment's LayerNorm, rounded."""
    T, d = 64, 128
    wl = workloads.make_fcnorm(T, d, d, gen_seed=7)
    w = torch.zeros(d, 3 * d, dtype=torch.float64)
    w[:, d:2 * d] = torch.eye(d, dtype=torch.float64)
    wl.weight = w.to(torch.bfloat16)
    run_case(wl, binding.SV_NORM_LAYER, with_bias=False, with_beta=True)


@pytest.mark.parametrize("norm", [binding.SV_NORM_LAYER, binding.SV_NORM_NONE], ids=["layernorm", "none"])
def test_full_size_on_sampled_rows(norm):
    """T = d = d_out = 4096 (the benchmarked size, 32 m-blocks of output
    tiles of the persistent GEMM, every CTA several tiles), through X and
    straight from the hidden states: 64 sampled tokens against the oracle on
    those tokens alone (tokens are normalised independently)."""
    T = d = d_out = 4096
    wl = workloads.make_fcnorm(T, d, d_out, gen_seed=2026)
    ctx = binding.SpecVerify(1, 1, 16, torch.float32)
    h = [x.cuda() for x in wl.h]
    layer = norm == binding.SV_NORM_LAYER
    out = binding.spec_verify_fc_norm(ctx.ctx, norm, *h, wl.weight.cuda(),
                                      gamma=wl.gamma.cuda() if layer else None,
                                      beta=wl.beta.cuda() if layer else None, bias=wl.bias.cuda())
    assert ctx.get_error() == (0, 0)
    rows = np.sort(np.random.default_rng(4).choice(T, size=64, replace=False))
    rows[0], rows[-1] = 0, T - 1
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    hs = [_f64(x[torch.from_numpy(rows)]) for x in wl.h]
    g = _f64(wl.gamma) if layer else None
    bt = _f64(wl.beta) if layer else None
    ref = ofc.fc_norm(*hs, _f64(wl.weight), norm, g, bt, _f64(wl.bias), 1e-5)
    bound = ofc.abs_bound(*hs, _f64(wl.weight), norm, g, bt, 1e-5)
    err = np.abs(got - ref)
    tol = 2.0 ** -8 * (bound + np.abs(ref)) + 1e-6
    assert (err <= tol).all(), f"worst error / tolerance {float((err / tol).max()):.3g}"
    ctx.close()


@pytest.mark.parametrize("T,d_out", [(640, 3872), (640, 4832), (640, 5792), (1280, 3392), (128, 256)])
@pytest.mark.parametrize("norm", [binding.SV_NORM_LAYER, binding.SV_NORM_NONE], ids=["layernorm", "none"])
def test_every_tile_width(T, d_out, norm):
    """The GEMM picks its output tile width (256, 224, 192, 160 or 128
    columns) from the shape and the SM count, and its ring depth from the
    width; on a 152-SM GB300 these shapes take 160, 192, 224, 256 and 128
    columns respectively (ragged last tiles included), through X
    (LayerNorm) and straight from the hidden states (no normalisation).  A
    narrow d keeps each case quick."""
    wl = workloads.make_fcnorm(T, 64, d_out, gen_seed=T + d_out)
    run_case(wl, norm, True, norm == binding.SV_NORM_LAYER)

"""Helpers shared by the GPU parity tests."""
import pytest
import torch

import sequence_attention_seq_gb300 as uly

# Attention tolerances against the fp64 oracle (bf16 I/O: fp32 accumulation, bf16 output).
TOL = {torch.float32: (1e-5, None), torch.bfloat16: (1.5e-2, 2e-3)}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    uly.load_library()  # a GPU without the built library is a failure, not a skip


def assert_close(got, ref, dtype, what=""):
    """got: CUDA/CPU tensor in the I/O dtype; ref: float64 oracle values."""
    g = got.detach().to("cpu", torch.float64)
    r = ref.to(torch.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    err = (g - r).abs()
    max_abs, mean_tol = TOL[dtype]
    assert torch.isfinite(g).all(), f"{what}: non-finite output"
    assert err.max().item() <= max_abs, f"{what}: max-abs {err.max().item():.3e} > {max_abs}"
    if mean_tol is not None:
        assert err.mean().item() <= mean_tol, f"{what}: mean-abs {err.mean().item():.3e} > {mean_tol}"
    return err.max().item(), err.mean().item()


# Gradients (bf16 I/O): every element within 1.5e-2 + 2^-7 |ref|, mean-abs <= 2e-3.  The
# absolute part is the output tolerance; the relative part covers the final rounding to
# bf16 (at most 2^-8 |ref|) plus the bf16 rounding of the P and dS operands of the tile
# products (at most 2^-8 of each term), which matter once gradients exceed 1 in magnitude.
GRAD_ATOL, GRAD_RTOL, GRAD_MEAN = 1.5e-2, 2.0 ** -7, 2e-3


def assert_close_grad(got, ref, what=""):
    g = got.detach().to("cpu", torch.float64)
    r = ref.to(torch.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite gradient"
    err = (g - r).abs()
    bound = GRAD_ATOL + GRAD_RTOL * r.abs()
    worst = (err / bound).max().item()
    assert worst <= 1.0, f"{what}: error {err.max().item():.3e} exceeds the bound (ratio {worst:.2f})"
    assert err.mean().item() <= GRAD_MEAN, f"{what}: mean-abs {err.mean().item():.3e} > {GRAD_MEAN}"
    return err.max().item(), err.mean().item()


# Element-wise bound scaled by the magnitude of each gradient element's terms
# (oracle.attention_bwd_magnitudes): |err| <= 1.5e-2 + 2^-7 |ref| + 2^-8 m.  Each term of a
# gradient sum is rounded to bf16 (P and dS before their tile products; D is formed from
# the bf16 output O), so the error of the sum is at most 2^-8 times the sum of the terms'
# magnitudes -- the textbook bound for a sum of rounded products.  Used where the bound above
# does not apply:
# - saturated softmax inputs, where dS = P (dP - D) is a small difference of large terms;
# - K/V heads shared by more than 4 query heads, where each dK/dV element sums many
#   bf16-rounded dS (or P) terms of both signs, whose rounding error scales with the sum of
#   their magnitudes, not with the (partly cancelled) result.
# An emulation of the kernel's roundings in float64 meets it with ratio <= 0.28 on both.
def assert_grad_within_rounding(got, ref, mag, what="", mean_tol=None):
    g = got.detach().to("cpu", torch.float64)
    r = ref.to(torch.float64)
    m = mag.to(torch.float64)
    assert g.shape == r.shape == m.shape, (g.shape, r.shape, m.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite gradient"
    err = (g - r).abs()
    bound = GRAD_ATOL + GRAD_RTOL * r.abs() + 2.0 ** -8 * m
    worst = (err / bound).max().item()
    assert worst <= 1.0, f"{what}: error {err.max().item():.3e} exceeds the bound (ratio {worst:.2f})"
    if mean_tol is not None:
        assert err.mean().item() <= mean_tol, f"{what}: mean-abs {err.mean().item():.3e} > {mean_tol}"
    return worst


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def device_ok():
    assert uly.ulysses_device_status(clear=True) == 0, "a kernel's bounded wait gave up"

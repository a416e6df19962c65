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


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def device_ok():
    assert uly.ulysses_device_status(clear=True) == 0, "a kernel's bounded wait gave up"

"""ulysses_dist_attn_fwd_noalloc, the entry point for callers that cannot allocate device
memory (their own pool already holds what they may use, or their host runtime gives them
no allocator): called through the C ABI on two calls in a row (the second call finds the
first call's data still in the library's fixed scratch), its output must equal the regular
unfused ulysses_dist_attn_fwd bit for bit -- both run the same kernels, so any difference
is a scratch-addressing or stale-data fault -- and match the oracle within the tolerances
the other tests use.

Collected last on purpose, so a run that stops at the first failure has already run
every other test."""
import ctypes

import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (1.5e-2, 2e-3), torch.float32: (1e-5, None)}
CODE = {torch.float32: 0, torch.bfloat16: 1}


def _ptrs(ts):
    a = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t.data_ptr()
    return a


def _noalloc(lib, qs, ks, vs, out, causal):
    P = len(qs)
    b, S, hq, d = qs[0].shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ulysses_dist_attn_fwd_noalloc(P, b, S * P, hq, ks[0].shape[2], d, CODE[qs[0].dtype], int(causal),
                                             _ptrs(qs), _ptrs(ks), _ptrs(vs), _ptrs(out), stream)


def _close(a, b, dtype):
    err = (a.double() - b.double()).abs()
    max_abs, mean_abs = TOL[dtype]
    assert err.max().item() <= max_abs
    if mean_abs is not None:
        assert err.mean().item() <= mean_abs


@pytest.mark.parametrize("P,b,s,hq,hkv,d,dtype,causal", [
    (4, 1, 1024, 8, 4, 128, torch.bfloat16, True),
    (2, 2, 320, 4, 2, 64, torch.bfloat16, False),
    (2, 1, 64, 4, 4, 16, torch.float32, False),
])
def test_noalloc_matches_regular_entry_point_twice(P, b, s, hq, hkv, d, dtype, causal):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sequence_attention_seq_gb300 import build as uly_build

    uly_build.build()
    lib = uly.load_library()
    for seed in (1, 2):  # two calls in a row, different inputs
        host = seq_shards_qkv(P, b, s, hq, hkv, d, dtype, seed=seed)
        qs, ks, vs = ([t.cuda() for t in x] for x in host)
        out = [torch.full_like(q, float("nan")) for q in qs]
        assert _noalloc(lib, qs, ks, vs, out, causal) == 0
        ref = uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=False)
        torch.cuda.synchronize()
        assert uly.ulysses_device_status(clear=True) == 0
        want = oracle.dist_attn_fwd(*host, causal)
        for o, r, w in zip(out, ref, want):
            assert torch.equal(o.contiguous().view(torch.uint8), r.contiguous().view(torch.uint8))
            _close(o.cpu(), w, dtype)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = uly.load_library()
    # the DiT-sized forward needs 256 MiB of scratch, beyond the fixed 64 MiB
    P, b, s, hq, d = 4, 2, 4096, 32, 128
    need = uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hq, d, torch.bfloat16, False)
    assert need > uly.NOALLOC_SCRATCH_BYTES
    qs = [torch.zeros((b, s // P, hq, d), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    out = [torch.empty_like(q) for q in qs]
    assert _noalloc(lib, qs, qs, qs, out, True) == 1  # ULY_ERR_INVALID_ARG, nothing enqueued

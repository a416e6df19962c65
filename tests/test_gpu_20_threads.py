"""The C ABI keeps no state between calls (argument records live on each call's stack), so
calls from several host threads, each on its own CUDA stream, must give exactly the results
the same calls give one after another.  ctypes releases the interpreter lock during each
library call, so the calls really overlap on the host.  (The no-allocation entry point is
left out: its calls share one scratch array by design.)"""
import threading

import pytest
import torch

import sequence_attention_seq_gb300 as uly
from gpu_util import bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, seq_shards_qkv, shard_seq

pytestmark = pytest.mark.gpu

# P, b, s, hq, hkv, d, causal: unfused and fused forwards, the training path and the exchanges
CASES = [(4, 1, 512, 8, 4, 128, True), (2, 2, 384, 4, 2, 64, False), (8, 1, 1024, 8, 8, 128, True),
         (3, 1, 384, 6, 3, 64, True)]


def _work(case, seed):
    P, b, s, hq, hkv, d, causal = case
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=seed, device="cuda")
    dos = shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=seed + 1, device="cuda"), P)
    fused = (s // P) % 128 == 0
    return P, causal, fused, qs, ks, vs, dos


def _run(job, stream):
    P, causal, fused, qs, ks, vs, dos = job
    with torch.cuda.stream(stream):
        out = {"fwd": uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=False, stream=stream)}
        if fused:
            out["fwd_fused"] = uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=True, stream=stream)
        o, lse = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal, stream=stream)
        out["grads"] = uly.ulysses_dist_attn_bwd(qs, ks, vs, o, dos, lse, causal, stream=stream)
        out["heads"] = uly.ulysses_a2a_seq2head(qs, stream=stream)
    return out


def _flat(out):
    res = []
    for key in sorted(out):
        v = out[key]
        if key == "grads":
            for part in v:
                res.extend(part)
        else:
            res.extend(v)
    return res


def test_concurrent_calls_from_host_threads_give_the_sequential_bits():
    need_gpu()
    jobs = [_work(c, seed=10 * i + 1) for i, c in enumerate(CASES)]
    torch.cuda.synchronize()
    # one after another, on the default stream
    want = [_flat(_run(j, torch.cuda.current_stream())) for j in jobs]
    torch.cuda.synchronize()
    device_ok()
    # every job three times over, the jobs in parallel host threads with a stream each
    got = [None] * len(jobs)
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            res = None
            for _ in range(3):
                res = _run(jobs[i], stream)
            stream.synchronize()
            got[i] = _flat(res)
        except Exception as e:  # noqa: BLE001
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    torch.cuda.synchronize()
    device_ok()
    assert not errors, errors
    for i, (g, w) in enumerate(zip(got, want)):
        assert g is not None and len(g) == len(w), f"job {i}"
        for n, (a, c) in enumerate(zip(g, w)):
            assert bits_equal(a, c), f"job {i}, result {n}"

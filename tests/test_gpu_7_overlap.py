"""The overlapped forward (exchanges of one head group on a side stream while another head
group's attention runs): the same bits as the plain unfused forward, for every chunk count
that divides the K/V heads of a rank; argument errors."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu

CASES = [
    # P, b, s, hq, hkv, d, dtype, causal, n_chunks
    (2, 1, 64, 4, 4, 16, torch.float32, False, 2),     # fp32 path
    (4, 2, 512, 8, 8, 128, torch.bfloat16, False, 2),
    (2, 1, 384, 8, 4, 128, torch.bfloat16, True, 2),   # grouped K/V
    (2, 2, 320, 16, 8, 64, torch.bfloat16, True, 4),   # ragged tail, 4 chunks
    (2, 1, 200, 4, 4, 128, torch.bfloat16, True, 1),   # one chunk
    (4, 2, 4096, 32, 32, 128, torch.bfloat16, True, 8),
    (4, 2, 4096, 32, 32, 128, torch.bfloat16, False, 4),
    (2, 1, 512, 8, 2, 128, torch.bfloat16, True, 4),     # one K/V head per rank shared by 4 chunks
    (2, 1, 512, 8, 4, 64, torch.bfloat16, False, 4),     # two K/V heads per rank, 2 chunks each
    (8, 1, 32768, 32, 8, 128, torch.bfloat16, True, 4),  # the GQA workload
]


@pytest.mark.parametrize("P,b,s,hq,hkv,d,dt,causal,nc", CASES)
def test_overlap_matches_unfused(P, b, s, hq, hkv, d, dt, causal, nc):
    need_gpu()
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, dt, seed=s + nc)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    over = uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, causal, n_chunks=nc)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(over[j], plain[j]), f"rank {j}"
    if s <= 512:
        want = oracle.dist_attn_fwd(qs, ks, vs, causal)
        for j in range(P):
            assert_close(over[j], want[j], dt, f"rank {j}")


def test_overlap_same_stream_and_repeat():
    need_gpu()
    qs, ks, vs = seq_shards_qkv(2, 1, 768, 8, 8, 128, torch.bfloat16, seed=4)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=False)
    main = torch.cuda.current_stream()
    a = uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, True, n_chunks=4, side_stream=main)
    b = uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, True, n_chunks=2)
    torch.cuda.synchronize()
    device_ok()
    for j in range(2):
        assert bits_equal(a[j], plain[j]) and bits_equal(b[j], plain[j])


def test_overlap_argument_errors():
    need_gpu()
    qs, ks, vs = seq_shards_qkv(2, 1, 256, 8, 8, 128, torch.bfloat16, seed=1)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    for bad in (0, 3, 8, 65):  # 4 local query heads: 3 and 8 do not divide them
        with pytest.raises(uly.UlyssesError) as e:
            uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, True, n_chunks=bad,
                                              workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
        assert e.value.status == 1
    with pytest.raises(uly.UlyssesError) as e:
        uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, True, n_chunks=2,
                                          workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 1
    torch.cuda.synchronize()
    device_ok()

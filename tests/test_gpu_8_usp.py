"""The two-level (Ulysses x Ring) forward on the GPU: against the oracle's explicit ring with
online-softmax merges, and bit for bit against the plain Ulysses forward over the same ranks
(every query attends to the same key tiles in the same order)."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu

CASES = [
    # Pu, Pr, b, s, hq, hkv, d, causal
    (2, 2, 1, 512, 4, 2, 128, True),
    (2, 2, 2, 512, 4, 4, 64, False),
    (4, 2, 1, 1024, 8, 4, 128, True),
    (2, 4, 1, 1024, 4, 2, 128, True),
    (1, 4, 1, 512, 2, 1, 128, True),     # ring only
    (4, 1, 1, 512, 8, 8, 64, True),      # Ulysses only
    (2, 2, 1, 768, 2, 2, 128, False),
    (4, 2, 1, 1024, 8, 8, 128, True),    # P | h_kv: also bitwise against plain Ulysses
    (2, 2, 2, 512, 8, 4, 64, False),
    (4, 8, 1, 2048, 4, 4, 64, True),     # 32 ranks: the wide parameter block
]


@pytest.mark.parametrize("Pu,Pr,b,s,hq,hkv,d,causal", CASES)
def test_usp_against_oracle_and_ulysses(Pu, Pr, b, s, hq, hkv, d, causal):
    need_gpu()
    P = Pu * Pr
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=s + 10 * Pu + Pr)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    out = uly.ulysses_usp_attn_fwd(qd, kd, vd, causal, Pu, Pr)
    # plain Ulysses over all P ranks needs P | h_kv; the two-level split only Pu | h_kv
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False) if hkv % P == 0 else None
    torch.cuda.synchronize()
    device_ok()
    want = oracle.usp_fwd(qs, ks, vs, causal, Pu, Pr)
    for j in range(P):
        assert_close(out[j], want[j], torch.bfloat16, f"rank {j}")
        if plain is not None:
            assert bits_equal(out[j], plain[j]), f"rank {j}: differs from the plain Ulysses forward"


def test_usp_full_size_example_sampled():
    """The pages' 256K-token 4 x 2 example at full length (h=16, d=128, causal): sampled
    output rows against the oracle's per-row evaluation of the same attention."""
    need_gpu()
    Pu, Pr, b, s, h, d = 4, 2, 1, 262144, 16, 128
    P = Pu * Pr
    qs, ks, vs = seq_shards_qkv(P, b, s, h, h, d, torch.bfloat16, seed=5, device="cuda")
    out = uly.ulysses_usp_attn_fwd(qs, ks, vs, True, Pu, Pr)
    torch.cuda.synchronize()
    device_ok()
    S = s // P
    g = torch.Generator().manual_seed(1)
    samples = [(int(j), 0, int(t), int(hh)) for j, t, hh in zip(torch.randint(0, P, (12,), generator=g),
                                                               torch.randint(0, S, (12,), generator=g),
                                                               torch.randint(0, h, (12,), generator=g))]
    samples += [(P - 1, 0, S - 1, h - 1), (0, 0, 0, 0)]
    qc, kc, vc = [x.cpu() for x in qs], [x.cpu() for x in ks], [x.cpu() for x in vs]
    want = oracle.dist_attn_rows(qc, kc, vc, True, samples)
    got = torch.stack([out[j][bb, t, hh].cpu() for (j, bb, t, hh) in samples])
    assert_close(got, want, torch.bfloat16, "sampled rows")


def test_usp_argument_errors():
    need_gpu()
    qs, ks, vs = seq_shards_qkv(4, 1, 512, 4, 4, 128, torch.bfloat16, seed=2)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    with pytest.raises(ValueError):   # 4 ranks are not 3 x 2
        uly.ulysses_usp_attn_fwd(qd, kd, vd, True, 3, 2)
    with pytest.raises(uly.UlyssesError) as e:   # workspace too small
        uly.ulysses_usp_attn_fwd(qd, kd, vd, True, 4, 1, workspace=torch.empty(256, dtype=torch.uint8,
                                                                              device="cuda"))
    assert e.value.status == 1
    with pytest.raises(uly.UlyssesError) as e:   # segment of 128 tokens per ring group: 512/8 = 64 is not a tile
        qs8, ks8, vs8 = seq_shards_qkv(8, 1, 512, 8, 8, 128, torch.bfloat16, seed=2)
        uly.ulysses_usp_attn_fwd([t.cuda() for t in qs8], [t.cuda() for t in ks8], [t.cuda() for t in vs8],
                                 True, 1, 8, workspace=torch.empty(1 << 24, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 2
    torch.cuda.synchronize()
    device_ok()

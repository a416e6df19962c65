"""The fused backward over 32 rank buffers (four tensor maps per rank: the wide parameter
block) against the unfused backward, bit for bit, and sampled gradient rows against the
oracle's per-row evaluation ("02 · DeepSpeed-Ulysses", section 5: each exchange's backward
is the swapped exchange, the local backward the ordinary one)."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close_grad, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,b,s,h,d,causal", [(32, 1, 4096, 32, 64, True), (24, 1, 3072, 24, 128, False)])
def test_fused_backward_many_ranks(P, b, s, h, d, causal):
    need_gpu()
    q, k, v = global_qkv(b, s, h, h, d, torch.bfloat16, seed=P + 5)
    do = global_grad(b, s, h, d, torch.bfloat16, seed=P + 6)
    qd, kd, vd, dod = ([t.cuda() for t in shard_seq(x, P)] for x in (q, k, v, do))
    o, lse = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, causal, fused=True)
    g_f = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal, fused=True)
    g_u = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal, fused=False)
    torch.cuda.synchronize()
    device_ok()
    for name, gf, gu in zip(("dq", "dk", "dv"), g_f, g_u):
        for j in range(P):
            assert bits_equal(gf[j], gu[j]), f"{name}: fused != unfused on rank {j}"
    dq, dk, dv = (torch.cat([x.cpu() for x in g], 1) for g in g_f)  # global [b, s, h, d]
    for gh in (0, h - 1):
        hs = slice(gh, gh + 1)
        qsm = [(0, 0, 0), (0, s // 2 + 3, 0), (0, s - 1, 0)]
        ksm = [(0, 0, 0), (0, s // 3, 0), (0, s - 1, 0)]
        wq, wk, wv = oracle.attention_bwd_rows(q[:, :, hs].contiguous(), k[:, :, hs].contiguous(),
                                               v[:, :, hs].contiguous(), do[:, :, hs].contiguous(), causal, qsm, ksm)
        assert_close_grad(torch.stack([dq[0, i, gh] for (_, i, _) in qsm]), wq, f"dq rows, head {gh}")
        assert_close_grad(torch.stack([dk[0, j, gh] for (_, j, _) in ksm]), wk, f"dk rows, head {gh}")
        assert_close_grad(torch.stack([dv[0, j, gh] for (_, j, _) in ksm]), wv, f"dv rows, head {gh}")

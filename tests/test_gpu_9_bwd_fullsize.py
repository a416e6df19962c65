"""The backward at the DiT workload's full size (P=4, b=2, s=4096, h=32, d=128, bf16), in
the launch configuration the benchmark times (fused and unfused distributed backward):
sampled dQ rows and dK/dV key rows against the oracle's per-row evaluation, and two
identities of the exact gradient that hold at any size -- sum_j dK_j = 0 (each row of dS
sums to zero, because D_i = sum_j P_ij dP_ij) and sum_j dV_j = sum over the group's query
heads of sum_i dO_i (each row of P sums to one)."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close_grad, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu

P, B, S_TOT, H, HKV, D = 4, 2, 4096, 32, 32, 128


@pytest.fixture(scope="module")
def dit_backward():
    need_gpu()
    q, k, v = global_qkv(B, S_TOT, H, HKV, D, torch.bfloat16, seed=31)
    do = global_grad(B, S_TOT, H, D, torch.bfloat16, seed=32)
    qs, ks, vs, dos = (shard_seq(x, P) for x in (q, k, v, do))
    qd, kd, vd, dod = ([t.cuda() for t in xs] for xs in (qs, ks, vs, dos))
    o, lse = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, True, fused=True)
    g_f = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, True, fused=True)
    g_u = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, True, fused=False)
    torch.cuda.synchronize()
    device_ok()
    grads = tuple(torch.cat([x.cpu() for x in g], 1) for g in g_f)  # global [b, s, heads, d]
    same = all(bits_equal(x[j], y[j]) for gf, gu in zip(g_f, g_u) for x, y in [(gf, gu)] for j in range(P))
    return q, k, v, do, grads, same


def test_fullsize_fused_equals_unfused(dit_backward):
    assert dit_backward[5]


def test_fullsize_sampled_rows(dit_backward):
    q, k, v, do, (dq, dk, dv), _ = dit_backward
    Hq = H // P
    for r, hh in ((0, 0), (3, Hq - 1)):  # two (head rank, local head) pairs
        sl = slice(r * Hq, (r + 1) * Hq)
        gh = r * Hq + hh
        qsm = [(0, 0, hh), (1, 1777, hh), (0, S_TOT - 1, hh)]
        ksm = [(1, 0, hh), (0, 2049, hh)]
        wq, wk, wv = oracle.attention_bwd_rows(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                                               v[:, :, sl].contiguous(), do[:, :, sl].contiguous(), True, qsm, ksm)
        got_q = torch.stack([dq[bb, i, gh] for (bb, i, _) in qsm])
        got_k = torch.stack([dk[bb, j, gh] for (bb, j, _) in ksm])
        got_v = torch.stack([dv[bb, j, gh] for (bb, j, _) in ksm])
        assert_close_grad(got_q, wq, f"dq rows, head {gh}")
        assert_close_grad(got_k, wk, f"dk rows, head {gh}")
        assert_close_grad(got_v, wv, f"dv rows, head {gh}")


def test_fullsize_gradient_identities(dit_backward):
    _, _, _, do, (dq, dk, dv), _ = dit_backward
    dk64, dv64, do64 = dk.double(), dv.double(), do.double()
    # sum over keys of dK is zero up to the bf16 rounding of each row
    s_k = dk64.sum(1)
    assert (s_k.abs() <= 2.0 ** -7 * dk64.abs().sum(1) + 1e-3).all()
    # sum over keys of dV equals the sum over queries of dO (MHA: the same head)
    s_v, s_o = dv64.sum(1), do64.sum(1)
    assert ((s_v - s_o).abs() <= 2.0 ** -7 * dv64.abs().sum(1) + 1e-2).all()
    assert torch.isfinite(dq.double()).all()

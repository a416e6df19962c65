"""The Python binding's argument checks (no GPU needed).  The C ABI receives only sizes and
pointers, so every per-rank list must hold exactly P tensors of the size the sizes imply;
a short list or a wrong-sized output would otherwise make a kernel read or write outside
a buffer.  Stand-in objects with the tensor attributes the checks read (shape, dtype,
device, contiguity) show that each entry point raises ValueError before it calls the
library."""
import pytest
import torch

import sequence_attention_seq_gb300 as uly


class Fake:
    """Looks like a contiguous CUDA tensor to the binding's checks; never dereferenced."""

    def __init__(self, shape, dtype=torch.bfloat16, dev=0, cuda=True, contiguous=True):
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.is_cuda = cuda
        self._dev = dev
        self._contig = contiguous

    def get_device(self):
        return self._dev

    def is_contiguous(self):
        return self._contig

    def dim(self):
        return len(self.shape)

    def data_ptr(self):
        raise AssertionError("the binding reached the library")

    def numel(self):
        n = 1
        for x in self.shape:
            n *= x
        return n

    def element_size(self):
        return 2


P, b, s, hq, hkv, d = 4, 1, 512, 8, 4, 64
S = s // P


def seq(h=hq, n=P, **kw):
    return [Fake((b, S, h, d), **kw) for _ in range(n)]


def head(h=hq // P, n=P, **kw):
    return [Fake((b, s, h, d), **kw) for _ in range(n)]


def lse(n=P, rows=hq // P, dtype=torch.float32):
    return [Fake((b, rows, s), dtype=dtype) for _ in range(n)]


def test_helper_checks_count_shape_dtype_device():
    q = seq()
    assert uly._same(q, "q") is q[0]
    with pytest.raises(ValueError, match="3 tensors given for 4 ranks"):
        uly._same(q[:3], "q", P)
    with pytest.raises(ValueError, match="no tensors"):
        uly._same([], "q")
    with pytest.raises(ValueError):
        uly._same(q[:3] + [Fake((b, S, hq, d + 1))], "q")
    with pytest.raises(ValueError):
        uly._same(q[:3] + [Fake((b, S, hq, d), dtype=torch.float32)], "q")
    with pytest.raises(ValueError):
        uly._same(q[:3] + [Fake((b, S, hq, d), dev=1)], "q")
    with pytest.raises(ValueError):
        uly._same(q[:3] + [Fake((b, S, hq, d), contiguous=False)], "q")
    with pytest.raises(ValueError, match="CUDA"):
        uly._same([Fake((b, S, hq, d), cuda=False)], "q")
    # dtype and device taken from a reference tensor, dtype overridable
    with pytest.raises(ValueError):
        uly._same(lse(), "lse", P, (b, hq // P, s), q[0])  # bf16 expected from q
    uly._same(lse(), "lse", P, (b, hq // P, s), q[0], torch.float32)


def test_exchanges_reject_bad_outputs():
    with pytest.raises(ValueError):
        uly.ulysses_a2a_seq2head(seq(), head()[:3])
    with pytest.raises(ValueError):
        uly.ulysses_a2a_seq2head(seq(), head(h=hq // P + 1))
    with pytest.raises(ValueError):
        uly.ulysses_a2a_head2seq(head(), seq(h=hq - 1))
    with pytest.raises(ValueError):
        uly.ulysses_a2a_pack(seq()[0], 0, P, out=Fake((P, b, S, hq // P, d + 8)))
    with pytest.raises(ValueError):
        uly.ulysses_a2a_unpack(Fake((P, b, S, hq // P, d)), 0, out=Fake((b, s, hq // P, d), dtype=torch.float32))


def test_forwards_reject_mismatched_ranks_and_outputs():
    q, k, v = seq(), seq(h=hkv), seq(h=hkv)
    with pytest.raises(ValueError, match="3 tensors given for 4 ranks"):
        uly.ulysses_dist_attn_fwd(q, k[:3], v, True)
    with pytest.raises(ValueError):
        uly.ulysses_dist_attn_fwd(q, k, seq(h=hkv + 1), True)
    with pytest.raises(ValueError):
        uly.ulysses_dist_attn_fwd(q, k, v, True, out_seq=seq()[:2])
    with pytest.raises(ValueError):
        uly.ulysses_dist_attn_fwd_lse(q, k, v, True, out_seq=seq(), lse=lse(rows=hq))
    with pytest.raises(ValueError):
        uly.ulysses_dist_attn_fwd_noalloc(q, k, v, True, seq(h=hq * 2))
    with pytest.raises(ValueError):
        uly.ulysses_dist_attn_fwd_overlap(q, k, v, True, out_seq=seq(n=P + 1))
    with pytest.raises(ValueError):
        uly.ulysses_local_attention(head(), head(h=1)[:1], head(h=1), True)
    with pytest.raises(ValueError):
        uly.ulysses_local_attention_fwd_lse(head(), head(h=1), head(h=1), True, out_head=head(), lse=lse(n=2))
    with pytest.raises(ValueError):
        uly.ulysses_usp_attn_fwd(seq(n=8), seq(h=hkv, n=8), seq(h=hkv, n=8), True, 4, 2, out_seq=seq(n=4))
    with pytest.raises(ValueError):
        uly.ulysses_usp_attn_fwd_lse(seq(n=8), seq(h=hkv, n=8), seq(h=hkv, n=8), True, 4, 2, out_seq=seq(n=8),
                                     lse=lse(n=8))


def test_backwards_reject_mismatched_tensors():
    q, k, v = seq(), seq(h=hkv), seq(h=hkv)
    o, do = seq(), seq()
    with pytest.raises(ValueError):  # dO of another shape
        uly.ulysses_dist_attn_bwd(q, k, v, o, seq(h=hq + 4), lse(), True)
    with pytest.raises(ValueError):  # statistics of the head layout's shape expected
        uly.ulysses_dist_attn_bwd(q, k, v, o, do, lse(rows=hq), True)
    with pytest.raises(ValueError):  # dK shaped like Q
        uly.ulysses_dist_attn_bwd(q, k, v, o, do, lse(), True, grads=(seq(), seq(), seq(h=hkv)))
    with pytest.raises(ValueError):  # too few dV tensors
        uly.ulysses_dist_attn_bwd(q, k, v, o, do, lse(), True, grads=(seq(), seq(h=hkv), seq(h=hkv, n=3)))
    with pytest.raises(ValueError):  # workspace on the host
        uly.ulysses_local_attention_bwd(head(), head(h=1), head(h=1), head(), head(), lse(), True,
                                        grads=(head(), head(h=1), head(h=1)),
                                        workspace=Fake((1 << 20,), dtype=torch.uint8, cuda=False))
    with pytest.raises(ValueError):
        uly.ulysses_usp_attn_bwd(seq(n=8), seq(h=hkv, n=8), seq(h=hkv, n=8), seq(n=8), seq(n=8), lse(n=2), True, 4, 2)


def test_valid_arguments_pass_the_checks():
    """Correct shapes (grouped K/V heads and the two-level layout included) get through every
    check and reach the library call, where the stand-ins refuse to give a pointer."""
    q, k, v = seq(), seq(h=hkv), seq(h=hkv)
    ws = Fake((1 << 20,), dtype=torch.uint8)
    blocks = Fake((P, b, S, hq // P, d))
    q8, k8, v8 = seq(n=8), seq(h=hkv, n=8), seq(h=hkv, n=8)
    lse8 = [Fake((b, hq // 4, 8 * S), dtype=torch.float32) for _ in range(4)]
    calls = [
        lambda: uly.ulysses_a2a_seq2head(seq(), head()),
        lambda: uly.ulysses_a2a_head2seq(head(), seq()),
        lambda: uly.ulysses_a2a_pack(seq()[0], 0, P, out=blocks),
        lambda: uly.ulysses_a2a_pack(head()[0], 1, P, out=blocks),
        lambda: uly.ulysses_a2a_unpack(blocks, 0, out=Fake((b, s, hq // P, d))),
        lambda: uly.ulysses_a2a_unpack(blocks, 1, out=Fake((b, S, hq, d))),
        lambda: uly.ulysses_local_attention(head(), head(h=1), head(h=1), True, out_head=head()),
        lambda: uly.ulysses_local_attention_fwd_lse(head(), head(h=1), head(h=1), True, out_head=head(), lse=lse()),
        lambda: uly.ulysses_dist_attn_fwd(q, k, v, True, out_seq=seq(), workspace=ws),
        lambda: uly.ulysses_dist_attn_fwd_lse(q, k, v, True, out_seq=seq(), lse=lse(), workspace=ws),
        lambda: uly.ulysses_dist_attn_fwd_noalloc(q, k, v, True, seq()),
        lambda: uly.ulysses_dist_attn_fwd_overlap(q, k, v, True, out_seq=seq(), workspace=ws, side_stream=object()),
        lambda: uly.ulysses_dist_attn_bwd(q, k, v, seq(), seq(), lse(), True, grads=(seq(), seq(h=hkv), seq(h=hkv)),
                                          workspace=ws),
        lambda: uly.ulysses_local_attention_bwd(head(), head(h=1), head(h=1), head(), head(), lse(), True,
                                                grads=(head(), head(h=1), head(h=1)), workspace=ws),
        lambda: uly.ulysses_usp_attn_fwd(q8, k8, v8, True, 4, 2, out_seq=seq(n=8), workspace=ws),
        lambda: uly.ulysses_usp_attn_fwd_lse(q8, k8, v8, True, 4, 2, out_seq=seq(n=8), lse=lse8, workspace=ws),
        lambda: uly.ulysses_usp_attn_bwd(q8, k8, v8, seq(n=8), seq(n=8), lse8, True, 4, 2,
                                         grads=(seq(n=8), seq(h=hkv, n=8), seq(h=hkv, n=8)), workspace=ws),
    ]
    for call in calls:
        with pytest.raises(AssertionError, match="reached the library"):
            call()

"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every function
include/ulysses.h declares, and rejects bad arguments before it touches the device."""
import ctypes
import os
import re

import pytest

import sequence_attention_seq_gb300 as uly
from sequence_attention_seq_gb300 import build as uly_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ulysses.h")

INVALID, UNSUPPORTED = 1, 2
FP32, BF16 = 0, 1


@pytest.fixture(scope="module")
def lib():
    uly_build.build()
    return uly.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ulysses_\w+)\s*\(", text)))


def test_header_declares_and_library_exports(lib):
    names = _declared()
    assert sorted(uly.EXPORTED_SYMBOLS) == names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def _arr(*vals):
    a = (ctypes.c_void_p * len(vals))()
    for i, v in enumerate(vals):
        a[i] = v
    return a


# fake, never dereferenced device addresses: validation fails before any CUDA call
A, B, C, D = 0x10000000, 0x20000000, 0x30000000, 0x40000000


def test_exchange_argument_errors(lib):
    f = lib.ulysses_a2a_seq2head
    ok_in, ok_out = _arr(A, B), _arr(C, D)
    assert f(0, 1, 64, 4, 16, FP32, ok_in, ok_out, None) == INVALID           # P < 1
    assert f(65, 1, 65 * 2, 65, 16, FP32, ok_in, ok_out, None) == INVALID     # P > 64
    assert f(2, 1, 63, 4, 16, FP32, ok_in, ok_out, None) == INVALID           # s % P
    assert f(2, 1, 64, 3, 16, FP32, ok_in, ok_out, None) == INVALID           # h % P
    assert f(2, 1, 64, 4, 16, 7, ok_in, ok_out, None) == INVALID              # dtype
    assert f(2, 1, 64, 4, 16, FP32, _arr(A, 0), ok_out, None) == INVALID      # null
    assert f(2, 1, 64, 4, 16, FP32, _arr(A, B + 4), ok_out, None) == INVALID  # misaligned
    assert f(2, 1, 64, 4, 16, FP32, ok_in, _arr(C, A + 64), None) == INVALID  # out overlaps in
    assert f(2, 1, 64, 4, 16, FP32, ok_in, _arr(C, C + 64), None) == INVALID  # outputs overlap
    g = lib.ulysses_a2a_head2seq
    assert g(2, 1, 64, 4, 16, FP32, ok_in, _arr(C, A), None) == INVALID


def test_attention_argument_errors(lib):
    f = lib.ulysses_local_attention
    q, k, v, o = _arr(A), _arr(B), _arr(C), _arr(D)
    assert f(1, 1, 64, 4, 3, 16, FP32, 0, q, k, v, o, None) == INVALID        # h_q % h_kv
    four = (_arr(A, A + 0x1000000, A + 0x2000000, A + 0x3000000), _arr(B, B + 0x1000000, B + 0x2000000, B + 0x3000000),
            _arr(C, C + 0x1000000, C + 0x2000000, C + 0x3000000), _arr(D, D + 0x1000000, D + 0x2000000, D + 0x3000000))
    # K/V heads and ranks must be multiples of one another (split or replicated): 6 and 4 are not
    assert f(4, 1, 64, 12, 6, 16, FP32, 0, *four, None) == INVALID
    assert f(1, 1, 64, 4, 4, 96, BF16, 0, q, k, v, o, None) == UNSUPPORTED    # bf16 needs d in {64,128}
    assert f(1, 1, 64, 4, 4, 6, FP32, 0, q, k, v, o, None) == UNSUPPORTED     # fp32 needs d % 4 == 0
    assert f(1, 1, 64, 4, 4, 260, FP32, 0, q, k, v, o, None) == UNSUPPORTED   # fp32 needs d <= 256
    assert f(1, 1, 64, 4, 4, 16, FP32, 0, q, k, v, _arr(A + 256), None) == INVALID  # o overlaps q


def test_dist_attn_errors_and_workspace(lib):
    ws = lib.ulysses_dist_attn_workspace_bytes
    e = 2
    P, b, s, hq, hkv, d = 4, 2, 4096, 32, 8, 128
    qh = b * s * (hq // P) * d * e
    kh = b * s * (hkv // P) * d * e
    assert ws(P, b, s, hq, hkv, d, BF16, 0) == P * (2 * qh + 2 * kh)
    assert ws(P, b, s, hq, hkv, d, BF16, 1) == 0
    assert ws(3, b, s, hq, hkv, d, BF16, 0) == 0  # invalid: h_q % P
    f = lib.ulysses_dist_attn_fwd
    qs = _arr(*[A + i * 0x1000000 for i in range(4)])
    ks = _arr(*[B + i * 0x1000000 for i in range(4)])
    vs = _arr(*[C + i * 0x1000000 for i in range(4)])
    os_ = _arr(*[D + i * 0x1000000 for i in range(4)])
    need = ws(P, b, s, hq, hkv, d, BF16, 0)
    wsp = 0x100000000
    assert f(P, b, s, hq, hkv, d, BF16, 0, qs, ks, vs, os_, None, need, 0, None) == INVALID   # no workspace
    assert f(P, b, s, hq, hkv, d, BF16, 0, qs, ks, vs, os_, wsp, need - 1, 0, None) == INVALID  # too small
    assert f(P, b, s, hq, hkv, d, BF16, 0, qs, ks, vs, os_, wsp + 16, need, 0, None) == INVALID  # 256-B align
    assert f(P, b, 4 * 96, hq, hkv, d, BF16, 1, qs, ks, vs, os_, None, 0, 1, None) == UNSUPPORTED  # (s/P)%128
    assert f(P, b, s, hq, hkv, 64, FP32, 1, qs, ks, vs, os_, None, 0, 1, None) == UNSUPPORTED     # fused fp32
    assert f(P, b, s, hq, hkv, 96, BF16, 1, qs, ks, vs, os_, None, 0, 1, None) == UNSUPPORTED     # d


def test_status_strings(lib):
    for code, name in enumerate(["ULY_OK", "ULY_ERR_INVALID_ARG", "ULY_ERR_UNSUPPORTED", "ULY_ERR_CUDA",
                                 "ULY_ERR_TIMEOUT"]):
        assert uly.ulysses_status_string(code) == name


def test_replicated_kv_workspace(lib):
    """Fewer K/V heads than ranks (h_kv | P): each rank holds one K/V head in head layout."""
    ws = lib.ulysses_dist_attn_workspace_bytes
    P, b, s, hq, d = 4, 1, 512, 8, 128
    r = lambda x: (x + 255) // 256 * 256
    qb, kb = r(b * s * (hq // P) * d * 2), r(b * s * 1 * d * 2)
    for hkv in (1, 2):
        assert ws(P, b, s, hq, hkv, d, BF16, 0) == P * (2 * qb + 2 * kb)
        assert ws(P, b, s, hq, hkv, d, BF16, 1) == 0          # fused: no workspace
    assert ws(P, b, s, 12, 6, d, BF16, 0) == 0               # 6 and 4: neither divides the other


def test_replicated_kv_overlap_workspace(lib):
    """The overlapped forward with fewer K/V heads than ranks: all chunks share each rank's
    one K/V head, so the workspace holds one K/V group next to every chunk's Q and O."""
    ws = lib.ulysses_dist_attn_overlap_workspace_bytes
    P, b, s, hq, d = 4, 1, 512, 8, 128
    r = lambda x: (x + 255) // 256 * 256
    for hkv in (1, 2):
        for nc in (1, 2):
            qb, kb = r(b * s * (hq // P // nc) * d * 2), r(b * s * 1 * d * 2)
            assert ws(P, b, s, hq, hkv, d, BF16, nc) == P * (2 * qb * nc + 2 * kb)
    assert ws(P, b, s, hq, 1, d, BF16, 4) == 0   # 2 query heads per rank do not split into 4 chunks
    assert ws(P, b, s, 12, 6, d, BF16, 1) == 0   # 6 and 4: neither divides the other


def test_replicated_kv_two_level_workspace(lib):
    """The two-level layout with fewer K/V heads than Ulysses ranks: one K/V head per rank of
    a group; the backward keeps fp32 dK/dV shares (twice the bf16 size) until they are summed."""
    fw, bw = lib.ulysses_usp_workspace_bytes, lib.ulysses_usp_bwd_workspace_bytes
    Pu, Pr, b, s, hq, d = 4, 2, 1, 1024, 8, 128
    r = lambda x: (x + 255) // 256 * 256
    L = s // Pr
    qb, kb = r(b * L * (hq // Pu) * d * 2), r(b * L * 1 * d * 2)
    ra = r(b * (hq // Pu) * ((s + 127) // 128 * 128) * 4)
    for hkv in (1, 2):
        assert fw(Pu, Pr, b, s, hq, hkv, d, BF16) == Pu * Pr * (2 * qb + 2 * kb)
        assert bw(Pu, Pr, b, s, hq, hkv, d, BF16) == Pu * Pr * (4 * qb + kb + 4 * kb) + Pu * 2 * ra
    assert fw(Pu, Pr, b, s, 12, 3, d, BF16) == 0   # 3 and 4: neither divides the other


def test_two_level_kv_head_rule(lib):
    """The two-level forward checks the K/V-head rule with the Ulysses degree Pu in place of P,
    before anything is enqueued: 3 K/V heads and Pu = 4 divide neither way."""
    f = lib.ulysses_usp_attn_fwd
    arr = lambda base: _arr(*[base + i * 0x1000000 for i in range(4)])
    q, k, v, o = arr(A), arr(B), arr(C), arr(D)
    assert f(4, 1, 1, 512, 12, 3, 128, BF16, 1, q, k, v, o, None, 0, None) == INVALID
    assert f(4, 1, 1, 512, 12, 5, 128, BF16, 1, q, k, v, o, None, 0, None) == INVALID   # h_q % h_kv
    assert f(4, 1, 1, 512, 6, 2, 128, BF16, 1, q, k, v, o, None, 0, None) == INVALID    # h_q % Pu


def test_pack_unpack_argument_errors(lib):
    # validation fails before any CUDA call: fake, never dereferenced addresses
    for f in (lib.ulysses_a2a_pack, lib.ulysses_a2a_unpack):
        assert f(2, 2, 1, 64, 4, 16, FP32, A, B, None) == INVALID       # direction not 0 or 1
        assert f(0, 2, 1, 63, 4, 16, FP32, A, B, None) == INVALID       # s % P
        assert f(1, 2, 1, 64, 3, 16, FP32, A, B, None) == INVALID       # h % P
        assert f(0, 2, 1, 64, 4, 16, FP32, 0, B, None) == INVALID       # null
        assert f(0, 2, 1, 64, 4, 16, FP32, A + 4, B, None) == INVALID   # misaligned
        assert f(0, 2, 1, 64, 4, 16, FP32, A, A + 1024, None) == INVALID  # out overlaps in (4 KB each side)
        assert f(0, 65, 1, 65, 65, 16, FP32, A, B, None) == INVALID     # P > 64
    # unpack(0) writes one piece of s*H*d elements: 2^26 tokens x 1 head x 256 fp32 is 2^32
    # 16-byte vectors, past the copy kernel's 32-bit index (the per-rank exchange checks pass)
    far_in, far_out = 1 << 48, 1 << 49  # 64 GiB each side: far apart so that they do not overlap
    assert lib.ulysses_a2a_unpack(0, 64, 1, 1 << 26, 64, 256, FP32, far_in, far_out, None) == INVALID


def _far(kind, n):
    """n fake, never dereferenced device addresses of one tensor kind, far from other kinds."""
    return _arr(*[(kind << 40) + (r << 32) for r in range(n)])


def test_empty_and_negative_sizes(lib):
    """Every entry point rejects a zero or negative size (P, b, s, heads, d) before it touches
    a pointer or the device; the workspace queries return 0 for them.  Each call below
    differs from a valid configuration (P=4 or Pu=Pr=2, b=1, s=512, h_q=8, h_kv=4, d=64,
    bf16) in one size only.  Only rejected calls are made: the addresses are fake."""
    q, k, v, o, do, dq, dk, dv, lse = (_far(i + 1, 4) for i in range(9))
    ws, wsn = 1 << 48, 1 << 40
    base = [4, 1, 512, 8, 4, 64]          # P, b, s, h_q, h_kv, d
    calls = {
        "ulysses_local_attention": lambda a: lib.ulysses_local_attention(*a, BF16, 0, q, k, v, o, None),
        "ulysses_dist_attn_fwd": lambda a: lib.ulysses_dist_attn_fwd(*a, BF16, 0, q, k, v, o, ws, wsn, 0, None),
        "ulysses_dist_attn_fwd_noalloc": lambda a: lib.ulysses_dist_attn_fwd_noalloc(*a, BF16, 0, q, k, v, o, None),
        "ulysses_local_attention_fwd_lse": lambda a: lib.ulysses_local_attention_fwd_lse(*a, BF16, 0, q, k, v, o, lse,
                                                                                         None),
        "ulysses_dist_attn_fwd_lse": lambda a: lib.ulysses_dist_attn_fwd_lse(*a, BF16, 0, q, k, v, o, lse, ws, wsn, 1,
                                                                             None),
        "ulysses_local_attention_bwd": lambda a: lib.ulysses_local_attention_bwd(*a, BF16, 0, q, k, v, o, do, lse, dq,
                                                                                 dk, dv, ws, wsn, None),
        "ulysses_dist_attn_bwd": lambda a: lib.ulysses_dist_attn_bwd(*a, BF16, 0, q, k, v, o, do, lse, dq, dk, dv, ws,
                                                                     wsn, 1, None),
        "ulysses_dist_attn_fwd_overlap": lambda a: lib.ulysses_dist_attn_fwd_overlap(*a, BF16, 0, q, k, v, o, ws, wsn,
                                                                                     2, None, None),
    }
    sizes = {
        "ulysses_dist_attn_workspace_bytes": lambda a: lib.ulysses_dist_attn_workspace_bytes(*a, BF16, 0),
        "ulysses_attn_bwd_workspace_bytes": lambda a: lib.ulysses_attn_bwd_workspace_bytes(*a, BF16, 1, 0),
        "ulysses_dist_attn_overlap_workspace_bytes":
            lambda a: lib.ulysses_dist_attn_overlap_workspace_bytes(*a, BF16, 2),
    }
    for i in range(len(base)):
        for bad in (0, -1):
            a = list(base)
            a[i] = bad
            for name, f in calls.items():
                assert f(a) == INVALID, f"{name} with size {i} = {bad}"
            for name, f in sizes.items():
                assert f(a) == 0, f"{name} with size {i} = {bad}"
    # the exchanges and their per-process halves: P, b, s, h, d
    ex = [2, 1, 64, 4, 16]
    for i in range(len(ex)):
        for bad in (0, -1):
            a = list(ex)
            a[i] = bad
            for f in (lib.ulysses_a2a_seq2head, lib.ulysses_a2a_head2seq):
                assert f(*a, FP32, q, o, None) == INVALID, f"exchange with size {i} = {bad}"
            for f in (lib.ulysses_a2a_pack, lib.ulysses_a2a_unpack):
                assert f(0, *a, FP32, A, B, None) == INVALID, f"pack/unpack with size {i} = {bad}"
    # the two-level calls: Pu, Pr, b, s, h_q, h_kv, d
    two = [2, 2, 1, 512, 8, 4, 64]
    for i in range(len(two)):
        for bad in (0, -1):
            a = list(two)
            a[i] = bad
            assert lib.ulysses_usp_workspace_bytes(*a, BF16) == 0
            assert lib.ulysses_usp_bwd_workspace_bytes(*a, BF16) == 0
            assert lib.ulysses_usp_attn_fwd(*a, BF16, 0, q, k, v, o, ws, wsn, None) == INVALID
            assert lib.ulysses_usp_attn_fwd_lse(*a, BF16, 0, q, k, v, o, lse, ws, wsn, None) == INVALID
            assert lib.ulysses_usp_attn_bwd(*a, BF16, 0, q, k, v, o, do, lse, dq, dk, dv, ws, wsn, None) == INVALID

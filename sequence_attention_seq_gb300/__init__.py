"""GB300 (sm_103a) Ulysses DistributedAttention forward: Python binding of the C ABI.

The binding only marshals arguments: it reads shapes from the tensors, allocates outputs
and workspace with PyTorch, and calls the functions of ``libulysses_gb300.so`` (declared
in ``include/ulysses.h``) on the current CUDA stream.  Every step of the computation runs
in the library's kernels; there is no fallback.  If the library is missing or cannot be
loaded, every call raises.

Layouts (per rank, row-major): seq layout ``[b, s/P, h, d]``, head layout
``[b, s, h/P, d]``.  A list of P tensors stands for the P sequence-parallel ranks.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "UlyssesError", "library_path", "load_library",
    "ulysses_a2a_seq2head", "ulysses_a2a_head2seq", "ulysses_local_attention",
    "ulysses_dist_attn_workspace_bytes", "ulysses_dist_attn_fwd", "ulysses_device_status",
    "ulysses_status_string", "EXPORTED_SYMBOLS", "ulysses_dist_attn_fwd_noalloc", "NOALLOC_SCRATCH_BYTES",
    "ulysses_local_attention_fwd_lse", "ulysses_dist_attn_fwd_lse", "ulysses_attn_bwd_workspace_bytes",
    "ulysses_local_attention_bwd", "ulysses_dist_attn_bwd", "ulysses_dist_attn_overlap_workspace_bytes",
    "ulysses_dist_attn_fwd_overlap", "ulysses_usp_workspace_bytes", "ulysses_usp_attn_fwd",
    "ulysses_usp_attn_fwd_lse", "ulysses_usp_bwd_workspace_bytes", "ulysses_usp_attn_bwd",
    "ulysses_wait_selftest", "ulysses_a2a_pack", "ulysses_a2a_unpack",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libulysses_gb300.so"

ULY_OK, ULY_ERR_INVALID_ARG, ULY_ERR_UNSUPPORTED, ULY_ERR_CUDA, ULY_ERR_TIMEOUT = range(5)
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}

# every function include/ulysses.h declares
EXPORTED_SYMBOLS = (
    "ulysses_a2a_seq2head", "ulysses_a2a_head2seq", "ulysses_local_attention",
    "ulysses_dist_attn_workspace_bytes", "ulysses_dist_attn_fwd", "ulysses_device_status",
    "ulysses_status_string", "ulysses_dist_attn_fwd_noalloc", "ulysses_local_attention_fwd_lse",
    "ulysses_dist_attn_fwd_lse", "ulysses_attn_bwd_workspace_bytes", "ulysses_local_attention_bwd",
    "ulysses_dist_attn_bwd", "ulysses_dist_attn_overlap_workspace_bytes", "ulysses_dist_attn_fwd_overlap",
    "ulysses_usp_workspace_bytes", "ulysses_usp_attn_fwd", "ulysses_usp_attn_fwd_lse",
    "ulysses_usp_bwd_workspace_bytes", "ulysses_usp_attn_bwd", "ulysses_wait_selftest",
    "ulysses_a2a_pack", "ulysses_a2a_unpack",
)

_lock = threading.Lock()
_lib = None


class UlyssesError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {_status_name(status)}")


def library_path():
    return os.path.join(_PKG, _LIB_NAME)


def load_library():
    """Load the C-ABI library (built by ``build.py``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{_LIB_NAME} is not built (run sequence_attention_seq_gb300/build.py); "
                               "this package has no CPU fallback")
        lib = ctypes.CDLL(path)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        pp = ctypes.POINTER(ctypes.c_void_p)
        for name in ("ulysses_a2a_seq2head", "ulysses_a2a_head2seq"):
            f = getattr(lib, name)
            f.argtypes = [i, i, i, i, i, i, pp, pp, vp]
            f.restype = i
        lib.ulysses_local_attention.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, vp]
        lib.ulysses_local_attention.restype = i
        lib.ulysses_dist_attn_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.ulysses_dist_attn_workspace_bytes.restype = sz
        lib.ulysses_dist_attn_fwd.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, vp, sz, i, vp]
        lib.ulysses_dist_attn_fwd.restype = i
        lib.ulysses_dist_attn_fwd_noalloc.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, vp]
        lib.ulysses_dist_attn_fwd_noalloc.restype = i
        lib.ulysses_local_attention_fwd_lse.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, pp, vp]
        lib.ulysses_local_attention_fwd_lse.restype = i
        lib.ulysses_dist_attn_fwd_lse.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, pp, vp, sz, i, vp]
        lib.ulysses_dist_attn_fwd_lse.restype = i
        lib.ulysses_attn_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i]
        lib.ulysses_attn_bwd_workspace_bytes.restype = sz
        lib.ulysses_local_attention_bwd.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, pp, pp, pp, pp, pp, vp,
                                                    sz, vp]
        lib.ulysses_local_attention_bwd.restype = i
        lib.ulysses_dist_attn_bwd.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, pp, pp, pp, pp, pp, vp, sz, i,
                                              vp]
        lib.ulysses_dist_attn_bwd.restype = i
        lib.ulysses_dist_attn_overlap_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.ulysses_dist_attn_overlap_workspace_bytes.restype = sz
        lib.ulysses_dist_attn_fwd_overlap.argtypes = [i, i, i, i, i, i, i, i, pp, pp, pp, pp, vp, sz, i, vp, vp]
        lib.ulysses_dist_attn_fwd_overlap.restype = i
        lib.ulysses_usp_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.ulysses_usp_workspace_bytes.restype = sz
        lib.ulysses_usp_attn_fwd.argtypes = [i, i, i, i, i, i, i, i, i, pp, pp, pp, pp, vp, sz, vp]
        lib.ulysses_usp_attn_fwd.restype = i
        lib.ulysses_usp_attn_fwd_lse.argtypes = [i, i, i, i, i, i, i, i, i, pp, pp, pp, pp, pp, vp, sz, vp]
        lib.ulysses_usp_attn_fwd_lse.restype = i
        lib.ulysses_usp_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.ulysses_usp_bwd_workspace_bytes.restype = sz
        lib.ulysses_usp_attn_bwd.argtypes = [i, i, i, i, i, i, i, i, i, pp, pp, pp, pp, pp, pp, pp, pp, pp, vp, sz,
                                             vp]
        lib.ulysses_usp_attn_bwd.restype = i
        for name in ("ulysses_a2a_pack", "ulysses_a2a_unpack"):
            f = getattr(lib, name)
            f.argtypes = [i, i, i, i, i, i, i, vp, vp, vp]
            f.restype = i
        lib.ulysses_wait_selftest.argtypes = [ctypes.c_ulonglong, vp]
        lib.ulysses_wait_selftest.restype = i
        lib.ulysses_device_status.argtypes = [i]
        lib.ulysses_device_status.restype = i
        lib.ulysses_status_string.argtypes = [i]
        lib.ulysses_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _status_name(status):
    try:
        return load_library().ulysses_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - naming an error must not raise another
        return f"status {status}"


def ulysses_status_string(status):
    return load_library().ulysses_status_string(int(status)).decode()


def _check(status, what):
    if status != ULY_OK:
        raise UlyssesError(status, what)


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))()
    for n, t in enumerate(tensors):
        arr[n] = t.data_ptr()
    return arr


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def _same(tensors, what, n=None, shape=None, like=None, dtype=None):
    """Checks a per-rank list of tensors and returns its first: n tensors (when n is given),
    each contiguous, on one CUDA device, of one shape and dtype.  The shape is `shape` when
    given, else the first tensor's; dtype and device are `like`'s when given (dtype may be
    overridden), else the first tensor's.  The library only sees pointers and sizes, so a
    list that is too short or a tensor of the wrong size must be stopped here."""
    if n is not None and len(tensors) != n:
        raise ValueError(f"{what}: {len(tensors)} tensors given for {n} ranks")
    if len(tensors) == 0:
        raise ValueError(f"{what}: no tensors given")
    t0 = tensors[0]
    if not t0.is_cuda:
        raise ValueError(f"{what}: tensors must live on a CUDA device")
    # one pass of cheap attribute reads: with 64 ranks a call checks several hundred tensors
    ref = t0 if like is None else like
    want_shape = t0.shape if shape is None else torch.Size(shape)
    want_dtype = ref.dtype if dtype is None else dtype
    dev = ref.get_device()
    for t in tensors:
        if t.shape != want_shape or t.dtype is not want_dtype or t.get_device() != dev or not t.is_cuda \
                or not t.is_contiguous():
            raise ValueError(f"{what}: every rank needs a contiguous {want_dtype} tensor of shape "
                             f"{tuple(want_shape)} on cuda:{dev}")
    return t0


def _workspace(workspace, like, what="workspace"):
    """(pointer, bytes) of a caller's workspace: a contiguous tensor on `like`'s device."""
    if workspace is None:
        return None, 0
    if not workspace.is_cuda or workspace.get_device() != like.get_device() or not workspace.is_contiguous():
        raise ValueError(f"{what}: a contiguous tensor on cuda:{like.get_device()} is needed")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def _kv_heads(tensors, what):
    """The head count (dimension 2) of a per-rank list of [b, tokens, heads, d] tensors."""
    if len(tensors) == 0 or tensors[0].dim() != 4:
        raise ValueError(f"{what}: per-rank tensors [b, tokens, heads, d] are needed")
    return tensors[0].shape[2]


def _seq_qkv(q_seq, k_seq, v_seq):
    """Checks seq-layout Q [b, s/P, h_q, d] and K, V [b, s/P, h_kv, d] of P ranks; returns
    (first Q tensor, P, b, s, h_q, h_kv, d)."""
    q0 = _same(q_seq, "q_seq")
    if q0.dim() != 4:
        raise ValueError("q_seq: per-rank tensors [b, s/P, h_q, d] are needed")
    P = len(q_seq)
    b, S, hq, d = q0.shape
    hkv = _kv_heads(k_seq, "k_seq")
    _same(k_seq, "k_seq", P, (b, S, hkv, d), q0)
    _same(v_seq, "v_seq", P, (b, S, hkv, d), q0)
    return q0, P, b, S * P, hq, hkv, d


def ulysses_a2a_seq2head(in_seq, out_head=None, stream=None):
    """All-to-all #1: P tensors [b, s/P, h, d] -> P tensors [b, s, h/P, d]."""
    t0 = _same(in_seq, "in_seq")
    P = len(in_seq)
    b, S, h, d = t0.shape
    if out_head is None:
        out_head = [torch.empty((b, S * P, h // P, d), dtype=t0.dtype, device=t0.device) for _ in range(P)]
    _same(out_head, "out_head", P, (b, S * P, h // P, d), t0)
    _check(load_library().ulysses_a2a_seq2head(P, b, S * P, h, d, _dtype_code(t0), _ptr_array(in_seq),
                                               _ptr_array(out_head), _stream(stream)), "ulysses_a2a_seq2head")
    return out_head


def ulysses_a2a_head2seq(in_head, out_seq=None, stream=None):
    """All-to-all #2: P tensors [b, s, h/P, d] -> P tensors [b, s/P, h, d]."""
    t0 = _same(in_head, "in_head")
    P = len(in_head)
    b, s, H, d = t0.shape
    if out_seq is None:
        out_seq = [torch.empty((b, s // P, H * P, d), dtype=t0.dtype, device=t0.device) for _ in range(P)]
    _same(out_seq, "out_seq", P, (b, s // P, H * P, d), t0)
    _check(load_library().ulysses_a2a_head2seq(P, b, s, H * P, d, _dtype_code(t0), _ptr_array(in_head),
                                               _ptr_array(out_seq), _stream(stream)), "ulysses_a2a_head2seq")
    return out_seq


def ulysses_a2a_pack(local, direction, P, out=None, stream=None):
    """One rank's send blocks for an all-to-all with P processes: direction 0 takes this
    rank's seq shard [b, s/P, h, d], direction 1 its head shard [b, s, h/P, d]; returns
    [P, b, s/P, h/P, d] (block i goes to rank i)."""
    _same([local], "local")
    if direction == 0:
        b, S, h, d = local.shape
        s = S * P
    elif direction == 1:
        b, s, H, d = local.shape
        S, h = s // P, H * P
    else:
        raise ValueError("direction must be 0 (seq -> head) or 1 (head -> seq)")
    if out is None:
        out = torch.empty((P, b, S, h // P, d), dtype=local.dtype, device=local.device)
    _same([out], "out", 1, (P, b, S, h // P, d), local)
    _check(load_library().ulysses_a2a_pack(direction, P, b, s, h, d, _dtype_code(local), local.data_ptr(),
                                           out.data_ptr(), _stream(stream)), "ulysses_a2a_pack")
    return out


def ulysses_a2a_unpack(recv, direction, out=None, stream=None):
    """This rank's layout after an all-to-all with P processes: recv [P, b, s/P, h/P, d]
    (block j came from rank j) -> direction 0: the head shard [b, s, h/P, d]; direction 1:
    the seq shard [b, s/P, h, d]."""
    _same([recv], "recv")
    P, b, S, H, d = recv.shape
    if direction not in (0, 1):
        raise ValueError("direction must be 0 (seq -> head) or 1 (head -> seq)")
    shape = (b, S * P, H, d) if direction == 0 else (b, S, H * P, d)
    if out is None:
        out = torch.empty(shape, dtype=recv.dtype, device=recv.device)
    _same([out], "out", 1, shape, recv)
    _check(load_library().ulysses_a2a_unpack(direction, P, b, S * P, H * P, d, _dtype_code(recv), recv.data_ptr(),
                                             out.data_ptr(), _stream(stream)), "ulysses_a2a_unpack")
    return out


def ulysses_local_attention(q_head, k_head, v_head, causal, out_head=None, stream=None):
    """Attention of every rank in head layout: softmax(Q K^T / sqrt(d)) V per local head."""
    q0 = _same(q_head, "q_head")
    P = len(q_head)
    b, s, Hq, d = q0.shape
    Hk = _kv_heads(k_head, "k_head")
    _same(k_head, "k_head", P, (b, s, Hk, d), q0)
    _same(v_head, "v_head", P, (b, s, Hk, d), q0)
    if out_head is None:
        out_head = [torch.empty_like(q) for q in q_head]
    _same(out_head, "out_head", P, q0.shape, q0)
    _check(load_library().ulysses_local_attention(
        P, b, s, Hq * P, Hk * P, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_head), _ptr_array(k_head),
        _ptr_array(v_head), _ptr_array(out_head), _stream(stream)), "ulysses_local_attention")
    return out_head


def ulysses_dist_attn_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, fused):
    return int(load_library().ulysses_dist_attn_workspace_bytes(P, b, s, h_q, h_kv, d, _DTYPES[dtype], int(bool(fused))))


def ulysses_dist_attn_fwd(q_seq, k_seq, v_seq, causal, fused=False, out_seq=None, workspace=None, stream=None):
    """The whole forward: all-to-all #1 (Q, K, V), attention, all-to-all #2.

    q_seq / k_seq / v_seq: P tensors [b, s/P, heads, d]; returns P tensors [b, s/P, h_q, d].
    ``workspace`` (a uint8 CUDA tensor) is allocated when not given and fused is False.
    """
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    if out_seq is None:
        out_seq = [torch.empty_like(q) for q in q_seq]
    _same(out_seq, "out_seq", P, q0.shape, q0)
    need = ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, q0.dtype, fused)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    _check(load_library().ulysses_dist_attn_fwd(
        P, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(out_seq), ws_ptr, ws_len, int(bool(fused)), _stream(stream)),
        "ulysses_dist_attn_fwd")
    return out_seq


def ulysses_device_status(clear=True):
    """Synchronise and report (and by default clear) the device-side error word."""
    return int(load_library().ulysses_device_status(int(bool(clear))))


# size of the library's fixed scratch array used by ulysses_dist_attn_fwd_noalloc
NOALLOC_SCRATCH_BYTES = 64 << 20


def ulysses_dist_attn_fwd_noalloc(q_seq, k_seq, v_seq, causal, out_seq, stream=None):
    """The unfused forward with the library's fixed scratch array as its workspace.

    For callers that cannot allocate device memory: ``out_seq`` (P tensors
    [b, s/P, h_q, d]) must be supplied, and nothing is allocated here or in the library.
    Calls that would need more than NOALLOC_SCRATCH_BYTES of scratch raise.  Calls that
    overlap on the GPU share the scratch and race; serialise them.
    """
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    _same(out_seq, "out_seq", P, q0.shape, q0)
    _check(load_library().ulysses_dist_attn_fwd_noalloc(
        P, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(out_seq), _stream(stream)), "ulysses_dist_attn_fwd_noalloc")
    return out_seq


# ------------------------------------------------------------------------------ training
def _rows_like(q_head_shape, device):
    b, s, Hq, _ = q_head_shape
    return torch.empty((b, Hq, s), dtype=torch.float32, device=device)


def ulysses_local_attention_fwd_lse(q_head, k_head, v_head, causal, out_head=None, lse=None, stream=None):
    """ulysses_local_attention plus the per-row log-sum-exp: returns (o_head, lse), lse being
    P fp32 tensors [b, h_q/P, s] (natural log of the sum of exp of the scaled scores)."""
    q0 = _same(q_head, "q_head")
    P = len(q_head)
    b, s, Hq, d = q0.shape
    Hk = _kv_heads(k_head, "k_head")
    _same(k_head, "k_head", P, (b, s, Hk, d), q0)
    _same(v_head, "v_head", P, (b, s, Hk, d), q0)
    if out_head is None:
        out_head = [torch.empty_like(q) for q in q_head]
    _same(out_head, "out_head", P, q0.shape, q0)
    if lse is None:
        lse = [_rows_like(q0.shape, q0.device) for _ in range(P)]
    _same(lse, "lse", P, (b, Hq, s), q0, torch.float32)
    _check(load_library().ulysses_local_attention_fwd_lse(
        P, b, s, Hq * P, Hk * P, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_head),
        _ptr_array(k_head), _ptr_array(v_head), _ptr_array(out_head), _ptr_array(lse), _stream(stream)),
        "ulysses_local_attention_fwd_lse")
    return out_head, lse


def ulysses_dist_attn_fwd_lse(q_seq, k_seq, v_seq, causal, fused=False, out_seq=None, lse=None, workspace=None,
                              stream=None):
    """The forward plus the log-sum-exp of every head rank's rows: returns (o_seq, lse) with
    lse P fp32 tensors [b, h_q/P, s] indexed like the head layout."""
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    if out_seq is None:
        out_seq = [torch.empty_like(q) for q in q_seq]
    _same(out_seq, "out_seq", P, q0.shape, q0)
    if lse is None:
        lse = [torch.empty((b, hq // P, s), dtype=torch.float32, device=q0.device) for _ in range(P)]
    _same(lse, "lse", P, (b, hq // P, s), q0, torch.float32)
    need = ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, q0.dtype, fused)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    _check(load_library().ulysses_dist_attn_fwd_lse(
        P, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(out_seq), _ptr_array(lse), ws_ptr, ws_len, int(bool(fused)), _stream(stream)),
        "ulysses_dist_attn_fwd_lse")
    return out_seq, lse


def ulysses_attn_bwd_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, dist, fused=False):
    return int(load_library().ulysses_attn_bwd_workspace_bytes(P, b, s, h_q, h_kv, d, _DTYPES[dtype],
                                                               int(bool(dist)), int(bool(fused))))


def _bwd_call(name, dist, q, k, v, o, do, lse, causal, grads, workspace, stream, fused=False):
    q0 = _same(q, "q")
    P = len(q)
    b, T, Hq, d = q0.shape  # T tokens (s/P seq layout, s head layout), Hq heads of the layout
    Hk = _kv_heads(k, "k")
    _same(k, "k", P, (b, T, Hk, d), q0)
    _same(v, "v", P, (b, T, Hk, d), q0)
    _same(o, "o", P, q0.shape, q0)
    _same(do, "do", P, q0.shape, q0)
    if dist:
        s, hq, hkv = T * P, Hq, Hk
    else:
        s, hq, hkv = T, Hq * P, Hk * P
    _same(lse, "lse", P, (b, hq // P, s), q0, torch.float32)
    if grads is None:
        grads = ([torch.empty_like(x) for x in q], [torch.empty_like(x) for x in k], [torch.empty_like(x) for x in v])
    dq, dk, dv = grads
    _same(dq, "dq", P, q0.shape, q0)
    _same(dk, "dk", P, (b, T, Hk, d), q0)
    _same(dv, "dv", P, (b, T, Hk, d), q0)
    need = ulysses_attn_bwd_workspace_bytes(P, b, s, hq, hkv, d, q0.dtype, dist, fused)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    args = [P, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q), _ptr_array(k), _ptr_array(v),
            _ptr_array(o), _ptr_array(do), _ptr_array(lse), _ptr_array(dq), _ptr_array(dk), _ptr_array(dv),
            ws_ptr, ws_len]
    if dist:
        args.append(int(bool(fused)))
    _check(getattr(load_library(), name)(*args, _stream(stream)), name)
    return dq, dk, dv


def ulysses_local_attention_bwd(q_head, k_head, v_head, o_head, do_head, lse, causal, grads=None, workspace=None,
                                stream=None):
    """Backward of the head-layout attention of every rank: returns (dq, dk, dv) head layout."""
    return _bwd_call("ulysses_local_attention_bwd", False, q_head, k_head, v_head, o_head, do_head, lse, causal,
                     grads, workspace, stream)


def ulysses_dist_attn_bwd(q_seq, k_seq, v_seq, o_seq, do_seq, lse, causal, grads=None, workspace=None, stream=None,
                          fused=False):
    """The DistributedAttention backward, seq layout in and out: returns (dq, dk, dv) seq layout.
    fused=True folds both exchanges into the kernels' tile addressing (same bits)."""
    return _bwd_call("ulysses_dist_attn_bwd", True, q_seq, k_seq, v_seq, o_seq, do_seq, lse, causal, grads,
                     workspace, stream, fused)


# ------------------------------------------------------------------------- overlapped forward
_side_streams = {}


def _side_stream(device):
    """One cached side stream per device for the overlapped forward's exchanges."""
    key = torch.device(device).index
    if key not in _side_streams:
        _side_streams[key] = torch.cuda.Stream(device=device)
    return _side_streams[key]


def ulysses_dist_attn_overlap_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, n_chunks):
    return int(load_library().ulysses_dist_attn_overlap_workspace_bytes(P, b, s, h_q, h_kv, d, _DTYPES[dtype],
                                                                       int(n_chunks)))


def ulysses_dist_attn_fwd_overlap(q_seq, k_seq, v_seq, causal, n_chunks=2, out_seq=None, workspace=None,
                                  stream=None, side_stream=None):
    """The unfused forward with the exchanges of one head group overlapped with the attention
    of the next (n_chunks head groups); same results, bit for bit, as ulysses_dist_attn_fwd."""
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    if out_seq is None:
        out_seq = [torch.empty_like(q) for q in q_seq]
    _same(out_seq, "out_seq", P, q0.shape, q0)
    if workspace is None:
        need = ulysses_dist_attn_overlap_workspace_bytes(P, b, s, hq, hkv, d, q0.dtype, n_chunks)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    side = side_stream if side_stream is not None else _side_stream(q0.device)
    _check(load_library().ulysses_dist_attn_fwd_overlap(
        P, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(out_seq), ws_ptr, ws_len,
        int(n_chunks), _stream(stream), ctypes.c_void_p(side.cuda_stream)), "ulysses_dist_attn_fwd_overlap")
    return out_seq


# ------------------------------------------------------------------ Ulysses x Ring forward
def ulysses_usp_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, dtype):
    return int(load_library().ulysses_usp_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, _DTYPES[dtype]))


def ulysses_usp_attn_fwd(q_seq, k_seq, v_seq, causal, Pu, Pr, out_seq=None, workspace=None, stream=None):
    """The two-level forward over P = Pu*Pr seq-partitioned ranks (rank j = g*Pu + u):
    all-to-all inside groups of Pu ranks, attention with the ring groups' K/V blocks,
    all-to-all back.  Returns P tensors [b, s/P, h_q, d]."""
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    if P != Pu * Pr:
        raise ValueError(f"{P} ranks given for Pu={Pu} x Pr={Pr}")
    if out_seq is None:
        out_seq = [torch.empty_like(q) for q in q_seq]
    _same(out_seq, "out_seq", P, q0.shape, q0)
    if workspace is None:
        need = ulysses_usp_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, q0.dtype)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    _check(load_library().ulysses_usp_attn_fwd(
        Pu, Pr, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(out_seq), ws_ptr, ws_len, _stream(stream)), "ulysses_usp_attn_fwd")
    return out_seq


def ulysses_usp_attn_fwd_lse(q_seq, k_seq, v_seq, causal, Pu, Pr, out_seq=None, lse=None, workspace=None,
                             stream=None):
    """The two-level forward plus its softmax statistics: returns (o_seq, lse) with lse Pu
    fp32 tensors [b, h_q/Pu, s] (Ulysses unit u's heads, every position)."""
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    if P != Pu * Pr:
        raise ValueError(f"{P} ranks given for Pu={Pu} x Pr={Pr}")
    if out_seq is None:
        out_seq = [torch.empty_like(q) for q in q_seq]
    _same(out_seq, "out_seq", P, q0.shape, q0)
    if lse is None:
        lse = [torch.empty((b, hq // Pu, s), dtype=torch.float32, device=q0.device) for _ in range(Pu)]
    _same(lse, "lse", Pu, (b, hq // Pu, s), q0, torch.float32)
    if workspace is None:
        need = ulysses_usp_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, q0.dtype)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    _check(load_library().ulysses_usp_attn_fwd_lse(
        Pu, Pr, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(out_seq), _ptr_array(lse), ws_ptr, ws_len, _stream(stream)),
        "ulysses_usp_attn_fwd_lse")
    return out_seq, lse


def ulysses_usp_bwd_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, dtype):
    return int(load_library().ulysses_usp_bwd_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, _DTYPES[dtype]))


def ulysses_usp_attn_bwd(q_seq, k_seq, v_seq, o_seq, do_seq, lse, causal, Pu, Pr, grads=None, workspace=None,
                         stream=None):
    """Backward of the two-level forward, seq layout in and out: returns (dq, dk, dv)."""
    q0, P, b, s, hq, hkv, d = _seq_qkv(q_seq, k_seq, v_seq)
    if P != Pu * Pr:
        raise ValueError(f"{P} ranks given for Pu={Pu} x Pr={Pr}")
    _same(o_seq, "o_seq", P, q0.shape, q0)
    _same(do_seq, "do_seq", P, q0.shape, q0)
    _same(lse, "lse", Pu, (b, hq // Pu, s), q0, torch.float32)
    if grads is None:
        grads = ([torch.empty_like(x) for x in q_seq], [torch.empty_like(x) for x in k_seq],
                 [torch.empty_like(x) for x in v_seq])
    dq, dk, dv = grads
    _same(dq, "dq", P, q0.shape, q0)
    _same(dk, "dk", P, k_seq[0].shape, q0)
    _same(dv, "dv", P, k_seq[0].shape, q0)
    if workspace is None:
        need = ulysses_usp_bwd_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, q0.dtype)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q0.device)
    ws_ptr, ws_len = _workspace(workspace, q0)
    _check(load_library().ulysses_usp_attn_bwd(
        Pu, Pr, b, s, hq, hkv, d, _dtype_code(q0), int(bool(causal)), _ptr_array(q_seq), _ptr_array(k_seq),
        _ptr_array(v_seq), _ptr_array(o_seq), _ptr_array(do_seq), _ptr_array(lse), _ptr_array(dq), _ptr_array(dk),
        _ptr_array(dv), ws_ptr, ws_len, _stream(stream)), "ulysses_usp_attn_bwd")
    return dq, dk, dv


def ulysses_wait_selftest(limit_ns=50_000_000, stream=None):
    """Enqueue one CTA whose bounded wait on a barrier that nothing completes gives up after
    limit_ns; ulysses_device_status() then reports the timeout (read it with clear=True)."""
    _check(load_library().ulysses_wait_selftest(int(limit_ns), _stream(stream)), "ulysses_wait_selftest")

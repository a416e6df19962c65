"""CPU oracle for the Ulysses DistributedAttention forward and backward, and the two-level
Ulysses x Ring forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import
this package.  The product path (``sequence_attention_seq_gb300``) never does, and this
package never imports the product.  The arithmetic lives in ``ulysses_oracle.c`` (plain
single-threaded fp64 C); this file only marshals arguments and composes the pipeline:

    all-to-all #1 on Q, K and V  ->  per-rank attention  ->  all-to-all #2 on O

("DeepSpeed-Ulysses 深度解析", section "核心设计：沿序列切分 + 两次 All-to-All",
steps 3-5).  Every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ulysses_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libulysses_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float64: 2}


def build(force=False):
    """Compile the oracle with plain gcc (-O2, strict IEEE: no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            lib.orc_all_to_all.argtypes = [i, sz, ctypes.POINTER(vp), ctypes.POINTER(vp)]
            lib.orc_all_to_all.restype = None
            for fn in (lib.orc_seq2head, lib.orc_head2seq):
                fn.argtypes = [i, i, i, i, i, i, ctypes.POINTER(vp), ctypes.POINTER(vp)]
                fn.restype = i
            lib.orc_attention.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp]
            lib.orc_attention.restype = i
            lib.orc_dist_attn_rows.argtypes = [i, i, i, i, i, i, i, i, ctypes.POINTER(vp),
                                               ctypes.POINTER(vp), ctypes.POINTER(vp), i, vp, vp]
            lib.orc_dist_attn_rows.restype = i
            lib.orc_attention_lse.argtypes = [i, i, i, i, i, i, i, vp, vp, vp]
            lib.orc_attention_lse.restype = i
            lib.orc_attention_bwd.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp]
            lib.orc_attention_bwd.restype = i
            lib.orc_usp_fwd.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                        ctypes.POINTER(vp), ctypes.POINTER(vp)]
            lib.orc_usp_fwd.restype = i
            lib.orc_attention_bwd_rows.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, i, vp, i, vp, vp, vp, vp]
            lib.orc_attention_bwd_rows.restype = i
            lib.orc_attention_bwd_magnitudes.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp]
            lib.orc_attention_bwd_magnitudes.restype = i
            _lib = lib
    return _lib


def _ptrs(tensors):
    arr = (ctypes.c_void_p * len(tensors))()
    for n, t in enumerate(tensors):
        arr[n] = t.data_ptr()
    return arr


def _cpu(t):
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    return t.contiguous()


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def all_to_all(chunks):
    """chunks[i][j] = rank i's j-th chunk (equal-size CPU tensors). Returns out[j][i]."""
    P = len(chunks)
    flat = [_cpu(c) for row in chunks for c in row]
    nbytes = flat[0].numel() * flat[0].element_size()
    recv = [torch.empty_like(flat[0]) for _ in range(P * P)]
    _load().orc_all_to_all(P, nbytes, _ptrs(flat), _ptrs(recv))
    return [[recv[j * P + i] for i in range(P)] for j in range(P)]


def seq2head(x_seq, h=None):
    """All-to-all #1: list of P tensors [b, s/P, h, d] -> list of P tensors [b, s, h/P, d]."""
    P = len(x_seq)
    xs = [_cpu(x) for x in x_seq]
    b, S, hh, d = xs[0].shape
    s = S * P
    out = [torch.empty((b, s, hh // P, d), dtype=xs[0].dtype) for _ in range(P)]
    _check(_load().orc_seq2head(P, b, s, hh, d, xs[0].element_size(), _ptrs(xs), _ptrs(out)), "seq2head")
    return out


def head2seq(x_head):
    """All-to-all #2: list of P tensors [b, s, h/P, d] -> list of P tensors [b, s/P, h, d]."""
    P = len(x_head)
    xs = [_cpu(x) for x in x_head]
    b, s, H, d = xs[0].shape
    out = [torch.empty((b, s // P, H * P, d), dtype=xs[0].dtype) for _ in range(P)]
    _check(_load().orc_head2seq(P, b, s, H * P, d, xs[0].element_size(), _ptrs(xs), _ptrs(out)), "head2seq")
    return out


def attention(q, k, v, causal):
    """One rank's local attention in head layout; returns float64 [b, s, h_q, d]."""
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    out = torch.empty((b, s, hq, d), dtype=torch.float64)
    _check(_load().orc_attention(b, s, hq, hkv, d, int(bool(causal)), DTYPE_CODE[q.dtype],
                                 q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr()), "attention")
    return out


def dist_attn_fwd(q_seq, k_seq, v_seq, causal):
    """The whole forward over P seq-partitioned ranks; returns P float64 [b, s/P, h_q, d]."""
    q_head = seq2head(q_seq)
    k_head = seq2head(k_seq)
    v_head = seq2head(v_seq)
    o_head = [attention(q, k, v, causal) for q, k, v in zip(q_head, k_head, v_head)]
    return head2seq(o_head)


def dist_attn_rows(q_seq, k_seq, v_seq, causal, samples):
    """Sampled output rows of the forward: samples = [(rank j, b, t, head), ...] ->
    float64 [n, d].  Same pipeline, evaluated per output row from the seq-layout inputs."""
    P = len(q_seq)
    qs, ks, vs = [_cpu(x) for x in q_seq], [_cpu(x) for x in k_seq], [_cpu(x) for x in v_seq]
    b, S, hq, d = qs[0].shape
    hkv = ks[0].shape[2]
    smp = np.ascontiguousarray(np.asarray(samples, dtype=np.int32).reshape(-1, 4))
    out = np.zeros((smp.shape[0], d), dtype=np.float64)
    _check(_load().orc_dist_attn_rows(P, b, S * P, hq, hkv, d, int(bool(causal)), DTYPE_CODE[qs[0].dtype],
                                      _ptrs(qs), _ptrs(ks), _ptrs(vs), smp.shape[0],
                                      smp.ctypes.data, out.ctypes.data), "dist_attn_rows")
    return torch.from_numpy(out)


def attention_lse(q, k, causal):
    """Per-row log-sum-exp (natural log) of one rank's scaled scores: float64 [b, h_q, s]."""
    q, k = _cpu(q), _cpu(k)
    b, s, hq, d = q.shape
    out = torch.empty((b, hq, s), dtype=torch.float64)
    _check(_load().orc_attention_lse(b, s, hq, k.shape[2], d, int(bool(causal)), DTYPE_CODE[q.dtype],
                                     q.data_ptr(), k.data_ptr(), out.data_ptr()), "attention_lse")
    return out


def attention_bwd(q, k, v, dout, causal):
    """Gradients (dq, dk, dv) of one rank's local attention in head layout, float64."""
    q, k, v, dout = _cpu(q), _cpu(k), _cpu(v), _cpu(dout)
    if not (q.dtype == k.dtype == v.dtype == dout.dtype):
        raise ValueError("q, k, v, dout must share a dtype")
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    dq = torch.empty((b, s, hq, d), dtype=torch.float64)
    dk = torch.empty((b, s, hkv, d), dtype=torch.float64)
    dv = torch.empty((b, s, hkv, d), dtype=torch.float64)
    _check(_load().orc_attention_bwd(b, s, hq, hkv, d, int(bool(causal)), DTYPE_CODE[q.dtype], q.data_ptr(),
                                     k.data_ptr(), v.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr()), "attention_bwd")
    return dq, dk, dv


def attention_bwd_magnitudes(q, k, v, dout, causal):
    """Per gradient element of one rank's local attention backward (head layout), the sum
    of the absolute values of its terms, with every dS_ij widened by P_ij E_i (the
    sensitivity of dS_ij to an output O known only to rounding accuracy): the magnitudes
    (mq, mk, mv), float64, that bound the effect of rounding the terms."""
    q, k, v, dout = _cpu(q), _cpu(k), _cpu(v), _cpu(dout)
    if not (q.dtype == k.dtype == v.dtype == dout.dtype):
        raise ValueError("q, k, v, dout must share a dtype")
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    mq = torch.empty((b, s, hq, d), dtype=torch.float64)
    mk = torch.empty((b, s, hkv, d), dtype=torch.float64)
    mv = torch.empty((b, s, hkv, d), dtype=torch.float64)
    _check(_load().orc_attention_bwd_magnitudes(b, s, hq, hkv, d, int(bool(causal)), DTYPE_CODE[q.dtype],
                                                q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                                mq.data_ptr(), mk.data_ptr(), mv.data_ptr()),
           "attention_bwd_magnitudes")
    return mq, mk, mv


def dist_attn_bwd(q_seq, k_seq, v_seq, do_seq, causal):
    """The Ulysses backward: all-to-all #1 on dO (the backward of all-to-all #2), per-rank
    attention backward, all-to-all #2 on dQ, dK, dV (the backward of all-to-all #1)
    ("02 · DeepSpeed-Ulysses", section 5).  Returns per-rank float64 seq-layout gradients."""
    q_head, k_head, v_head = seq2head(q_seq), seq2head(k_seq), seq2head(v_seq)
    do_head = seq2head(do_seq)
    grads = [attention_bwd(q, k, v, g, causal) for q, k, v, g in zip(q_head, k_head, v_head, do_head)]
    return (head2seq([x[0] for x in grads]), head2seq([x[1] for x in grads]), head2seq([x[2] for x in grads]))


def usp_fwd(q_seq, k_seq, v_seq, causal, Pu, Pr):
    """The two-level (Ulysses inside groups of Pu ranks, ring across Pr groups) forward over
    P = Pu*Pr seq-partitioned ranks, rank j = g*Pu + u; returns P float64 [b, s/P, h_q, d]."""
    P = len(q_seq)
    if P != Pu * Pr:
        raise ValueError("len(q_seq) must be Pu * Pr")
    qs, ks, vs = [_cpu(x) for x in q_seq], [_cpu(x) for x in k_seq], [_cpu(x) for x in v_seq]
    if not (qs[0].dtype == ks[0].dtype == vs[0].dtype):
        raise ValueError("q, k, v must share a dtype")
    b, S, hq, d = qs[0].shape
    out = [torch.empty((b, S, hq, d), dtype=torch.float64) for _ in range(P)]
    _check(_load().orc_usp_fwd(Pu, Pr, b, S * P, hq, ks[0].shape[2], d, int(bool(causal)), DTYPE_CODE[qs[0].dtype],
                               _ptrs(qs), _ptrs(ks), _ptrs(vs), _ptrs(out)), "usp_fwd")
    return out


def usp_group_exchange(x_seq, Pu):
    """Step 1 of the two-level forward alone: all-to-all #1 inside every group of Pu
    consecutive ranks; returns per-rank head-layout tensors [b, s/Pr, h/Pu, d]."""
    out = []
    for g in range(len(x_seq) // Pu):
        out += seq2head(list(x_seq[g * Pu:(g + 1) * Pu]))
    return out


def attention_bwd_rows(q, k, v, dout, causal, q_samples, k_samples):
    """Selected gradient rows of one rank's local attention (head layout):
    q_samples = [(b, i, head), ...] -> dq rows; k_samples = [(b, j, kv_head), ...] -> dk, dv
    rows (summed over the query heads of the group).  Returns float64 (dq [nq, d], dk, dv [nk, d])."""
    q, k, v, dout = _cpu(q), _cpu(k), _cpu(v), _cpu(dout)
    b, s, hq, d = q.shape
    qa = np.ascontiguousarray(np.asarray(q_samples, dtype=np.int32).reshape(-1, 3))
    ka = np.ascontiguousarray(np.asarray(k_samples, dtype=np.int32).reshape(-1, 3))
    dq = np.zeros((qa.shape[0], d)); dk = np.zeros((ka.shape[0], d)); dv = np.zeros((ka.shape[0], d))
    _check(_load().orc_attention_bwd_rows(b, s, hq, k.shape[2], d, int(bool(causal)), DTYPE_CODE[q.dtype],
                                          q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                          qa.shape[0], qa.ctypes.data, ka.shape[0], ka.ctypes.data,
                                          dq.ctypes.data, dk.ctypes.data, dv.ctypes.data), "attention_bwd_rows")
    return torch.from_numpy(dq), torch.from_numpy(dk), torch.from_numpy(dv)

"""Float64 CPU oracle for grouped-query attention with learned sinks.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The
sink-attention library never imports it, and it imports nothing from the
library: the two share only the seeded input generators.

The arithmetic lives in ``sinkattn_oracle.c`` (plain loops in double
precision). This module only marshals arrays into it. What it computes is the
definition on page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink
Attention": a softmax over the scaled Q.K scores together with one learned
per-head sink logit, whose value row is zero, followed by a weighted sum of V.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_attention.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i,
                                         p, i, i, i, ctypes.c_double, p, p, p, p, i]
        lib.oracle_attention.restype = i
        lib.oracle_attention_rows.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i,
                                              p, i, i, ctypes.c_double, p,
                                              ctypes.c_long, p, p, i]
        lib.oracle_attention_rows.restype = i
        lib.oracle_merge.argtypes = [p, p, i, ctypes.c_long, i, i, p, p, p]
        lib.oracle_merge.restype = i
        _LIB = lib
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _bits(x):
    """bf16 data as a contiguous uint16 array of its bit patterns.

    Accepts a torch bf16 tensor (reinterpreted, not converted) or a numpy
    uint16 array of bit patterns.
    """
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x):
    if x is None:
        return None
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy() if hasattr(x, "detach") else np.asarray(x)
    return np.ascontiguousarray(x, dtype=np.int32)


def _f32(x):
    if x is None:
        return None
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy() if hasattr(x, "detach") else np.asarray(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


class _KV:
    """K/V source in either layout, kept alive while the C call runs."""

    def __init__(self, k, v, cu_seqlens_k=None, block_table=None, seqlens_k=None):
        self.k = _bits(k)
        self.v = _bits(v)
        self.cu_k = _i32(cu_seqlens_k)
        self.block_table = _i32(block_table)
        self.seqlens_k = _i32(seqlens_k)
        if self.cu_k is None:
            if self.block_table is None or self.seqlens_k is None:
                raise ValueError("give cu_seqlens_k, or block_table and seqlens_k")
            self.max_pages = self.block_table.shape[1]
            self.page_size = self.k.shape[2]
        else:
            self.max_pages = 0
            self.page_size = 0


def attention(q, k, v, cu_seqlens_q, cu_seqlens_k=None, *, block_table=None,
              seqlens_k=None, hq, hkv, head_dim, sinks=None, causal=True,
              window=0, scale, kv_begin=None, kv_end=None, use_sink=True,
              nthreads=None):
    """Sink attention for every query row.

    q: bf16 [total_q, hq, head_dim]; K/V contiguous bf16 [total_k, hkv, D]
    with cu_seqlens_k, or paged bf16 [num_pages, hkv, page_size, D] with
    block_table [batch, max_pages] and seqlens_k [batch]. Returns float64
    (out [total_q, hq, D], lse [total_q, hq]); lse is a natural log.
    kv_begin/kv_end restrict each sequence to a key range (a split-KV block);
    use_sink=False leaves the sink out of that block.
    """
    qb = _bits(q)
    cu_q = _i32(cu_seqlens_q)
    kv = _KV(k, v, cu_seqlens_k, block_table, seqlens_k)
    s = _f32(sinks)
    kb = _i32(kv_begin)
    ke = _i32(kv_end)
    batch = len(cu_q) - 1
    total_q = int(cu_q[-1])
    out = np.empty((total_q, hq, head_dim), dtype=np.float64)
    lse = np.empty((total_q, hq), dtype=np.float64)
    rc = _lib().oracle_attention(
        _ptr(qb), _ptr(cu_q), _ptr(kv.k), _ptr(kv.v), _ptr(kv.cu_k),
        _ptr(kv.block_table), _ptr(kv.seqlens_k), kv.max_pages, kv.page_size,
        batch, hq, hkv, head_dim, _ptr(s), 1 if use_sink else 0,
        1 if causal else 0, int(window), float(scale), _ptr(kb), _ptr(ke),
        _ptr(out), _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return out, lse


def attention_rows(rows, q, k, v, cu_seqlens_q, cu_seqlens_k=None, *,
                   block_table=None, seqlens_k=None, hq, hkv, head_dim,
                   sinks=None, causal=True, window=0, scale, nthreads=None):
    """The same definition for selected rows only.

    rows: int array [n, 3] of (sequence b, q-head h, query index i within b).
    Returns float64 (out [n, D], lse [n]).
    """
    r = _i32(rows).reshape(-1, 3)
    qb = _bits(q)
    cu_q = _i32(cu_seqlens_q)
    kv = _KV(k, v, cu_seqlens_k, block_table, seqlens_k)
    s = _f32(sinks)
    batch = len(cu_q) - 1
    n = r.shape[0]
    out = np.empty((n, head_dim), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _lib().oracle_attention_rows(
        _ptr(qb), _ptr(cu_q), _ptr(kv.k), _ptr(kv.v), _ptr(kv.cu_k),
        _ptr(kv.block_table), _ptr(kv.seqlens_k), kv.max_pages, kv.page_size,
        batch, hq, hkv, head_dim, _ptr(s), 1 if causal else 0, int(window),
        float(scale), _ptr(r), n, _ptr(out), _ptr(lse),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return out, lse


def merge(partial_o, partial_lse, sinks=None):
    """Merge split-KV blocks by log-sum-exp; the sink, if given, enters once.

    partial_o: [nsplit, rows, hq, D]; partial_lse: [nsplit, rows, hq] (natural
    log, -inf for an empty block). Returns float64 (out [rows, hq, D],
    lse [rows, hq]).
    """
    po = np.ascontiguousarray(np.asarray(partial_o, dtype=np.float64))
    pl = np.ascontiguousarray(np.asarray(partial_lse, dtype=np.float64))
    nsplit, rows, hq, d = po.shape
    assert pl.shape == (nsplit, rows, hq)
    s = _f32(sinks)
    out = np.empty((rows, hq, d), dtype=np.float64)
    lse = np.empty((rows, hq), dtype=np.float64)
    rc = _lib().oracle_merge(_ptr(po), _ptr(pl), nsplit, rows, hq, d, _ptr(s),
                             _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return out, lse

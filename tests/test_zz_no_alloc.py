"""sinkattn_decode_noalloc, the decode entry point that allocates nothing.

Callers that may not allocate device memory (a memory planner that owns every
device byte, a plugin host that forbids allocation while enqueueing, a
latency-critical loop where cudaMalloc/cudaFree could synchronise the device)
use this entry point; its split-KV scratch is a fixed array inside the
library. Called here through the C ABI (ctypes), several times in a row on
different inputs (split and unsplit plans, paged and contiguous caches,
head_dim 64 and 128), each time against sinkattn_decode with a caller
workspace and against the oracle, within the parity tolerance of the other
tests. This file is collected last.
"""
import ctypes

import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import sinkattn as B
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, to_np

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _oracle(c):
    import oracle
    cu_q = torch.arange(0, c.batch + 1, dtype=torch.int32)
    if c.paged:
        return oracle.attention(c.q, c.k_cache, c.v_cache, cu_q, block_table=c.block_table,
                                seqlens_k=c.seqlens_k_t, hq=c.hq, hkv=c.hkv,
                                head_dim=c.head_dim, sinks=c.sinks, causal=True,
                                window=c.window, scale=c.scale)
    return oracle.attention(c.q, c.k, c.v, cu_q, c.kv_indptr, hq=c.hq, hkv=c.hkv,
                            head_dim=c.head_dim, sinks=c.sinks, causal=True, window=c.window,
                            scale=c.scale)


def _noalloc_c_abi(lib, c, dev, num_splits=0):
    """One call of sinkattn_decode_noalloc through the C ABI."""
    q = c.q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((c.batch, c.hq), dtype=torch.float32, device=dev)
    sinks = c.sinks.to(dev)
    if c.paged:
        k, v = c.k_cache.to(dev), c.v_cache.to(dev)
        indptr, table, seql = None, c.block_table.to(dev), c.seqlens_k_t.to(dev)
        rows, maxp, ps = k.shape[0], table.shape[1], k.shape[2]
    else:
        k, v = c.k.to(dev), c.v.to(dev)
        indptr, table, seql = c.kv_indptr.to(dev), None, None
        rows, maxp, ps = k.shape[0], 0, 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.sinkattn_decode_noalloc(_p(q), _p(k), _p(v), _p(indptr), _p(table), _p(seql), rows,
                                     maxp, ps, c.batch, c.max_seqlen_k, c.hq, c.hkv, c.head_dim,
                                     _p(sinks), B.Mask(1, c.window, c.scale), num_splits, _p(out),
                                     _p(lse), stream)
    assert st == B.SINKATTN_OK, (st, lib.sinkattn_last_cuda_error())
    # the existing entry point, with its own workspace, on the same inputs
    ref_out, ref_lse = sa.sinkattn_decode(q, k, v, kv_indptr=indptr, block_table=table,
                                          seqlens_k=seql, max_seqlen_k=c.max_seqlen_k,
                                          sinks=sinks, window=c.window, scale=c.scale,
                                          num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse, ref_out, ref_lse


# Calls in a row on different inputs: the automatic split plan (contiguous and
# paged), a 128-token window (one warp per sequence and KV head, no scratch
# used), and head_dim 128 with an explicit split count whose scratch (partials
# of twice the width) still fits the array.
CASES = [
    ("contig", lambda: S.make_decode("noalloc_a", [3000, 100, 5000, 4097, 1], 64, 8, seed=201),
     0),
    ("paged", lambda: S.make_decode("noalloc_b", [2500, 7000, 33, 1030], 64, 8, seed=202,
                                    paged=True, sink_std=2.0), 0),
    ("window128", lambda: S.make_decode("noalloc_c", [3000, 90, 128, 1, 700], 64, 8, seed=203,
                                        window=128, paged=True), 0),
    ("d128_splits", lambda: S.make_decode("noalloc_d", [6000, 4097, 1, 300], 64, 8, seed=204,
                                          head_dim=128), 5),
]


def test_noalloc_decode_matches_workspace_decode_twice():
    lib = sa.load()
    dev = torch.device("cuda", 0)
    for name, mk, ns in CASES:
        c = mk()
        if ns:
            need = lib.sinkattn_decode_workspace_size(c.batch, c.max_seqlen_k, c.hq, c.hkv,
                                                      c.head_dim, c.window, ns)
            assert 0 < need <= B.SINKATTN_NOALLOC_SCRATCH_BYTES
        out, lse, ref_out, ref_lse = _noalloc_c_abi(lib, c, dev, ns)
        # the same kernels and split plan as the workspace call: equal results
        check_close(out, lse, to_np(ref_out), to_np(ref_lse), "noalloc vs decode " + name)
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), name
        ro, rl = _oracle(c)
        check_close(out, lse, ro, rl, "noalloc vs oracle " + name)


def test_noalloc_rejects_plans_beyond_its_scratch():
    lib = sa.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call is rejected first
    need = lib.sinkattn_decode_workspace_size(256, 32768, 64, 8, 64, 0, 64)
    assert need > (32 << 20)
    st = lib.sinkattn_decode_noalloc(fake, fake, fake, fake, None, None, 1000, 0, 0, 256, 32768,
                                     64, 8, 64, None, B.Mask(1, 0, 0.125), 64, fake, None, None)
    assert st == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL

"""GPU prefill of packed queries against a paged KV cache, against the float64
oracle (which reads the same pages through the same block table)."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, cuda

pytestmark = pytest.mark.gpu


def run_paged(c, max_seqlen_k=None, block_table=None, seqlens_k=None):
    return sa.sinkattn_prefill_paged(
        c.q.cuda(), c.cu_seqlens_q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(),
        (c.block_table if block_table is None else block_table).cuda(),
        (c.seqlens_k_t if seqlens_k is None else seqlens_k).cuda(), c.max_seqlen_q,
        c.max_seqlen_k if max_seqlen_k is None else max_seqlen_k, sinks=cuda(c.sinks),
        causal=c.causal, window=c.window, scale=c.scale)


def oracle_paged(oracle, c):
    return oracle.attention(c.q, c.k_cache, c.v_cache, c.cu_seqlens_q,
                            block_table=c.block_table, seqlens_k=c.seqlens_k_t, hq=c.hq,
                            hkv=c.hkv, head_dim=c.head_dim, sinks=c.sinks, causal=c.causal,
                            window=c.window, scale=c.scale)


def poison_unreferenced(c):
    """NaN into every page slot no sequence references (spare pages, the tail
    of each last page): the result must not depend on them."""
    used = torch.zeros(c.k_cache.shape[0], c.page_size, dtype=torch.bool)
    for b, L in enumerate(c.seqlens_k):
        for j in range(L):
            used[int(c.block_table[b, j // c.page_size]), j % c.page_size] = True
    free = ~used
    for t in (c.k_cache, c.v_cache):
        t.permute(0, 2, 1, 3)[free] = float("nan")


# (query lengths, key lengths): chunked (lq < lk), lq == lk, more queries than
# keys, empty sequences, lengths around the 128-row tile and page boundaries
SHAPES = [
    ([64], [64]),
    ([1], [1]),
    ([129], [129]),
    ([200], [700]),
    ([130], [40]),
    ([300, 17, 256, 1], [1000, 17, 256, 33]),
    ([0, 64, 0, 5], [0, 64, 5, 300]),
    ([513, 128], [2049, 128]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
# page sizes below, at and above the 8-row swizzle atom and the 128-key tile
@pytest.mark.parametrize("page_size", [16, 1, 7, 128, 8, 64, 256])
def test_prefill_paged_shapes(oracle_lib, shape, page_size):
    lq, lk = shape
    c = S.make_prefill_paged("pshape", lq, lk, 8, 2, seed=81 + sum(lk) + page_size,
                             page_size=page_size, spare_pages=3, sink_std=1.5)
    poison_unreferenced(c)
    out, lse = run_paged(c)
    ro, rl = oracle_paged(oracle_lib, c)
    check_close(out, lse, ro, rl, "paged prefill %s page=%d" % (shape, page_size))


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 1), (True, 128), (True, 300),
                                           (False, 50)])
def test_prefill_paged_masks(oracle_lib, causal, window):
    c = S.make_prefill_paged("pmask", [300, 45, 700], [1300, 45, 900], 8, 2, seed=83 + window,
                             causal=causal, window=window, page_size=16, spare_pages=2)
    poison_unreferenced(c)
    out, lse = run_paged(c)
    ro, rl = oracle_paged(oracle_lib, c)
    check_close(out, lse, ro, rl, "paged prefill causal=%s w=%d" % (causal, window))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (12, 3), (64, 8)])
def test_prefill_paged_groups_and_no_sink(oracle_lib, hq, hkv):
    for with_sinks in (True, False):
        c = S.make_prefill_paged("pgrp", [190, 260], [400, 260], hq, hkv, seed=85 + hq,
                                 with_sinks=with_sinks, page_size=16)
        out, lse = run_paged(c)
        ro, rl = oracle_paged(oracle_lib, c)
        check_close(out, lse, ro, rl, "paged hq=%d hkv=%d sinks=%s" % (hq, hkv, with_sinks))


def _contiguous_copy(c):
    """The paged tokens laid out as packed contiguous K/V."""
    ks, vs = [], []
    for b, L in enumerate(c.seqlens_k):
        j = torch.arange(L)
        pages = c.block_table[b, j // c.page_size].long()
        ks.append(c.k_cache[pages, :, j % c.page_size])
        vs.append(c.v_cache[pages, :, j % c.page_size])
    return torch.cat(ks), torch.cat(vs), S.offsets(c.seqlens_k)


@pytest.mark.parametrize("window", [0, 128])
def test_paged_equals_contiguous_bitwise(window):
    """Staging packs the pages in sequence order, so the kernel sees the same
    rows as the contiguous call and the results are bitwise equal."""
    c = S.make_prefill_paged("peq", [700, 1, 333, 2000], [3000, 1, 333, 2100], 64, 8, seed=87,
                             window=window, page_size=16, spare_pages=5)
    k, v, cu_k = _contiguous_copy(c)
    a = run_paged(c)
    b = sa.sinkattn_prefill(c.q.cuda(), k.cuda(), v.cuda(), c.cu_seqlens_q.cuda(), cu_k.cuda(),
                            c.max_seqlen_q, c.max_seqlen_k, sinks=c.sinks.cuda(), causal=True,
                            window=window, scale=c.scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_paged_slack_in_max_seqlen_k(oracle_lib):
    """A host bound larger than every Lk_b (a table with spare columns) only
    grows the staging."""
    c = S.make_prefill_paged("pslack", [100, 300], [500, 300], 8, 2, seed=89, page_size=16)
    table = torch.zeros((2, 64), dtype=torch.int32)
    table[:, :c.block_table.shape[1]] = c.block_table
    out, lse = run_paged(c, max_seqlen_k=64 * 16, block_table=table)
    ro, rl = oracle_paged(oracle_lib, c)
    check_close(out, lse, ro, rl, "slack max_seqlen_k")


def test_paged_bad_page_and_length_are_reported():
    """A block-table entry outside the cache and a length above the host bound
    are caught by the gather's own checks: error codes 2 and 3, finite output."""
    c = S.make_prefill_paged("pbad", [64], [300], 8, 2, seed=91, page_size=16)
    assert sa.sinkattn_get_device_error() == 0
    table = c.block_table.clone()
    table[0, 3] = c.k_cache.shape[0] + 1000
    out, lse = run_paged(c, block_table=table)
    assert sa.sinkattn_get_device_error() == 2
    assert torch.isfinite(out.float()).all()
    out, lse = run_paged(c, max_seqlen_k=256, block_table=c.block_table[:, :16].contiguous())
    assert sa.sinkattn_get_device_error() == 3
    assert torch.isfinite(out.float()).all()


def _sample_rows(c, per_seq, seed):
    g = torch.Generator().manual_seed(seed)
    rows = []
    for b, lq in enumerate(c.seqlens_q):
        if lq == 0:
            continue
        idx = set([0, lq - 1, min(lq - 1, 127), min(lq - 1, 128)])
        idx |= set(torch.randint(0, lq, (per_seq,), generator=g).tolist())
        for i in sorted(idx):
            for h in torch.randint(0, c.hq, (2,), generator=g).tolist():
                rows.append((b, h, i))
    return np.array(rows, dtype=np.int32)


def _every_item_rows(c, seed):
    """One random row of every (sequence, 128-row query tile, query head): every
    work item of the call, ragged last tiles included."""
    g = torch.Generator().manual_seed(seed)
    rows = []
    for b, lq in enumerate(c.seqlens_q):
        for qt in range((lq + 127) // 128):
            n = min(128, lq - qt * 128)
            pick = torch.randint(0, n, (c.hq,), generator=g).tolist()
            rows += [(b, h, qt * 128 + i) for h, i in enumerate(pick)]
    return np.array(rows, dtype=np.int32)


def _check_rows(oracle, c, out, lse, rows, what):
    ro, rl = oracle.attention_rows(rows, c.q, c.k_cache, c.v_cache, c.cu_seqlens_q,
                                   block_table=c.block_table, seqlens_k=c.seqlens_k_t, hq=c.hq,
                                   hkv=c.hkv, head_dim=c.head_dim, sinks=c.sinks, causal=c.causal,
                                   window=c.window, scale=c.scale)
    cu = c.cu_seqlens_q.tolist()
    pr = torch.tensor([cu[b] + i for b, _, i in rows], device=out.device)
    ph = torch.tensor([h for _, h, _ in rows], device=out.device)
    check_close(out[pr, ph], lse[pr, ph], ro, rl, what)


def test_paged_chunked_prefill_full_config(oracle_lib):
    """4096 queries at the end of a 131072-token context held in 16-token pages
    under a permuted block table. One row of every (query tile, head) item,
    and sampled rows, against the oracle."""
    c = S.paged_chunked_prefill()
    out, lse = run_paged(c)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, c, out, lse, _every_item_rows(c, 92), "paged_chunked_prefill items")
    _check_rows(oracle_lib, c, out, lse, _sample_rows(c, 40, 93), "paged_chunked_prefill")


def test_paged_prefill_batch_full_config(oracle_lib):
    """16 sequences, new chunks of 256..2048 tokens after 1k..32k cached tokens.
    One row of every (query tile, head) item, and sampled rows, against the
    oracle."""
    c = S.paged_prefill_batch()
    out, lse = run_paged(c)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, c, out, lse, _every_item_rows(c, 94), "paged_prefill_batch items")
    _check_rows(oracle_lib, c, out, lse, _sample_rows(c, 12, 95), "paged_prefill_batch")
    assert sa.sinkattn_get_device_error() == 0


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("page_size", [16, 7])
def test_prefill_paged_head_dim_128(oracle_lib, shape, page_size):
    lq, lk = shape
    c = S.make_prefill_paged("pd128", lq, lk, 8, 2, seed=141 + sum(lk) + page_size,
                             page_size=page_size, spare_pages=3, sink_std=1.5, head_dim=128)
    poison_unreferenced(c)
    out, lse = run_paged(c)
    ro, rl = oracle_paged(oracle_lib, c)
    check_close(out, lse, ro, rl, "paged d128 %s page=%d" % (shape, page_size))


def test_paged_equals_contiguous_bitwise_head_dim_128():
    c = S.make_prefill_paged("peq128", [700, 1, 333], [3000, 1, 500], 16, 4, seed=143,
                             page_size=16, spare_pages=5, head_dim=128)
    k, v, cu_k = _contiguous_copy(c)
    a = run_paged(c)
    b = sa.sinkattn_prefill(c.q.cuda(), k.cuda(), v.cuda(), c.cu_seqlens_q.cuda(), cu_k.cuda(),
                            c.max_seqlen_q, c.max_seqlen_k, sinks=c.sinks.cuda(), causal=True,
                            scale=c.scale)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])

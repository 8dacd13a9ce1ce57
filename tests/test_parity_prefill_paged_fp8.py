"""GPU prefill against a paged fp8 e4m3 KV cache, against the float64 oracle.

The oracle decodes the same e4m3 codes exactly (oracle/fp8.py), applies the
per-KV-head scales and runs the float64 forward on those values."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, cuda
from oracle import backward as OB
from oracle import fp8 as F

pytestmark = pytest.mark.gpu


def run(c, num_splits=0, scales=True, block_table=None):
    return sa.sinkattn_prefill_paged_fp8(
        c.q.cuda(), c.cu_seqlens_q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(),
        (c.block_table if block_table is None else block_table).cuda(), c.seqlens_k_t.cuda(),
        c.max_seqlen_q, c.max_seqlen_k, k_scale=cuda(c.k_scale) if scales else None,
        v_scale=cuda(c.v_scale) if scales else None, sinks=cuda(c.sinks), causal=c.causal,
        window=c.window, scale=c.scale, num_splits=num_splits)


def _dequant_seq(c, b, scales=True):
    """float64 K, V [Lk_b, hkv, D] of sequence b, read through its block table."""
    L = c.seqlens_k[b]
    j = np.arange(L)
    pages = c.block_table[b].numpy()[j // c.page_size]
    kc = c.k_cache.numpy()[pages, :, j % c.page_size]
    vc = c.v_cache.numpy()[pages, :, j % c.page_size]
    ks = c.k_scale if scales else torch.ones(c.hkv)
    vs = c.v_scale if scales else torch.ones(c.hkv)
    return (F.dequantize(kc.reshape(L, c.hkv, c.head_dim), ks, 1),
            F.dequantize(vc.reshape(L, c.hkv, c.head_dim), vs, 1))


def reference(c, scales=True):
    kd, vd = zip(*[_dequant_seq(c, b, scales) for b in range(c.batch)])
    cu_k = np.concatenate([[0], np.cumsum(c.seqlens_k)]).astype(np.int64)
    return OB.forward(c.q, np.concatenate(kd), np.concatenate(vd), c.cu_seqlens_q, cu_k,
                      hq=c.hq, hkv=c.hkv, sinks=c.sinks, causal=c.causal, window=c.window,
                      scale=c.scale)


def reference_rows(c, rows):
    """Sampled (sequence, head, query) rows: each one is the oracle's forward of
    that single query over exactly the keys the mask lets it see."""
    group = c.hq // c.hkv
    cache = {}
    outs, lses = [], []
    for b, h, i in rows:
        if b not in cache:
            cache = {b: _dequant_seq(c, b)}
        kd, vd = cache[b]
        lq, lk = c.seqlens_q[b], c.seqlens_k[b]
        p = lk - lq + i
        hi = min(lk, p + 1) if c.causal else lk
        lo = max(0, p - c.window + 1) if c.window > 0 else 0
        g = h // group
        q = c.q[int(c.cu_seqlens_q[b]) + i, h].reshape(1, 1, -1)
        o, l = OB.forward(q, kd[lo:hi, g:g + 1], vd[lo:hi, g:g + 1], np.array([0, 1]),
                          np.array([0, hi - lo]), hq=1, hkv=1, sinks=c.sinks[h:h + 1],
                          causal=False, scale=c.scale)
        outs.append(o[0, 0])
        lses.append(l[0, 0])
    return np.stack(outs), np.array(lses)


SHAPES = [
    ([64], [64]),
    ([1], [1]),
    ([129], [129]),
    ([200], [700]),
    ([130], [40]),
    ([300, 17, 256, 1], [1000, 17, 256, 33]),
    ([0, 64, 0, 5], [0, 64, 5, 300]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("page_size,d", [(16, 64), (7, 64), (16, 128)])
def test_prefill_paged_fp8_shapes(shape, page_size, d):
    lq, lk = shape
    c = S.make_prefill_paged("p8", lq, lk, 8, 2, seed=151 + sum(lk) + page_size + d,
                             page_size=page_size, spare_pages=3, sink_std=1.5, head_dim=d,
                             kv_dtype="fp8")
    out, lse = run(c)
    ro, rl = reference(c)
    check_close(out, lse, ro, rl, "paged fp8 %s page=%d d=%d" % (shape, page_size, d))


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 1), (True, 128), (False, 50)])
def test_prefill_paged_fp8_masks(causal, window):
    c = S.make_prefill_paged("p8m", [300, 45, 700], [1300, 45, 900], 8, 2, seed=153 + window,
                             causal=causal, window=window, page_size=16, kv_dtype="fp8")
    out, lse = run(c)
    ro, rl = reference(c)
    check_close(out, lse, ro, rl, "paged fp8 causal=%s w=%d" % (causal, window))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (12, 3), (64, 8)])
def test_prefill_paged_fp8_groups_and_splits(hq, hkv):
    c = S.make_prefill_paged("p8g", [190, 260], [900, 260], hq, hkv, seed=155 + hq,
                             page_size=16, kv_dtype="fp8")
    ro, rl = reference(c)
    for num_splits in (0, 3):
        out, lse = run(c, num_splits=num_splits)
        check_close(out, lse, ro, rl, "paged fp8 hq=%d hkv=%d splits=%d"
                    % (hq, hkv, num_splits))


def test_prefill_paged_fp8_null_scales_mean_one():
    """Codes drawn for unit scales (values ~N(0, 1) in e4m3): NULL scales give
    the oracle's result for scale 1, bitwise equal to explicit ones."""
    c = S.make_prefill_paged("p8u", [190, 260], [900, 260], 64, 8, seed=156, page_size=16,
                             kv_dtype="fp8")
    one = torch.ones(c.hkv)
    c.k_cache = S.e4m3_codes(tuple(c.k_cache.shape), 1561, one, 1)
    c.v_cache = S.e4m3_codes(tuple(c.v_cache.shape), 1562, one, 1)
    out, lse = run(c, scales=False)
    ro, rl = reference(c, scales=False)
    check_close(out, lse, ro, rl, "paged fp8 NULL scales")
    c.k_scale, c.v_scale = one, one
    o2, l2 = run(c)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_prefill_paged_fp8_table_permutation_invariant():
    """The same tokens under another page placement give bitwise equal results."""
    c = S.make_prefill_paged("p8perm", [300, 100], [1000, 400], 16, 2, seed=157,
                             page_size=16, spare_pages=4, kv_dtype="fp8")
    a = run(c)
    perm = torch.randperm(c.k_cache.shape[0], generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    c2 = S.make_prefill_paged("p8perm", [300, 100], [1000, 400], 16, 2, seed=157,
                              page_size=16, spare_pages=4, kv_dtype="fp8")
    c2.k_cache = c.k_cache[perm].contiguous()  # new page n holds old page perm[n]
    c2.v_cache = c.v_cache[perm].contiguous()
    table = inv[c.block_table.long()].to(torch.int32)
    b = run(c2, block_table=table)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_prefill_paged_fp8_full_config():
    """4096 queries at the end of a 131072-token context in 16-token fp8
    pages. Sampled rows against the oracle."""
    c = S.paged_chunked_prefill_fp8()
    out, lse = run(c)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(159)
    idx = set(torch.randint(0, 4096, (36,), generator=g).tolist())
    idx = sorted(idx | {0, 127, 128, 4095})
    rows = [(0, int(torch.randint(0, c.hq, (1,), generator=g)), i) for i in idx]
    ro, rl = reference_rows(c, rows)
    pr = torch.tensor([i for _, _, i in rows], device=out.device)
    ph = torch.tensor([h for _, h, _ in rows], device=out.device)
    check_close(out[pr, ph], lse[pr, ph], ro, rl, "paged_chunked_prefill_fp8")
    assert sa.sinkattn_get_device_error() == 0

"""GPU-only invariants of the sink-attention kernels (no oracle needed).

- paged and contiguous decode of the same tokens are bitwise equal under the
  same split plan (the layout changes addresses only);
- permuting the pages (and the block table with them) changes nothing;
- decode of a sequence's last token equals the last row of its prefill
  (within the parity tolerance: different kernels, same definition);
- the decode result does not depend on the number of KV splits (tolerance);
- repeated calls are bitwise identical (no floating-point atomics).
"""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_pair

pytestmark = pytest.mark.gpu

LENS = [700, 1, 2049, 333, 4096, 17]


def _paged_from_contig(c, page_size, seed):
    """The same tokens as a contiguous case, scattered over randomly ordered pages."""
    g = torch.Generator().manual_seed(seed)
    npages = [(l + page_size - 1) // page_size for l in c.seqlens_k]
    total = sum(npages)
    perm = torch.randperm(total, generator=g)
    kc = torch.zeros((total, c.hkv, page_size, 64), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    table = torch.zeros((c.batch, max(npages)), dtype=torch.int32)
    at = 0
    for b, L in enumerate(c.seqlens_k):
        k0 = int(c.kv_indptr[b])
        for i in range(npages[b]):
            page = int(perm[at + i])
            table[b, i] = page
            lo, hi = i * page_size, min(L, (i + 1) * page_size)
            kc[page, :, : hi - lo] = c.k[k0 + lo:k0 + hi].transpose(0, 1)
            vc[page, :, : hi - lo] = c.v[k0 + lo:k0 + hi].transpose(0, 1)
        at += npages[b]
    return kc, vc, table


def _decode_contig(c, ns=0, window=0):
    return sa.sinkattn_decode(c.q.cuda(), c.k.cuda(), c.v.cuda(), kv_indptr=c.kv_indptr.cuda(),
                              max_seqlen_k=c.max_seqlen_k, sinks=c.sinks.cuda(), window=window,
                              num_splits=ns)


@pytest.mark.parametrize("window", [0, 300])
@pytest.mark.parametrize("ns", [0, 3])
def test_paged_equals_contiguous_bitwise(ns, window):
    c = S.make_decode("inv", LENS, 64, 8, seed=301)
    out_c, lse_c = _decode_contig(c, ns, window)
    kc, vc, table = _paged_from_contig(c, 16, seed=302)
    out_p, lse_p = sa.sinkattn_decode(c.q.cuda(), kc.cuda(), vc.cuda(), block_table=table.cuda(),
                                      seqlens_k=torch.tensor(LENS, dtype=torch.int32).cuda(),
                                      max_seqlen_k=c.max_seqlen_k, sinks=c.sinks.cuda(),
                                      window=window, num_splits=ns)
    assert torch.equal(out_c, out_p)
    assert torch.equal(lse_c, lse_p)


def test_page_permutation_invariance():
    c = S.make_decode("perm", LENS, 64, 8, seed=303)
    kc, vc, table = _paged_from_contig(c, 16, seed=304)
    kc2, vc2, table2 = _paged_from_contig(c, 16, seed=305)
    assert not torch.equal(table, table2)
    sl = torch.tensor(LENS, dtype=torch.int32).cuda()
    a = sa.sinkattn_decode(c.q.cuda(), kc.cuda(), vc.cuda(), block_table=table.cuda(),
                           seqlens_k=sl, max_seqlen_k=c.max_seqlen_k, sinks=c.sinks.cuda())
    b = sa.sinkattn_decode(c.q.cuda(), kc2.cuda(), vc2.cuda(), block_table=table2.cuda(),
                           seqlens_k=sl, max_seqlen_k=c.max_seqlen_k, sinks=c.sinks.cuda())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("window", [0, 128])
def test_decode_equals_last_prefill_row(window):
    lens = [130, 1000, 4097, 64]
    p = S.make_prefill("pf", lens, lens, 64, 8, seed=306, window=window)
    out_p, lse_p = sa.sinkattn_prefill(p.q.cuda(), p.k.cuda(), p.v.cuda(),
                                       p.cu_seqlens_q.cuda(), p.cu_seqlens_k.cuda(),
                                       p.max_seqlen_q, p.max_seqlen_k, sinks=p.sinks.cuda(),
                                       causal=True, window=window)
    last = (p.cu_seqlens_q[1:] - 1).long()
    q_last = p.q[last].contiguous()
    out_d, lse_d = sa.sinkattn_decode(q_last.cuda(), p.k.cuda(), p.v.cuda(),
                                      kv_indptr=p.cu_seqlens_k.cuda(), max_seqlen_k=max(lens),
                                      sinks=p.sinks.cuda(), window=window)
    check_pair(out_d, lse_d, out_p[last.cuda()], lse_p[last.cuda()],
               "decode vs last prefill row w=%d" % window)


def test_decode_independent_of_split_count():
    c = S.make_decode("ns", LENS, 64, 8, seed=307)
    ref_o, ref_l = _decode_contig(c, 1)
    for ns in (2, 5, 17, 64):
        o, l = _decode_contig(c, ns)
        check_pair(o, l, ref_o, ref_l, "splits %d vs 1" % ns)


def test_repeated_calls_are_bitwise_identical():
    c = S.make_decode("det", LENS, 64, 8, seed=308)
    a = _decode_contig(c, 7)
    b = _decode_contig(c, 7)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    p = S.make_prefill("detp", [300, 1200], [300, 1200], 64, 8, seed=309)
    args = (p.q.cuda(), p.k.cuda(), p.v.cuda(), p.cu_seqlens_q.cuda(), p.cu_seqlens_k.cuda(),
            p.max_seqlen_q, p.max_seqlen_k)
    x = sa.sinkattn_prefill(*args, sinks=p.sinks.cuda())
    y = sa.sinkattn_prefill(*args, sinks=p.sinks.cuda())
    assert torch.equal(x[0], y[0]) and torch.equal(x[1], y[1])


@pytest.mark.parametrize("hq,d", [(8, 64), (6, 64), (4, 128)])
@pytest.mark.parametrize("causal,window", [(False, 0), (False, 100), (True, 0), (True, 50)])
def test_split_prefill_repeats_bitwise(causal, window, hq, d):
    """Split-KV prefill repeated 12 times gives bitwise the same output each
    time (a race between the softmax's O rescaling or epilogue and the P V
    products would show up here as run-to-run differences): two heads per
    item (groups of 4), one head per item in two CTAs per SM (groups of 3)
    and head_dim 128."""
    p = S.make_prefill("dets", [1, 77, 300, 129, 0, 513, 1000],
                       [1, 200, 300, 129, 5, 1000, 1000], hq, 2, seed=3, causal=causal,
                       window=window, head_dim=d)
    args = (p.q.cuda(), p.k.cuda(), p.v.cuda(), p.cu_seqlens_q.cuda(), p.cu_seqlens_k.cuda(),
            p.max_seqlen_q, p.max_seqlen_k)
    ref = None
    for _ in range(12):
        o, l = sa.sinkattn_prefill(*args, sinks=p.sinks.cuda(), causal=causal, window=window,
                                   num_splits=3)
        torch.cuda.synchronize()
        if ref is None:
            ref = (o.clone(), l.clone())
        else:
            assert torch.equal(o, ref[0]) and torch.equal(l, ref[1])


def test_no_device_error_after_the_suite():
    assert sa.sinkattn_get_device_error() == 0


def _off16(like):
    """A tensor shaped like `like` whose data starts 16 bytes past a 32-byte
    boundary (the ABI asks for 16-byte alignment only)."""
    n = like.numel()
    buf = torch.empty(n + 64, dtype=like.dtype, device=like.device)
    base = buf.data_ptr()
    start = ((32 - base % 32) % 32 + 16) // like.element_size()
    t = buf[start:start + n].view(like.shape)
    assert t.data_ptr() % 32 == 16
    return t


def test_outputs_aligned_to_16_bytes_only_match():
    """Outputs on a 16-byte (not 32-byte) boundary take the 16-byte store path
    and give bitwise the same results as 32-byte aligned ones."""
    c = S.make_prefill("al", [1, 300, 129, 513], [1, 500, 129, 1000], 8, 2, seed=41,
                       device="cuda")
    cq, ck, sk = c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda(), c.sinks.cuda()
    for w in (0, 100):
        out, lse = sa.sinkattn_prefill(c.q, c.k, c.v, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                       sinks=sk, window=w)
        o16 = _off16(out)
        sa.sinkattn_prefill(c.q, c.k, c.v, cq, ck, c.max_seqlen_q, c.max_seqlen_k, sinks=sk,
                            window=w, out=o16)
        torch.cuda.synchronize()
        assert torch.equal(out, o16)
        dout = S.bf16_normal(tuple(c.q.shape), 43, device="cuda")
        g = sa.sinkattn_prefill_backward(c.q, c.k, c.v, out, lse, dout, cq, ck, c.max_seqlen_q,
                                         c.max_seqlen_k, sinks=sk, window=w)
        dq16, dk16, dv16 = _off16(g[0]), _off16(g[1]), _off16(g[2])
        g16 = sa.sinkattn_prefill_backward(c.q, c.k, c.v, out, lse, dout, cq, ck,
                                           c.max_seqlen_q, c.max_seqlen_k, sinks=sk, window=w,
                                           dq=dq16, dk=dk16, dv=dv16)
        torch.cuda.synchronize()
        for a, b in zip(g[:3], g16[:3]):
            assert torch.equal(a, b)
        assert torch.equal(g[3], g16[3])
    assert sa.sinkattn_get_device_error() == 0

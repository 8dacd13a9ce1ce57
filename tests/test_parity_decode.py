"""GPU decode (contiguous and paged KV) against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, cuda

pytestmark = pytest.mark.gpu


def run_decode(c, num_splits=0, window=None):
    w = c.window if window is None else window
    if c.paged:
        return sa.sinkattn_decode(c.q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(),
                                  block_table=c.block_table.cuda(),
                                  seqlens_k=c.seqlens_k_t.cuda(), max_seqlen_k=c.max_seqlen_k,
                                  sinks=cuda(c.sinks), window=w, scale=c.scale,
                                  num_splits=num_splits)
    return sa.sinkattn_decode(c.q.cuda(), c.k.cuda(), c.v.cuda(), kv_indptr=c.kv_indptr.cuda(),
                              max_seqlen_k=c.max_seqlen_k, sinks=cuda(c.sinks), window=w,
                              scale=c.scale, num_splits=num_splits)


def oracle_decode(oracle, c, window=None):
    w = c.window if window is None else window
    cu_q = torch.arange(0, c.batch + 1, dtype=torch.int32)
    if c.paged:
        return oracle.attention(c.q, c.k_cache, c.v_cache, cu_q, block_table=c.block_table,
                                seqlens_k=c.seqlens_k_t, hq=c.hq, hkv=c.hkv,
                                head_dim=c.head_dim, sinks=c.sinks, causal=True, window=w,
                                scale=c.scale)
    return oracle.attention(c.q, c.k, c.v, cu_q, c.kv_indptr, hq=c.hq, hkv=c.hkv,
                            head_dim=c.head_dim, sinks=c.sinks, causal=True, window=w,
                            scale=c.scale)


# lengths chosen to span several 32-token slabs, several 512-token blocks and
# ragged tails (1, 31, 33, 127, 129, 511, 513, ...), plus an empty context
LENS = [1, 31, 32, 33, 127, 128, 129, 511, 512, 513, 1000, 1537, 2048, 3001, 0, 77]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (64, 8), (24, 3)])
@pytest.mark.parametrize("window", [0, 1, 100, 600])
def test_decode_contiguous_small(oracle_lib, hq, hkv, window):
    c = S.make_decode("small", LENS, hq, hkv, seed=41 + hq + window, window=window, sink_std=1.5)
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "decode contig hq=%d hkv=%d w=%d" % (hq, hkv, window))


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 40])
def test_decode_split_counts(oracle_lib, num_splits):
    c = S.make_decode("splits", [5000, 4097, 1, 300, 6144], 64, 8, seed=43)
    out, lse = run_decode(c, num_splits=num_splits)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "splits=%d" % num_splits)


def test_decode_without_sinks(oracle_lib):
    c = S.make_decode("nosink", LENS, 32, 4, seed=45, with_sinks=False)
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "no sinks")
    # the empty context gives out = 0 and lse = -inf
    e = LENS.index(0)
    assert torch.all(out[e] == 0) and torch.all(torch.isneginf(lse[e]))


def test_decode_large_sink_and_empty(oracle_lib):
    c = S.make_decode("bigsink", [0, 5, 700], 8, 1, seed=47)
    c.sinks = torch.full((8,), 60.0)
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "large sink")
    assert torch.all(out[0] == 0) and torch.allclose(lse[0].cpu(), torch.full((8,), 60.0))


# Unsplit calls with a visible span of at most 128 tokens run one warp per
# (sequence, KV head); num_splits = 2 forces the four-warp blocks on the same
# inputs. 7 sequences x 3 KV heads = 21 pairs leave three warps of the last
# block without work.
SHORT = [0, 1, 31, 100, 128, 33, 127]


@pytest.mark.parametrize("paged,page_size", [(False, 16), (True, 16), (True, 7)])
@pytest.mark.parametrize("window,d", [(0, 64), (77, 64), (0, 128), (64, 128)])
def test_decode_one_warp_per_pair(oracle_lib, paged, page_size, window, d):
    c = S.make_decode("pair", SHORT, 6, 3, seed=49 + window + d + page_size, window=window,
                      sink_std=1.5, paged=paged, page_size=page_size, head_dim=d)
    ro, rl = oracle_decode(oracle_lib, c)
    for num_splits in (0, 2):
        out, lse = run_decode(c, num_splits=num_splits)
        check_close(out, lse, ro, rl, "pair paged=%s w=%d d=%d splits=%d"
                    % (paged, window, d, num_splits))
    e = SHORT.index(0)
    assert torch.all(out[e] == 0)


@pytest.mark.parametrize("window", [0, 16, 200])
@pytest.mark.parametrize("page_size", [16, 32, 24])
def test_decode_paged_small(oracle_lib, window, page_size):
    c = S.make_decode("paged", LENS, 64, 8, seed=49 + window, window=window, paged=True,
                      page_size=page_size, sink_std=2.0)
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "paged w=%d ps=%d" % (window, page_size))


# head_dim 128: 16-token warp steps, 256-byte rows, 8 output dims per thread
@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("window", [0, 1, 100])
@pytest.mark.parametrize("hq,hkv", [(64, 8), (24, 3)])
def test_decode_head_dim_128(oracle_lib, paged, window, hq, hkv):
    c = S.make_decode("d128", LENS, hq, hkv, seed=161 + window + hq, window=window, paged=paged,
                      page_size=16, sink_std=1.5, head_dim=128)
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "decode d=128 paged=%s w=%d hq=%d" % (paged, window, hq))


@pytest.mark.parametrize("num_splits", [1, 5, 33])
def test_decode_head_dim_128_splits(oracle_lib, num_splits):
    c = S.make_decode("d128s", [5000, 4097, 1, 300, 6144], 64, 8, seed=163, head_dim=128)
    out, lse = run_decode(c, num_splits=num_splits)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "d=128 splits=%d" % num_splits)


def _sample_seqs(batch, k, seed):
    g = torch.Generator().manual_seed(seed)
    return sorted(set([0, batch - 1] + torch.randperm(batch, generator=g)[:k].tolist()))


def test_decode_contig_full_config(oracle_lib):
    """64 sequences, KV lengths uniform in [1024, 8192], 64 q / 8 kv heads:
    every output against the oracle."""
    c = S.decode_contig()
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "decode_contig")


@pytest.mark.parametrize("window", [0, 128])
def test_decode_paged_full_config(oracle_lib, window):
    """256 sequences, contexts uniform in [1024, 32768], 16-token pages with a
    permuted block table: the whole batch on the GPU; against the oracle, every
    sequence (all heads) with the 128-token window and 64 sampled sequences
    (all heads) without it."""
    c = S.paged_decode(window=window, device="cuda")
    out, lse = sa.sinkattn_decode(c.q, c.k_cache, c.v_cache, block_table=c.block_table.cuda(),
                                  seqlens_k=c.seqlens_k_t.cuda(), max_seqlen_k=c.max_seqlen_k,
                                  sinks=c.sinks.cuda(), window=window, scale=c.scale)
    torch.cuda.synchronize()
    seqs = _sample_seqs(c.batch, 62, 51) if window == 0 else list(range(c.batch))
    # compact copy of the sampled sequences' pages for the oracle
    tabs, lens, pages = [], [], []
    at = 0
    for b in seqs:
        n = (c.seqlens_k[b] + 15) // 16
        pages.append(c.block_table[b, :n])
        tabs.append(torch.arange(at, at + n, dtype=torch.int32))
        lens.append(c.seqlens_k[b])
        at += n
    maxp = max(t.numel() for t in tabs)
    table = torch.zeros((len(seqs), maxp), dtype=torch.int32)
    for i, t in enumerate(tabs):
        table[i, :t.numel()] = t
    idx = torch.cat(pages).long().cuda()
    kc = c.k_cache[idx].cpu()
    vc = c.v_cache[idx].cpu()
    q = c.q[seqs].cpu()
    cu_q = torch.arange(0, len(seqs) + 1, dtype=torch.int32)
    ro, rl = oracle_lib.attention(q, kc, vc, cu_q, block_table=table,
                                  seqlens_k=torch.tensor(lens, dtype=torch.int32), hq=64, hkv=8,
                                  head_dim=64, sinks=c.sinks, causal=True, window=window,
                                  scale=c.scale)
    check_close(out[seqs], lse[seqs], ro, rl, "paged_decode w=%d" % window)


# Groups above 8 query heads per KV head: tiles of 8 heads (the last one
# partial for 12 and 24), one block or warp per tile, over contiguous and
# paged caches, automatic and explicit split plans, the one-warp-per-pair
# form (window 100) and head_dim 128.
@pytest.mark.parametrize("hq,hkv", [(16, 1), (64, 4), (12, 1), (24, 1), (64, 1)])
@pytest.mark.parametrize("paged,window", [(False, 0), (True, 0), (False, 100), (True, 100)])
def test_decode_groups_above_eight(oracle_lib, hq, hkv, paged, window):
    c = S.make_decode("bigroup", LENS, hq, hkv, seed=171 + hq + hkv + window, window=window,
                      paged=paged, page_size=16, sink_std=1.5)
    ro, rl = oracle_decode(oracle_lib, c)
    for num_splits in (0, 3):
        out, lse = run_decode(c, num_splits=num_splits)
        check_close(out, lse, ro, rl, "group %d paged=%s w=%d splits=%d"
                    % (hq // hkv, paged, window, num_splits))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_group_sixteen_long_contexts(oracle_lib, d):
    """64 q / 4 kv heads (groups of 16) over long contexts: split plans with
    the last-block merge per (sequence, KV head, head tile)."""
    c = S.make_decode("g16long", [5000, 4097, 1, 300, 6144, 0, 12000], 64, 4, seed=181 + d,
                      head_dim=d)
    out, lse = run_decode(c)
    ro, rl = oracle_decode(oracle_lib, c)
    check_close(out, lse, ro, rl, "group 16 long d=%d" % d)

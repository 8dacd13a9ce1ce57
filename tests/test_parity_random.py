"""Seeded random configurations against the float64 oracle.

Each case draws its own batch, ragged lengths (with the tile edges 0, 1,
127, 128, 129, 255, 256, 257 mixed in), head counts and group size,
head_dim, mask, scale, sink presence and split count, so that combinations
the hand-written cases do not list are exercised too. The seeds are fixed:
a failure names its case and reproduces."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, check_grad, cuda
from oracle import backward as OB

pytestmark = pytest.mark.gpu

EDGES = [0, 1, 127, 128, 129, 255, 256, 257]


def _length(rng, hi):
    return int(rng.choice(EDGES)) if rng.rand() < 0.4 else int(rng.randint(0, hi + 1))


def _heads(rng, max_hq):
    hkv = int(rng.choice([1, 2, 4]))
    groups = [g for g in (1, 2, 3, 4, 8, 16) if hkv * g <= max_hq]
    return hkv * int(rng.choice(groups)), hkv


def _mask(rng):
    causal = bool(rng.rand() < 0.7)
    window = 0 if rng.rand() < 0.5 else int(rng.randint(1, 300))
    return causal, window


def _prefill_case(seed, max_len=400):
    rng = np.random.RandomState(seed)
    d = int(rng.choice([64, 128]))
    hq, hkv = _heads(rng, 16 if d == 128 else 32)
    batch = int(rng.randint(1, 5))
    lq = [_length(rng, max_len) for _ in range(batch)]
    # keys: the queries are the last lq of lk positions; sometimes fewer keys
    lk = [q + (int(rng.randint(0, 300)) if rng.rand() < 0.6 else 0) if rng.rand() < 0.9
          else _length(rng, max_len) for q in lq]
    causal, window = _mask(rng)
    c = S.make_prefill("rand%d" % seed, lq, lk, hq, hkv, seed=seed, causal=causal,
                       window=window, sink_std=float(rng.choice([1.0, 3.0])),
                       with_sinks=bool(rng.rand() < 0.8),
                       scale=None if rng.rand() < 0.5 else float(rng.uniform(0.05, 0.3)),
                       head_dim=d)
    splits = int(rng.choice([0, 0, 1, 2, 3]))
    return c, splits


@pytest.mark.parametrize("seed", list(range(1000, 1040)))
def test_random_prefill(oracle_lib, seed):
    c, splits = _prefill_case(seed)
    out, lse = sa.sinkattn_prefill(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.cu_seqlens_q.cuda(),
                                   c.cu_seqlens_k.cuda(), c.max_seqlen_q, c.max_seqlen_k,
                                   sinks=cuda(c.sinks), causal=c.causal, window=c.window,
                                   scale=c.scale, num_splits=splits)
    ro, rl = oracle_lib.attention(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, hq=c.hq,
                                  hkv=c.hkv, head_dim=c.head_dim, sinks=c.sinks,
                                  causal=c.causal, window=c.window, scale=c.scale)
    check_close(out, lse, ro, rl, "random prefill seed=%d (lq=%s lk=%s hq=%d hkv=%d d=%d "
                "causal=%s w=%d splits=%d)" % (seed, c.seqlens_q, c.seqlens_k, c.hq, c.hkv,
                                                c.head_dim, c.causal, c.window, splits))


@pytest.mark.parametrize("seed", list(range(4000, 4020)))
def test_random_paged_prefill(oracle_lib, seed):
    """Chunked prefill against a paged cache: the queries of sequence b are the
    last lq_b of its lk_b positions."""
    rng = np.random.RandomState(seed)
    d = int(rng.choice([64, 128]))
    hq, hkv = _heads(rng, 16 if d == 128 else 32)
    batch = int(rng.randint(1, 5))
    lq = [_length(rng, 300) for _ in range(batch)]
    lk = [q + int(rng.randint(0, 600)) for q in lq]
    causal, window = _mask(rng)
    c = S.make_prefill_paged("rpaged%d" % seed, lq, lk, hq, hkv, seed=seed, causal=causal,
                             window=window, with_sinks=bool(rng.rand() < 0.8),
                             page_size=int(rng.choice([1, 7, 16, 64])),
                             spare_pages=int(rng.randint(0, 4)), head_dim=d)
    out, lse = sa.sinkattn_prefill_paged(
        c.q.cuda(), c.cu_seqlens_q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(),
        c.block_table.cuda(), c.seqlens_k_t.cuda(), c.max_seqlen_q, c.max_seqlen_k,
        sinks=cuda(c.sinks), causal=c.causal, window=c.window, scale=c.scale)
    ro, rl = oracle_lib.attention(c.q, c.k_cache, c.v_cache, c.cu_seqlens_q,
                                  block_table=c.block_table, seqlens_k=c.seqlens_k_t, hq=hq,
                                  hkv=hkv, head_dim=d, sinks=c.sinks, causal=c.causal,
                                  window=c.window, scale=c.scale)
    check_close(out, lse, ro, rl, "random paged prefill seed=%d (lq=%s lk=%s hq=%d hkv=%d "
                "d=%d causal=%s w=%d page=%d)" % (seed, lq, lk, hq, hkv, d, c.causal, c.window,
                                                   c.page_size))
    assert sa.sinkattn_get_device_error() == 0


@pytest.mark.parametrize("seed", list(range(2000, 2040)))
def test_random_decode(oracle_lib, seed):
    rng = np.random.RandomState(seed)
    d = int(rng.choice([64, 128]))
    hq, hkv = _heads(rng, 64)
    batch = int(rng.randint(1, 13))
    lens = [_length(rng, 3000) for _ in range(batch)]
    window = 0 if rng.rand() < 0.5 else int(rng.randint(1, 600))
    paged = bool(rng.rand() < 0.5)
    page = int(rng.choice([1, 7, 16, 64]))
    c = S.make_decode("rand%d" % seed, lens, hq, hkv, seed=seed, window=window,
                      sink_std=float(rng.choice([1.0, 3.0])), with_sinks=bool(rng.rand() < 0.8),
                      paged=paged, page_size=page,
                      scale=None if rng.rand() < 0.5 else float(rng.uniform(0.05, 0.3)),
                      head_dim=d)
    splits = int(rng.choice([0, 0, 1, 2, 5]))
    mk = max(max(lens), 1)
    if paged:
        out, lse = sa.sinkattn_decode(c.q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(),
                                      block_table=c.block_table.cuda(),
                                      seqlens_k=c.seqlens_k_t.cuda(), max_seqlen_k=mk,
                                      sinks=cuda(c.sinks), window=window, scale=c.scale,
                                      num_splits=splits)
        ro, rl = oracle_lib.attention(c.q, c.k_cache, c.v_cache,
                                      torch.arange(0, batch + 1, dtype=torch.int32),
                                      block_table=c.block_table, seqlens_k=c.seqlens_k_t,
                                      hq=hq, hkv=hkv, head_dim=d, sinks=c.sinks, causal=True,
                                      window=window, scale=c.scale)
    else:
        out, lse = sa.sinkattn_decode(c.q.cuda(), c.k.cuda(), c.v.cuda(),
                                      kv_indptr=c.kv_indptr.cuda(), max_seqlen_k=mk,
                                      sinks=cuda(c.sinks), window=window, scale=c.scale,
                                      num_splits=splits)
        ro, rl = oracle_lib.attention(c.q, c.k, c.v, torch.arange(0, batch + 1, dtype=torch.int32),
                                      c.kv_indptr, hq=hq, hkv=hkv, head_dim=d, sinks=c.sinks,
                                      causal=True, window=window, scale=c.scale)
    check_close(out, lse, ro, rl, "random decode seed=%d (lens=%s hq=%d hkv=%d d=%d w=%d "
                "paged=%s page=%d splits=%d)" % (seed, lens, hq, hkv, d, window, paged, page,
                                                  splits))


@pytest.mark.parametrize("seed", list(range(3000, 3010)))
def test_random_backward(seed):
    c, _ = _prefill_case(seed, max_len=260)
    dout = S.bf16_normal(tuple(c.q.shape), seed + 7)
    args = (c.q.cuda(), c.k.cuda(), c.v.cuda())
    cq, ck = c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda()
    out, lse = sa.sinkattn_prefill(*args, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                   sinks=cuda(c.sinks), causal=c.causal, window=c.window,
                                   scale=c.scale)
    got = sa.sinkattn_prefill_backward(*args, out, lse, dout.cuda(), cq, ck, c.max_seqlen_q,
                                       c.max_seqlen_k, sinks=cuda(c.sinks), causal=c.causal,
                                       window=c.window, scale=c.scale)
    ref = OB.backward(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, dout, hq=c.hq, hkv=c.hkv,
                      sinks=c.sinks, causal=c.causal, window=c.window, scale=c.scale)
    what = "random backward seed=%d (lq=%s lk=%s hq=%d hkv=%d d=%d causal=%s w=%d)" % (
        seed, c.seqlens_q, c.seqlens_k, c.hq, c.hkv, c.head_dim, c.causal, c.window)
    for g, r, name in zip(got[:3], ref[:3], ("dq", "dk", "dv")):
        check_grad(g, r, what + " " + name)
    if ref[3] is None:
        assert got[3] is None
    else:
        check_grad(got[3], ref[3], what + " dsinks", dense=True)
    assert sa.sinkattn_get_device_error() == 0

"""GPU prefill (packed variable-length sequences) against the float64 oracle."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, cuda

pytestmark = pytest.mark.gpu


def run_prefill(c, device_tensors=False, num_splits=0):
    t = (lambda x: x) if device_tensors else cuda
    return sa.sinkattn_prefill(t(c.q), t(c.k), t(c.v), c.cu_seqlens_q.cuda(),
                               c.cu_seqlens_k.cuda(), c.max_seqlen_q, c.max_seqlen_k,
                               sinks=cuda(c.sinks), causal=c.causal, window=c.window,
                               scale=c.scale, num_splits=num_splits)


def oracle_prefill(oracle, c):
    return oracle.attention(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, hq=c.hq, hkv=c.hkv,
                            head_dim=c.head_dim, sinks=c.sinks, causal=c.causal, window=c.window,
                            scale=c.scale)


def test_prefill_tiny_config(oracle_lib):
    """1 sequence of 64 tokens, causal, 4 q heads sharing 1 KV head, scale 1/8."""
    c = S.tiny_prefill()
    out, lse = run_prefill(c)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "tiny_prefill")


# q/k lengths that span several 128-row tiles with ragged tails, chunked
# queries (lq < lk), more queries than keys, and empty sequences
SHAPES = [
    ([1], [1]),
    ([127], [127]),
    ([128], [128]),
    ([129], [129]),
    ([300, 17, 256, 1], [300, 17, 256, 1]),
    ([200], [700]),          # chunked: queries are the last 200 of 700 positions
    ([130], [40]),           # more queries than keys: first 90 see nothing
    ([0, 64, 0], [0, 64, 5]),
    ([513], [513]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 1), (True, 128),
                                           (True, 129), (False, 50)])
def test_prefill_shapes(oracle_lib, shape, causal, window):
    lq, lk = shape
    c = S.make_prefill("shape", lq, lk, 8, 2, seed=61 + sum(lq), causal=causal, window=window,
                       sink_std=1.5)
    out, lse = run_prefill(c)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "prefill %s causal=%s w=%d" % (shape, causal, window))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (12, 3), (64, 8)])
def test_prefill_groups_and_no_sink(oracle_lib, hq, hkv):
    for with_sinks in (True, False):
        c = S.make_prefill("grp", [190, 260], [190, 260], hq, hkv, seed=67 + hq,
                           with_sinks=with_sinks)
        out, lse = run_prefill(c)
        ro, rl = oracle_prefill(oracle_lib, c)
        check_close(out, lse, ro, rl, "hq=%d hkv=%d sinks=%s" % (hq, hkv, with_sinks))


def test_prefill_keyless_tiles_between_others(oracle_lib):
    """Many sequences whose first query tiles see no key (more queries than keys,
    causal) mixed with long ones: the persistent grid then meets tiles without
    keys between tiles with keys on the same CTA."""
    lq = [400] * 20 + [1000] * 20
    lk = [100] * 20 + [2000] * 20
    c = S.make_prefill("keyless", lq, lk, 8, 2, seed=75)
    out, lse = run_prefill(c)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "keyless tiles")


def test_prefill_large_sink(oracle_lib):
    c = S.make_prefill("bigsink", [300], [300], 4, 1, seed=69)
    c.sinks = torch.tensor([40.0, -40.0, 0.0, 12.0])
    out, lse = run_prefill(c)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "large sink")


# split-KV: every (query tile, heads) item cut into n key ranges, merged by
# log-sum-exp, the sink counted in the first range only
SPLIT_SHAPES = [
    ([129], [129]),
    ([200], [1500]),
    ([300, 17, 256, 1], [300, 900, 256, 40]),
    ([130], [40]),
    ([0, 64, 0], [0, 64, 5]),
]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[str(i) for i in range(len(SPLIT_SHAPES))])
@pytest.mark.parametrize("num_splits", [2, 3, 7, 64])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 200)])
def test_prefill_explicit_splits(oracle_lib, shape, num_splits, causal, window):
    lq, lk = shape
    c = S.make_prefill("split", lq, lk, 8, 2, seed=101 + sum(lk) + num_splits, causal=causal,
                       window=window, sink_std=1.5)
    out, lse = run_prefill(c, num_splits=num_splits)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "prefill %s splits=%d causal=%s w=%d"
                % (shape, num_splits, causal, window))


@pytest.mark.parametrize("with_sinks", [True, False])
def test_prefill_splits_sink_counted_once(oracle_lib, with_sinks):
    """Large sinks make a double-counted (or dropped) sink visible at once."""
    c = S.make_prefill("split_sink", [300], [2000], 4, 1, seed=103, with_sinks=with_sinks)
    if with_sinks:
        c.sinks = torch.tensor([9.0, -30.0, 0.0, 4.0])
    out, lse = run_prefill(c, num_splits=5)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "split sink once (sinks=%s)" % with_sinks)


def test_prefill_splits_odd_group(oracle_lib):
    """Groups of 3 query heads per KV head run one head per item."""
    c = S.make_prefill("split_odd", [250, 90], [1300, 600], 12, 4, seed=105)
    out, lse = run_prefill(c, num_splits=6)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "split odd group")


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
    """One random row of every (sequence, 128-row query tile, query head) in
    the call, plus every head of each sequence's first and last row: every
    work item the kernel schedules (a tile and its heads) is checked, ragged
    last tiles included."""
    g = torch.Generator().manual_seed(seed)
    rows = []
    for b, lq in enumerate(c.seqlens_q):
        for qt in range((lq + 127) // 128):
            n = min(128, lq - qt * 128)
            pick = torch.randint(0, n, (c.hq,), generator=g).tolist()
            rows += [(b, h, qt * 128 + i) for h, i in enumerate(pick)]
        if lq > 0:
            rows += [(b, h, i) for i in sorted({0, lq - 1}) for h in range(c.hq)]
    return np.array(sorted(set(rows)), dtype=np.int32)


def _check_rows(oracle, c, out, lse, rows, what):
    ro, rl = oracle.attention_rows(rows, c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, hq=c.hq,
                                   hkv=c.hkv, head_dim=c.head_dim, sinks=c.sinks, causal=c.causal,
                                   window=c.window, scale=c.scale)
    cu = c.cu_seqlens_q.tolist()
    pr = torch.tensor([cu[b] + i for b, _, i in rows], device=out.device)
    ph = torch.tensor([h for _, h, _ in rows], device=out.device)
    check_close(out[pr, ph], lse[pr, ph], ro, rl, what)


@pytest.mark.parametrize("window", [0, 128])
def test_prefill_varlen_full_config(oracle_lib, window):
    """16 sequences, lengths uniform in [512, 4096], 64 q / 8 kv heads, causal;
    full and sliding window 128. Every output row and head against the
    oracle."""
    c = S.varlen_prefill(window=window)
    out, lse = run_prefill(c)
    torch.cuda.synchronize()
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "varlen_prefill w=%d (every row)" % window)
    assert sa.sinkattn_get_device_error() == 0


def test_prefill_long_context_auto_splits(oracle_lib):
    """256 queries at the end of a 131072-token context: too few query tiles to
    fill the SMs, so the automatic plan splits the keys. Sampled rows against
    the oracle, and the whole output against the unsplit call."""
    c = S.long_context_prefill()
    ws_auto = sa.sinkattn_prefill_workspace_size(1, 256, 131072, 256, 131072, 64, 8)
    ws_one = sa.sinkattn_prefill_workspace_size(1, 256, 131072, 256, 131072, 64, 8,
                                                num_splits=1)
    assert ws_auto > ws_one  # the plan did split
    q, k, v = c.q.cuda(), c.k.cuda(), c.v.cuda()
    args = (q, k, v, c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda(), 256, 131072)
    out, lse = sa.sinkattn_prefill(*args, sinks=c.sinks.cuda())
    torch.cuda.synchronize()
    _check_rows(oracle_lib, c, out, lse, _sample_rows(c, 60, 107), "long_context_prefill")
    o1, l1 = sa.sinkattn_prefill(*args, sinks=c.sinks.cuda(), num_splits=1)
    # both are within the oracle's tolerance; between them, bf16 rounding only
    d = (out.float() - o1.float()).abs()
    assert float(d.max()) <= 2e-2
    assert float(d.sum() / o1.float().abs().sum()) <= 2e-3
    assert float((lse - l1).abs().max()) <= 1e-3


def test_prefill_chunked_full_config(oracle_lib):
    """4096 query tokens at positions 126976..131071 of a 131072-token causal
    context. One row of every (query tile, head) item, and sampled rows,
    against the oracle."""
    c = S.chunked_prefill()
    out, lse = run_prefill(c)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, c, out, lse, _every_item_rows(c, 72), "chunked_prefill items")
    _check_rows(oracle_lib, c, out, lse, _sample_rows(c, 40, 73), "chunked_prefill")


# head_dim 128: one head per item, two 64-dim blocks per tile, a two-stage
# K/V ring, O in 128 TMEM columns
D128_MASKS = [(True, 0), (False, 0), (True, 1), (True, 128), (False, 50)]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("causal,window", D128_MASKS)
def test_prefill_head_dim_128_shapes(oracle_lib, shape, causal, window):
    lq, lk = shape
    c = S.make_prefill("d128", lq, lk, 8, 2, seed=131 + sum(lq), causal=causal, window=window,
                       sink_std=1.5, head_dim=128)
    out, lse = run_prefill(c)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "d128 %s causal=%s w=%d" % (shape, causal, window))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (12, 3), (64, 8)])
def test_prefill_head_dim_128_groups_and_no_sink(oracle_lib, hq, hkv):
    for with_sinks in (True, False):
        c = S.make_prefill("d128grp", [190, 260], [300, 260], hq, hkv, seed=133 + hq,
                           with_sinks=with_sinks, head_dim=128)
        out, lse = run_prefill(c)
        ro, rl = oracle_prefill(oracle_lib, c)
        check_close(out, lse, ro, rl, "d128 hq=%d hkv=%d sinks=%s" % (hq, hkv, with_sinks))


def test_prefill_head_dim_128_keyless_and_large_sink(oracle_lib):
    c = S.make_prefill("d128kl", [400] * 6 + [700] * 6, [100] * 6 + [900] * 6, 4, 1, seed=135,
                       head_dim=128)
    c.sinks = torch.tensor([30.0, -30.0, 0.0, 9.0])
    out, lse = run_prefill(c)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "d128 keyless tiles, large sinks")


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[str(i) for i in range(len(SPLIT_SHAPES))])
@pytest.mark.parametrize("num_splits", [2, 7])
def test_prefill_head_dim_128_splits(oracle_lib, shape, num_splits):
    lq, lk = shape
    c = S.make_prefill("d128split", lq, lk, 8, 2, seed=137 + sum(lk) + num_splits,
                       sink_std=1.5, head_dim=128)
    out, lse = run_prefill(c, num_splits=num_splits)
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out, lse, ro, rl, "d128 %s splits=%d" % (shape, num_splits))


def test_prefill_head_dim_128_varlen_full_config(oracle_lib):
    """varlen_prefill's lengths and heads at head_dim 128. One row of every
    (query tile, head) item, and sampled rows, against the oracle."""
    c = S.varlen_prefill_d128()
    out, lse = run_prefill(c)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, c, out, lse, _every_item_rows(c, 138), "varlen_prefill_d128 items")
    _check_rows(oracle_lib, c, out, lse, _sample_rows(c, 16, 139), "varlen_prefill_d128")
    assert sa.sinkattn_get_device_error() == 0


def test_prefill_groups_of_three_full_config(oracle_lib):
    """varlen_prefill's lengths with 24 q / 8 kv heads: one head per work
    item, two CTAs per SM. One row of every (query tile, head) item, and
    sampled rows, against the oracle."""
    c = S.varlen_prefill_g3()
    out, lse = run_prefill(c)
    torch.cuda.synchronize()
    _check_rows(oracle_lib, c, out, lse, _every_item_rows(c, 176), "varlen_prefill_g3 items")
    _check_rows(oracle_lib, c, out, lse, _sample_rows(c, 16, 177), "varlen_prefill_g3")
    assert sa.sinkattn_get_device_error() == 0


def test_prefill_length_above_bound_is_reported(oracle_lib):
    """A query length above the host's max_seqlen_q: that sequence's tiles past
    the bound are dropped and the device error word records code 3; the other
    sequences are unaffected."""
    c = S.make_prefill("bound", [300, 100], [300, 100], 8, 2, seed=93)
    assert sa.sinkattn_get_device_error() == 0
    out, lse = sa.sinkattn_prefill(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.cu_seqlens_q.cuda(),
                                   c.cu_seqlens_k.cuda(), 200, c.max_seqlen_k,
                                   sinks=cuda(c.sinks))
    assert sa.sinkattn_get_device_error() == 3
    ro, rl = oracle_prefill(oracle_lib, c)
    check_close(out[:256], lse[:256], ro[:256], rl[:256], "rows within the bound")
    check_close(out[300:], lse[300:], ro[300:], rl[300:], "the other sequence")
    out, lse = run_prefill(c)
    assert sa.sinkattn_get_device_error() == 0

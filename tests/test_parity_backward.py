"""GPU backward of sink-attention prefill against the float64 oracle.

The GPU forward supplies out and lse (as a training step would); the oracle
differentiates the exact definition at the same bf16 inputs."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_grad, cuda
from oracle import backward as OB

pytestmark = pytest.mark.gpu


def run(c, dout):
    args = (c.q.cuda(), c.k.cuda(), c.v.cuda())
    cq, ck = c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda()
    out, lse = sa.sinkattn_prefill(*args, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                   sinks=cuda(c.sinks), causal=c.causal, window=c.window,
                                   scale=c.scale)
    return sa.sinkattn_prefill_backward(*args, out, lse, dout.cuda(), cq, ck, c.max_seqlen_q,
                                        c.max_seqlen_k, sinks=cuda(c.sinks), causal=c.causal,
                                        window=c.window, scale=c.scale)


def reference(c, dout, seqs=None):
    return OB.backward(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, dout, hq=c.hq, hkv=c.hkv,
                       sinks=c.sinks, causal=c.causal, window=c.window, scale=c.scale,
                       seqs=seqs)


def compare(c, got, ref, what, rows_q=None, rows_k=None):
    dq, dk, dv, ds = got
    rq, rk, rv, rs = ref
    sel_q = slice(None) if rows_q is None else rows_q
    sel_k = slice(None) if rows_k is None else rows_k
    check_grad(dq[sel_q], rq[sel_q], what + " dq")
    check_grad(dk[sel_k], rk[sel_k], what + " dk")
    check_grad(dv[sel_k], rv[sel_k], what + " dv")
    if rs is None:
        assert ds is None
    else:
        check_grad(ds, rs, what + " dsinks", dense=True)


def dout_for(c, seed):
    return S.bf16_normal(tuple(c.q.shape), seed)


SHAPES = [
    ([1], [1]),
    ([64], [64]),
    ([129], [129]),
    ([300, 17, 256, 1], [300, 17, 256, 1]),
    ([200], [700]),          # chunked: queries are the last 200 of 700 positions
    ([130], [40]),           # more queries than keys: the first 90 see nothing
    ([0, 64, 0], [0, 64, 5]),
    ([513], [513]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 1), (True, 128),
                                           (False, 50)])
def test_backward_shapes(shape, causal, window):
    lq, lk = shape
    c = S.make_prefill("bwd", lq, lk, 8, 2, seed=121 + sum(lk), causal=causal, window=window,
                       sink_std=1.5)
    dout = dout_for(c, 7 + sum(lq))
    compare(c, run(c, dout), reference(c, dout), "bwd %s causal=%s w=%d" % (shape, causal, window))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (12, 3), (64, 8)])
def test_backward_groups_and_no_sink(hq, hkv):
    for with_sinks in (True, False):
        c = S.make_prefill("bgrp", [190, 260], [390, 260], hq, hkv, seed=123 + hq,
                           with_sinks=with_sinks)
        dout = dout_for(c, 11 + hq)
        compare(c, run(c, dout), reference(c, dout), "bwd hq=%d hkv=%d sinks=%s"
                % (hq, hkv, with_sinks))


def test_backward_large_sinks():
    c = S.make_prefill("bsink", [300], [300], 4, 1, seed=125)
    c.sinks = torch.tensor([9.0, -30.0, 0.0, 4.0])
    dout = dout_for(c, 13)
    compare(c, run(c, dout), reference(c, dout), "bwd large sinks")


def test_backward_repeated_calls_bitwise_identical():
    c = S.make_prefill("bdet", [700, 300], [900, 300], 16, 2, seed=127)
    dout = dout_for(c, 17)
    a = run(c, dout)
    b = run(c, dout)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("d,causal,window", [(64, True, 0), (64, False, 100), (64, True, 50),
                                             (128, True, 0), (128, False, 0)])
def test_backward_repeats_bitwise(d, causal, window):
    """Ten backward calls on the same inputs are bitwise identical (a race
    between the asynchronous lse / D copies, the deferred dQ epilogue and the
    tensor-core products would show as run-to-run differences)."""
    c = S.make_prefill("brep", [1, 77, 300, 129, 0, 513], [1, 200, 300, 129, 5, 700], 8, 2,
                       seed=131, causal=causal, window=window, head_dim=d)
    dout = dout_for(c, 19).cuda()
    args = (c.q.cuda(), c.k.cuda(), c.v.cuda())
    cq, ck = c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda()
    out, lse = sa.sinkattn_prefill(*args, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                   sinks=cuda(c.sinks), causal=causal, window=window)
    ref = None
    for _ in range(10):
        g = sa.sinkattn_prefill_backward(*args, out, lse, dout, cq, ck, c.max_seqlen_q,
                                         c.max_seqlen_k, sinks=cuda(c.sinks), causal=causal,
                                         window=window)
        torch.cuda.synchronize()
        g = [x.clone() for x in g]
        if ref is None:
            ref = g
        else:
            for x, y in zip(g, ref):
                assert torch.equal(x, y)


@pytest.mark.parametrize("window", [0, 128])
def test_backward_varlen_full_config(window):
    """16 sequences, lengths uniform in [512, 4096], 64 q / 8 kv heads, causal:
    the whole batch on the GPU; the first and the last sequence (every head,
    every row) against the oracle."""
    c = S.varlen_prefill(window=window)
    dout = dout_for(c, 19)
    got = run(c, dout)
    torch.cuda.synchronize()
    seqs = [0, c.batch - 1]
    ref = reference(c, dout, seqs=seqs)
    cq, ck = c.cu_seqlens_q.tolist(), c.cu_seqlens_k.tolist()
    rq = np.concatenate([np.arange(cq[b], cq[b + 1]) for b in seqs])
    rk = np.concatenate([np.arange(ck[b], ck[b + 1]) for b in seqs])
    # dsinks sums over every sequence: the oracle's partial sum covers two
    got = got[:3] + (None,)
    ref = ref[:3] + (None,)
    compare(c, got, ref, "bwd varlen w=%d" % window, rows_q=rq, rows_k=rk)


# head_dim 128: items carry a 64-dim half of the output gradient; S and dP
# run over both 64-dim swizzle blocks
@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 1), (True, 128)])
def test_backward_head_dim_128_shapes(shape, causal, window):
    lq, lk = shape
    c = S.make_prefill("bwd128", lq, lk, 8, 2, seed=151 + sum(lk), causal=causal, window=window,
                       sink_std=1.5, head_dim=128)
    dout = dout_for(c, 29 + sum(lq))
    compare(c, run(c, dout), reference(c, dout),
            "bwd d128 %s causal=%s w=%d" % (shape, causal, window))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (12, 3), (16, 2)])
def test_backward_head_dim_128_groups_and_no_sink(hq, hkv):
    for with_sinks in (True, False):
        c = S.make_prefill("bgrp128", [190, 260], [390, 260], hq, hkv, seed=153 + hq,
                           with_sinks=with_sinks, head_dim=128)
        dout = dout_for(c, 31 + hq)
        compare(c, run(c, dout), reference(c, dout), "bwd d128 hq=%d hkv=%d sinks=%s"
                % (hq, hkv, with_sinks))


def test_backward_head_dim_128_large_sinks_and_repeat():
    c = S.make_prefill("bsink128", [300, 700], [300, 900], 4, 1, seed=155, head_dim=128)
    c.sinks = torch.tensor([9.0, -30.0, 0.0, 4.0])
    dout = dout_for(c, 33)
    a = run(c, dout)
    compare(c, a, reference(c, dout), "bwd d128 large sinks")
    b = run(c, dout)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_head_dim_128_varlen_full_config():
    """varlen_prefill's lengths and heads at head_dim 128: the whole batch on
    the GPU; the first and the last sequence (every head, every row) against
    the oracle."""
    c = S.varlen_prefill_d128()
    dout = dout_for(c, 35)
    got = run(c, dout)
    torch.cuda.synchronize()
    seqs = [0, c.batch - 1]
    ref = reference(c, dout, seqs=seqs)
    cq, ck = c.cu_seqlens_q.tolist(), c.cu_seqlens_k.tolist()
    rq = np.concatenate([np.arange(cq[b], cq[b + 1]) for b in seqs])
    rk = np.concatenate([np.arange(ck[b], ck[b + 1]) for b in seqs])
    compare(c, got[:3] + (None,), ref[:3] + (None,), "bwd varlen d128", rows_q=rq, rows_k=rk)


def test_no_device_error_after_backward():
    assert sa.sinkattn_get_device_error() == 0


def test_backward_key_length_above_bound_is_reported():
    """A key length above the host's max_seqlen_k: the key-tile list is cut to
    the bound and the device error word records code 3; dq, whose kernel walks
    every key of its sequence, still matches the oracle."""
    c = S.make_prefill("bbound", [300, 64], [300, 64], 8, 2, seed=95)
    dout = S.bf16_normal(tuple(c.q.shape), 96)
    args = (c.q.cuda(), c.k.cuda(), c.v.cuda())
    cq, ck = c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda()
    out, lse = sa.sinkattn_prefill(*args, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                   sinks=cuda(c.sinks), scale=c.scale)
    assert sa.sinkattn_get_device_error() == 0
    dq, dk, dv, ds = sa.sinkattn_prefill_backward(*args, out, lse, dout.cuda(), cq, ck,
                                                  c.max_seqlen_q, 200, sinks=cuda(c.sinks),
                                                  scale=c.scale)
    assert sa.sinkattn_get_device_error() == 3
    rq = reference(c, dout)[0]
    check_grad(dq, rq, "dq with a short key bound")

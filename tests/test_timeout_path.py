"""The bounded-wait timeout path of the tcgen05 kernels, exercised on purpose.

Every mbarrier wait in the prefill and backward kernels is bounded: one that
runs out records code 1 in the device error word, and the CTA then stops
issuing work, waits (with the normal one-second bound) for the copies and
products it already issued, frees its tensor memory and exits. The testing
hook sinkattn_debug_stall_waits makes each CTA wait, before its first scores,
on a barrier that nothing completes, bounded by 2 ms, so the call takes that
path while copies and products are in flight; nothing faults and no wait is
unbounded. The test then turns the hook off and checks that the very next call
is correct again (against the oracle) with a clean error word.
"""
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, check_grad

pytestmark = pytest.mark.gpu

STALL_NS = 2_000_000


def _prefill(c):
    return sa.sinkattn_prefill(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.cu_seqlens_q.cuda(),
                               c.cu_seqlens_k.cuda(), c.max_seqlen_q, c.max_seqlen_k,
                               sinks=c.sinks.cuda(), causal=c.causal, window=c.window,
                               scale=c.scale)


def _run_with_short_waits(fn):
    """fn() with the stall hook on; returns the device error code."""
    torch.cuda.synchronize()
    assert sa.sinkattn_get_device_error() == 0
    sa.sinkattn_debug_stall_waits(STALL_NS)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        sa.sinkattn_debug_stall_waits(0)
    return sa.sinkattn_get_device_error()


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (3, 1, 64), (4, 1, 128)],
                         ids=["two_heads_per_item", "one_head_dual", "head_dim_128"])
def test_prefill_timeout_path_then_recovers(oracle_lib, hq, hkv, d):
    c = S.make_prefill("timeout", [300, 200], [300, 700], hq, hkv, seed=211, head_dim=d)
    assert _run_with_short_waits(lambda: _prefill(c)) == 1
    out, lse = _prefill(c)
    ro, rl = oracle_lib.attention(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, hq=c.hq,
                                  hkv=c.hkv, head_dim=c.head_dim, sinks=c.sinks,
                                  causal=c.causal, window=c.window, scale=c.scale)
    check_close(out, lse, ro, rl, "prefill after a timed-out call")
    assert sa.sinkattn_get_device_error() == 0


def test_backward_timeout_path_then_recovers():
    from oracle import backward as OB
    c = S.make_prefill("timeout_bwd", [300, 200], [300, 700], 8, 2, seed=213)
    out, lse = _prefill(c)
    dout = S.bf16_normal(tuple(c.q.shape), 214)
    args = (c.q.cuda(), c.k.cuda(), c.v.cuda(), out, lse, dout.cuda(), c.cu_seqlens_q.cuda(),
            c.cu_seqlens_k.cuda(), c.max_seqlen_q, c.max_seqlen_k)
    kw = dict(sinks=c.sinks.cuda(), causal=c.causal, window=c.window, scale=c.scale)
    assert _run_with_short_waits(lambda: sa.sinkattn_prefill_backward(*args, **kw)) == 1
    dq, dk, dv, ds = sa.sinkattn_prefill_backward(*args, **kw)
    rq, rk, rv, rs = OB.backward(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, dout, hq=c.hq,
                                 hkv=c.hkv, sinks=c.sinks, causal=c.causal, window=c.window,
                                 scale=c.scale)
    check_grad(dq, rq, "dq after a timed-out call")
    check_grad(dk, rk, "dk after a timed-out call")
    check_grad(dv, rv, "dv after a timed-out call")
    check_grad(ds, rs, "dsinks after a timed-out call", dense=True)
    assert sa.sinkattn_get_device_error() == 0

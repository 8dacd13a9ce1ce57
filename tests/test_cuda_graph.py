"""Every call only enqueues work on the caller's stream, so it can be captured
in a CUDA graph: replays give bitwise the results of the eager calls.

Decode with a split plan exercises the counter-zeroing kernel and the
programmatic dependent launch of the decode grid inside a graph, and that the
merge counters are back at zero after every replay."""
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm up on a side stream (as torch requires), then capture fn()."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _replay_matches(g, outs, refs, reps=4):
    for _ in range(reps):
        for o in outs:
            o.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            assert torch.equal(o, r)


@pytest.mark.parametrize("paged,fp8", [(False, False), (True, False), (False, True),
                                       (True, True)])
def test_decode_graph_replay(paged, fp8):
    c = S.make_decode("graph", [5000, 1, 3000, 8192, 77], 64, 8, seed=171, paged=paged,
                      kv_dtype="fp8" if fp8 else "bf16", device="cuda")
    out = torch.empty_like(c.q)
    lse = torch.empty((c.batch, c.hq), dtype=torch.float32, device="cuda")
    ws = torch.empty(sa.sinkattn_decode_workspace_size(c.batch, c.max_seqlen_k, c.hq, c.hkv),
                     dtype=torch.uint8, device="cuda")
    kv = (dict(block_table=c.block_table.cuda(), seqlens_k=c.seqlens_k_t.cuda())
          if paged else dict(kv_indptr=c.kv_indptr.cuda()))
    k, v = (c.k_cache, c.v_cache) if paged else (c.k, c.v)
    sk = c.sinks.cuda()
    extra = dict(k_scale=c.k_scale.cuda(), v_scale=c.v_scale.cuda()) if fp8 else {}
    f = sa.sinkattn_decode_fp8 if fp8 else sa.sinkattn_decode

    def call():
        f(c.q, k, v, max_seqlen_k=c.max_seqlen_k, sinks=sk, out=out, lse=lse, workspace=ws,
          **kv, **extra)

    call()
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    g = _capture(call)
    _replay_matches(g, [out, lse], [ref_o, ref_l])
    # eager again after the replays: the counters were left at zero
    out.fill_(0)
    call()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o)


def test_prefill_and_backward_graph_replay():
    c = S.make_prefill("graph_pf", [300, 17, 900], [300, 400, 900], 16, 2, seed=173,
                       device="cuda")
    cq, ck, sk = c.cu_seqlens_q.cuda(), c.cu_seqlens_k.cuda(), c.sinks.cuda()
    out = torch.empty_like(c.q)
    lse = torch.empty((c.q.shape[0], c.hq), dtype=torch.float32, device="cuda")
    ws = torch.empty(sa.sinkattn_prefill_workspace_size(c.batch, c.q.shape[0], c.k.shape[0],
                                                        c.max_seqlen_q, c.max_seqlen_k, c.hq,
                                                        c.hkv, num_splits=3),
                     dtype=torch.uint8, device="cuda")
    dout = S.bf16_normal(tuple(c.q.shape), 175, device="cuda")
    dq, dk, dv = torch.empty_like(c.q), torch.empty_like(c.k), torch.empty_like(c.v)
    dsk = torch.empty_like(sk)
    bws = torch.empty(sa.sinkattn_prefill_backward_workspace_size(
        c.batch, c.q.shape[0], c.k.shape[0], c.hq, c.hkv), dtype=torch.uint8, device="cuda")
    lib = sa.load()

    def call():
        sa.sinkattn_prefill(c.q, c.k, c.v, cq, ck, c.max_seqlen_q, c.max_seqlen_k, sinks=sk,
                            num_splits=3, out=out, lse=lse, workspace=ws)
        sa.sinkattn_prefill_backward(c.q, c.k, c.v, out, lse, dout, cq, ck, c.max_seqlen_q,
                                     c.max_seqlen_k, sinks=sk, dq=dq, dk=dk, dv=dv,
                                     dsinks=dsk, workspace=bws)

    call()
    torch.cuda.synchronize()
    refs = [t.clone() for t in (out, lse, dq, dk, dv, dsk)]
    g = _capture(call)
    _replay_matches(g, [out, lse, dq, dk, dv, dsk], refs)
    assert lib is not None and sa.sinkattn_get_device_error() == 0

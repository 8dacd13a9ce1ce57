"""Pins of the float64 backward oracle (oracle/backward.py), on the CPU.

- Its forward equals the C oracle's forward on bf16 inputs.
- Its gradients equal central finite differences of its forward, for every
  coordinate of q, k, v and the sinks, on tiny problems (causal, windowed and
  unmasked; with and without sinks; rows that see no key).
- Without sinks its gradients equal torch autograd through the library's
  float64 scaled-dot-product attention.
- Plausible mistakes planted in its source make one of these pins fail.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as OB

# (query lengths, key lengths, hq, hkv, d, causal, window, with sinks)
TINY = [
    ([3, 4], [5, 4], 4, 2, 8, True, 0, True),
    ([3, 4], [5, 4], 4, 2, 8, True, 0, False),
    ([5], [5], 2, 1, 4, False, 0, True),
    ([4, 2], [6, 2], 3, 3, 4, True, 3, True),
    ([3], [1], 2, 2, 4, True, 0, True),     # more queries than keys: empty rows
    ([3], [1], 2, 2, 4, True, 0, False),    # empty rows without sink: all-zero rows
]


def _case(spec, seed):
    lq, lk, hq, hkv, d, causal, window, with_sinks = spec
    g = np.random.default_rng(seed)
    tq, tk = sum(lq), sum(lk)
    q = g.standard_normal((tq, hq, d))
    k = g.standard_normal((tk, hkv, d))
    v = g.standard_normal((tk, hkv, d))
    do = g.standard_normal((tq, hq, d))
    sinks = g.standard_normal(hq) if with_sinks else None
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    kw = dict(hq=hq, hkv=hkv, causal=causal, window=window, scale=0.7)
    return q, k, v, do, sinks, cq, ck, kw


def _loss(mod, q, k, v, do, sinks, cq, ck, kw):
    out, _ = mod.forward(q, k, v, cq, ck, sinks=sinks, **kw)
    return float((out * do).sum())


def _fd_grad(mod, x, f, h=1e-5):
    g = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


def check_fd(mod, spec, seed=0):
    q, k, v, do, sinks, cq, ck, kw = _case(spec, seed)
    f = lambda: _loss(mod, q, k, v, do, sinks, cq, ck, kw)
    dq, dk, dv, ds = mod.backward(q, k, v, cq, ck, do, sinks=sinks, **kw)
    for name, x, got in (("dq", q, dq), ("dk", k, dk), ("dv", v, dv)):
        want = _fd_grad(mod, x, f)
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7), name
    if sinks is None:
        assert ds is None
    else:
        want = _fd_grad(mod, sinks, f)
        assert np.allclose(ds, want, rtol=1e-6, atol=1e-7), "dsinks"


@pytest.mark.parametrize("spec", TINY, ids=[str(i) for i in range(len(TINY))])
def test_backward_matches_finite_differences(spec):
    check_fd(OB, spec)


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 5)])
def test_forward_matches_c_oracle(oracle_lib, causal, window):
    from attention_learned_sinks_gb300 import synthetic as S
    for with_sinks in (True, False):
        c = S.make_prefill("fwd", [7, 0, 20, 3], [9, 4, 20, 1], 8, 2, seed=31,
                           causal=causal, window=window, with_sinks=with_sinks)
        ro, rl = oracle_lib.attention(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, hq=8,
                                      hkv=2, head_dim=64, sinks=c.sinks, causal=causal,
                                      window=window, scale=c.scale)
        o, l = OB.forward(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, hq=8, hkv=2,
                          sinks=c.sinks, causal=causal, window=window, scale=c.scale)
        assert np.allclose(o, ro, rtol=0, atol=1e-12)
        fin = np.isfinite(rl)
        assert np.array_equal(fin, np.isfinite(l))
        assert np.allclose(l[fin], rl[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_without_sinks_is_sdpa_autograd(causal):
    """No sink: plain attention, whose gradients torch's float64 SDPA gives."""
    g = np.random.default_rng(5)
    lq, lk, hq, hkv, d = 6, 9, 4, 2, 8
    q = g.standard_normal((lq, hq, d))
    k = g.standard_normal((lk, hkv, d))
    v = g.standard_normal((lk, hkv, d))
    do = g.standard_normal((lq, hq, d))
    cq, ck = np.array([0, lq]), np.array([0, lk])
    dq, dk, dv, _ = OB.backward(q, k, v, cq, ck, do, hq=hq, hkv=hkv, causal=causal, scale=0.3)
    tq = torch.tensor(q).transpose(0, 1).requires_grad_()
    tk = torch.tensor(k).transpose(0, 1).requires_grad_()
    tv = torch.tensor(v).transpose(0, 1).requires_grad_()
    kk = tk.repeat_interleave(hq // hkv, dim=0)
    vv = tv.repeat_interleave(hq // hkv, dim=0)
    mask = None
    if causal:  # bottom-right alignment: query i sits at position lk - lq + i
        mask = torch.tensor(np.arange(lk)[None, :] <= (lk - lq) + np.arange(lq)[:, None])
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=mask, scale=0.3)
    out.backward(torch.tensor(do).transpose(0, 1))
    assert np.allclose(dq, tq.grad.transpose(0, 1).numpy(), atol=1e-12)
    assert np.allclose(dk, tk.grad.transpose(0, 1).numpy(), atol=1e-12)
    assert np.allclose(dv, tv.grad.transpose(0, 1).numpy(), atol=1e-12)


def test_backward_row_sum_identity():
    """Per row the softmax Jacobian sums to zero over [sink, scores], so
    sum_j dS_ij = P_c,i D_i = -(row i's share of dsink). With every query row
    equal to one vector q, sum_j dk_j = scale * sum_i (sum_j dS_ij) q
    = -scale * dsink * q."""
    g = np.random.default_rng(9)
    lq, lk, d = 5, 7, 4
    qrow = g.standard_normal(d)
    q = np.tile(qrow, (lq, 1, 1))
    k = g.standard_normal((lk, 1, d))
    v = g.standard_normal((lk, 1, d))
    do = g.standard_normal((lq, 1, d))
    sinks = np.array([0.4])
    cq, ck = np.array([0, lq]), np.array([0, lk])
    _, dk, _, ds = OB.backward(q, k, v, cq, ck, do, hq=1, hkv=1, sinks=sinks, causal=True,
                               scale=0.5)
    # sum_j dk_j = scale * sum_i (sum_j dS_ij) q = scale * (-dsink) * qrow
    assert np.allclose(dk.sum(axis=0)[0], 0.5 * (-ds[0]) * qrow, atol=1e-12)


MUTANTS = {
    "D term dropped": ("ds = p * (dp - d_row[:, None])", "ds = p * dp"),
    "dsink sign": ("dsink[h] += -(pc * d_row).sum()", "dsink[h] += (pc * d_row).sum()"),
    "dk without scale": ("dk[k0:k1, g] += scale * (ds.T @ qh)", "dk[k0:k1, g] += ds.T @ qh"),
    "dv from dS": ("dv[k0:k1, g] += p.T @ doh", "dv[k0:k1, g] += ds.T @ doh"),
    "dq transposed operand": ("dq[q0:q1, h] = scale * (ds @ kg)",
                              "dq[q0:q1, h] = scale * (p @ kg)"),
    "sink left out of Z": ("den = ec + e.sum(axis=1)", "den = e.sum(axis=1)"),
    "kv head by modulo": ("            g = h // group\n            sink = sk[h] if sk is not None "
                          "else -np.inf\n            qh,",
                          "            g = h % hkv\n            sink = sk[h] if sk is not None "
                          "else -np.inf\n            qh,"),
    "window one key too wide": ("vis &= j > pos - window", "vis &= j >= pos - window"),
}


def _mutant(old, new):
    import inspect
    import types
    src = inspect.getsource(OB)
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_backward_mutant")
    exec(compile(src.replace(old, new), "oracle_backward_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    mod = _mutant(*MUTANTS[name])
    caught = False
    for spec in TINY:
        try:
            check_fd(mod, spec)
        except AssertionError:
            caught = True
            break
    if not caught:
        # the forward-side mistakes move forward and backward together; the
        # C oracle (pinned on its own) catches those
        try:
            c_q = np.random.default_rng(3).standard_normal((6, 4, 64)).astype(np.float32)
            tq = torch.tensor(c_q).to(torch.bfloat16)
            tk = torch.tensor(c_q[:, :2]).to(torch.bfloat16)
            cu = torch.tensor([0, 6], dtype=torch.int32)
            sinks = torch.tensor([0.3, -0.2, 1.0, 0.0])
            ro, _ = oracle.attention(tq, tk, tk, cu, cu, hq=4, hkv=2, head_dim=64, sinks=sinks,
                                     causal=True, window=2, scale=0.125)
            o, _ = mod.forward(tq, tk, tk, cu, cu, hq=4, hkv=2, sinks=sinks, causal=True,
                               window=2, scale=0.125)
            assert np.allclose(o, ro, atol=1e-12)
        except AssertionError:
            caught = True
    assert caught, "no pin failed for mutant: " + name

"""Pins for the float64 oracle, each against something other than the oracle.

1. 40-digit decimal brute force on tiny inputs, written without the oracle's
   max shift (exp of raw logits), over every mask mode, both K/V layouts,
   grouped heads, ragged and empty sequences.
2. Closed-form cases (tests/golden/closed_form.json).
3. With no sink the result is ordinary attention: torch's float64
   scaled_dot_product_attention with an explicit boolean mask.
4. A sink far above every score drives the output to 0 and the lse to the sink.
5. out_sink = out_plain * sigmoid(lse_plain - sink) and
   lse_sink = logaddexp(lse_plain, sink) (sink enters the denominator only).
6. Splitting the keys into blocks, placing the sink in exactly one block and
   merging by log-sum-exp gives the unsplit result, whichever block holds it.
7. A window at least the context length changes nothing; causal with one
   query at the end of its context changes nothing.

Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention" fixes
the definition these pins check (sink logit in the softmax, no value row, sink
counted in one block only when the KV sequence is split).
"""
import json
import math
import os
import re
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

from attention_learned_sinks_gb300 import synthetic as S

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- helpers ---

def _dec_inputs(t):
    """bf16 tensor -> nested lists of exact Decimals."""
    f = t.float().numpy()
    return np.vectorize(lambda x: Decimal(float(x)), otypes=[object])(f)


def brute_force(case_q, case_k, case_v, cu_q, lens_k, hq, hkv, sinks, causal,
                window, scale):
    """Decimal reference. K/V given per sequence as [Lk, hkv, D] arrays."""
    getcontext().prec = 40
    G = hq // hkv
    D = case_q.shape[-1]
    sc = Decimal(float(scale))
    outs, lses = [], []
    qd = _dec_inputs(case_q)
    for b in range(len(lens_k)):
        kd = _dec_inputs(case_k[b])
        vd = _dec_inputs(case_v[b])
        lq = int(cu_q[b + 1] - cu_q[b])
        lk = lens_k[b]
        for i in range(lq):
            row_o, row_l = [], []
            for g in range(hkv):
                for r in range(G):
                    h = g * G + r
                    pos = lk - lq + i
                    weights = []
                    for j in range(lk):
                        if causal and j > pos:
                            continue
                        if window and not (j > pos - window):
                            continue
                        s = sum(qd[int(cu_q[b]) + i, h, c] * kd[j, g, c] for c in range(D)) * sc
                        weights.append((s.exp(), j))
                    den = sum((w for w, _ in weights), Decimal(0))
                    if sinks is not None:
                        den += Decimal(float(sinks[h])).exp()
                    if den == 0:
                        row_o.append([Decimal(0)] * D)
                        row_l.append(None)
                        continue
                    o = [sum((w * vd[j, g, c] for w, j in weights), Decimal(0)) / den
                         for c in range(D)]
                    row_o.append(o)
                    row_l.append(den.ln())
            outs.append(row_o)
            lses.append(row_l)
    return outs, lses


def _gather_paged(case, b):
    """K/V of sequence b as [Lk, hkv, D] from a paged cache (test-side gather)."""
    L = case.seqlens_k[b]
    n = (L + case.page_size - 1) // case.page_size
    pages = case.block_table[b, :n].long()
    kk = case.k_cache[pages].permute(0, 2, 1, 3).reshape(-1, case.hkv, case.head_dim)[:L]
    vv = case.v_cache[pages].permute(0, 2, 1, 3).reshape(-1, case.hkv, case.head_dim)[:L]
    return kk, vv


def _oracle_prefill(oracle, c, **kw):
    args = dict(hq=c.hq, hkv=c.hkv, head_dim=c.head_dim, sinks=c.sinks,
                causal=c.causal, window=c.window, scale=c.scale)
    args.update(kw)
    return oracle.attention(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, **args)


# ------------------------------------------------------- 1. brute force ---

TINY = [
    # (lens_q, lens_k, hq, hkv, D, causal, window, sinks)
    ([3], [3], 2, 1, 4, True, 0, True),
    ([3], [5], 2, 2, 3, True, 0, True),      # bottom-right alignment
    ([4, 2], [4, 5], 4, 2, 2, True, 2, True),
    ([5], [5], 2, 1, 4, False, 0, True),
    ([5], [5], 2, 1, 2, False, 2, True),     # left bound only
    ([2, 0, 3], [2, 4, 3], 2, 1, 3, True, 1, True),  # empty q sequence
    ([4], [2], 2, 1, 2, True, 0, True),      # more queries than keys
    ([3], [0], 2, 1, 2, True, 0, True),      # no keys at all
    ([3], [4], 4, 2, 3, True, 0, False),
    ([1, 1], [5, 3], 4, 1, 4, True, 3, True),  # decode-like
]


@pytest.mark.parametrize("spec", TINY, ids=[str(i) for i in range(len(TINY))])
def test_oracle_matches_decimal_brute_force(oracle_lib, spec):
    lens_q, lens_k, hq, hkv, D, causal, window, with_sinks = spec
    seed = 100 + TINY.index(spec)
    c = S.make_prefill("tiny", lens_q, lens_k, hq, hkv, seed=seed, causal=causal,
                       window=window, with_sinks=with_sinks, sink_std=1.5,
                       scale=0.7, head_dim=D)
    out, lse = _oracle_prefill(oracle_lib, c)
    ks = [c.k[int(c.cu_seqlens_k[b]):int(c.cu_seqlens_k[b + 1])] for b in range(c.batch)]
    vs = [c.v[int(c.cu_seqlens_k[b]):int(c.cu_seqlens_k[b + 1])] for b in range(c.batch)]
    bo, bl = brute_force(c.q, ks, vs, c.cu_seqlens_q, lens_k, hq, hkv,
                         c.sinks, causal, window, c.scale)
    assert out.shape[0] == len(bo)
    for r in range(len(bo)):
        for h in range(hq):
            ref = np.array([float(x) for x in bo[r][h]])
            assert np.max(np.abs(out[r, h] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
            if bl[r][h] is None:
                assert lse[r, h] == -math.inf
            else:
                assert abs(lse[r, h] - float(bl[r][h])) <= 1e-12 * max(1.0, abs(float(bl[r][h])))


@pytest.mark.parametrize("window", [0, 3, 20])
def test_oracle_paged_matches_brute_force(oracle_lib, window):
    lens = [5, 17, 1, 33]
    c = S.make_decode("tiny_paged", lens, 4, 2, seed=7, window=window, paged=True,
                      page_size=4, head_dim=4, scale=0.6)
    cu_q = torch.arange(0, c.batch + 1, dtype=torch.int32)
    out, lse = oracle_lib.attention(c.q, c.k_cache, c.v_cache, cu_q,
                                    block_table=c.block_table, seqlens_k=c.seqlens_k_t,
                                    hq=4, hkv=2, head_dim=4, sinks=c.sinks,
                                    causal=True, window=window, scale=c.scale)
    ks, vs = zip(*[_gather_paged(c, b) for b in range(c.batch)])
    bo, bl = brute_force(c.q, ks, vs, cu_q, lens, 4, 2, c.sinks, True, window, c.scale)
    for b in range(c.batch):
        for h in range(4):
            ref = np.array([float(x) for x in bo[b][h]])
            assert np.max(np.abs(out[b, h] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
            assert abs(lse[b, h] - float(bl[b][h])) <= 1e-12 * max(1.0, abs(float(bl[b][h])))


# ------------------------------------------------------ 2. closed forms ---

def _eval_expr(expr):
    getcontext().prec = 40
    ns = {"D": Decimal, "e": Decimal(1).exp(), "ln": lambda x: Decimal(x).ln(),
          "exp": lambda x: Decimal(x).exp()}
    src = re.sub(r"(?<![A-Za-z_])(\d+(?:\.\d+)?)", r"D('\1')", expr)
    return eval(src, {"__builtins__": {}}, ns)


def test_oracle_closed_forms(oracle_lib):
    with open(os.path.join(HERE, "golden", "closed_form.json")) as f:
        spec = json.load(f)
    for cs in spec["cases"]:
        D = cs["D"]
        q = torch.tensor(cs["q"], dtype=torch.float32).to(torch.bfloat16).reshape(-1, 1, D)
        k = torch.tensor(cs["k"], dtype=torch.float32).to(torch.bfloat16).reshape(-1, 1, D)
        v = torch.tensor(cs["v"], dtype=torch.float32).to(torch.bfloat16).reshape(-1, 1, D)
        assert torch.equal(q.float().reshape(-1, D), torch.tensor(cs["q"])), "inputs must be exact in bf16"
        sinks = None if cs["sink"] is None else torch.tensor([cs["sink"]], dtype=torch.float32)
        cu_q = torch.tensor([0, q.shape[0]], dtype=torch.int32)
        cu_k = torch.tensor([0, k.shape[0]], dtype=torch.int32)
        out, lse = oracle_lib.attention(q, k, v, cu_q, cu_k, hq=1, hkv=1, head_dim=D,
                                        sinks=sinks, causal=cs["causal"],
                                        window=cs["window"], scale=cs["scale"])
        for i, row in enumerate(cs["expect_out"]):
            for c_, ex in enumerate(row):
                assert abs(out[i, 0, c_] - float(_eval_expr(ex))) <= 1e-14, (cs["name"], i, c_)
            assert abs(lse[i, 0] - float(_eval_expr(cs["expect_lse"][i]))) <= 1e-14, cs["name"]


# ------------------------------------------ 3. no sink = ordinary attention ---

@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 7), (False, 5)])
def test_oracle_without_sink_is_sdpa(oracle_lib, causal, window):
    lens_q = [9, 1, 23]
    lens_k = [9, 14, 30]
    c = S.make_prefill("sdpa", lens_q, lens_k, 8, 2, seed=11, causal=causal,
                       window=window, with_sinks=False, head_dim=16, scale=0.3)
    out, lse = _oracle_prefill(oracle_lib, c)
    G = c.hq // c.hkv
    for b in range(c.batch):
        q0, q1 = int(c.cu_seqlens_q[b]), int(c.cu_seqlens_q[b + 1])
        k0, k1 = int(c.cu_seqlens_k[b]), int(c.cu_seqlens_k[b + 1])
        lq, lk = q1 - q0, k1 - k0
        q = c.q[q0:q1].double().permute(1, 0, 2)                      # [hq, lq, D]
        k = c.k[k0:k1].double().permute(1, 0, 2).repeat_interleave(G, 0)
        v = c.v[k0:k1].double().permute(1, 0, 2).repeat_interleave(G, 0)
        pos = torch.arange(lq).unsqueeze(1) + (lk - lq)
        j = torch.arange(lk).unsqueeze(0)
        mask = torch.ones(lq, lk, dtype=torch.bool)
        if causal:
            mask &= j <= pos
        if window:
            mask &= j > pos - window
        ok = mask.any(1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=mask, scale=c.scale)                      # [hq, lq, D]
        ref = ref.permute(1, 0, 2).numpy()
        got = out[q0:q1]
        assert np.max(np.abs(got[ok.numpy()] - ref[ok.numpy()])) <= 1e-12
        # lse of plain attention: logsumexp of the visible scaled scores
        s = (q @ k.transpose(1, 2)) * c.scale
        s = s.masked_fill(~mask, -math.inf)
        ref_lse = torch.logsumexp(s, dim=-1).permute(1, 0).numpy()
        assert np.max(np.abs(lse[q0:q1][ok.numpy()] - ref_lse[ok.numpy()])) <= 1e-12
        assert np.all(out[q0:q1][~ok.numpy()] == 0)
        assert np.all(lse[q0:q1][~ok.numpy()] == -math.inf)


# --------------------------------------------------------- 4. large sink ---

def test_oracle_large_sink_drives_output_to_zero(oracle_lib):
    c = S.make_prefill("big", [12, 20], [12, 20], 4, 2, seed=13, causal=True,
                       with_sinks=False, head_dim=8, scale=0.5)
    _, lse_plain = _oracle_prefill(oracle_lib, c)
    # per head: 60 above the largest score any row of that head can see
    G = c.hq // c.hkv
    smax = []
    for h in range(c.hq):
        qh = c.q[:, h].double()
        kh = c.k[:, h // G].double()
        smax.append(float((qh @ kh.T).max()) * c.scale)
    sinks = torch.tensor(smax, dtype=torch.float32) + 60.0
    out, lse = _oracle_prefill(oracle_lib, c, sinks=sinks)
    vmax = float(c.v.double().abs().max())
    bound = math.exp(-60.0) * vmax * 20
    assert np.max(np.abs(out)) <= bound
    assert np.max(np.abs(lse - sinks.double().numpy()[None, :])) <= 20 * math.exp(-59.0)
    assert np.all(lse_plain < sinks.double().numpy()[None, :])


# --------------------------------------------- 5. scaling identity --------

@pytest.mark.parametrize("window", [0, 6])
def test_oracle_sink_scales_plain_attention(oracle_lib, window):
    c = S.make_prefill("scal", [7, 16, 3], [7, 25, 40], 6, 3, seed=17, causal=True,
                       window=window, sink_std=2.0, head_dim=16, scale=0.25)
    out_s, lse_s = _oracle_prefill(oracle_lib, c)
    out_p, lse_p = _oracle_prefill(oracle_lib, c, sinks=None)
    sink = c.sinks.double().numpy()[None, :]
    ok = np.isfinite(lse_p)
    sig = 1.0 / (1.0 + np.exp(sink - lse_p))          # sum e^s / (sum e^s + e^sink)
    assert np.max(np.abs(out_s - out_p * sig[:, :, None])[ok]) <= 1e-12
    assert np.max(np.abs(lse_s - np.logaddexp(lse_p, sink))[ok]) <= 1e-12
    # rows that see nothing: output 0, lse = sink
    assert np.all(out_s[~ok] == 0)
    assert np.all(np.abs(lse_s - np.broadcast_to(sink, lse_s.shape))[~ok] == 0)


# --------------------------------------------- 6. split invariance --------

@pytest.mark.parametrize("nsplit", [1, 2, 3, 5])
def test_oracle_split_blocks_merge_to_whole(oracle_lib, nsplit):
    c = S.make_prefill("split", [6, 1, 11], [30, 9, 11], 4, 1, seed=19 + nsplit,
                       causal=True, window=0, sink_std=1.0, head_dim=8, scale=0.4)
    whole_o, whole_l = _oracle_prefill(oracle_lib, c)
    lens_k = np.array(c.seqlens_k)
    rng = np.random.default_rng(nsplit)
    # random cut points per sequence (blocks may be empty)
    cuts = [np.sort(rng.integers(0, L + 1, size=nsplit - 1)) for L in lens_k]
    bounds = [np.concatenate([[0], cu, [L]]) for cu, L in zip(cuts, lens_k)]
    for sink_block in range(nsplit):
        po, pl = [], []
        for kb in range(nsplit):
            begin = np.array([bd[kb] for bd in bounds], dtype=np.int32)
            end = np.array([bd[kb + 1] for bd in bounds], dtype=np.int32)
            o, l = _oracle_prefill(oracle_lib, c, kv_begin=begin, kv_end=end,
                                   use_sink=(kb == sink_block))
            po.append(o)
            pl.append(l)
        mo, ml = oracle_lib.merge(np.stack(po), np.stack(pl))
        assert np.max(np.abs(mo - whole_o)) <= 1e-12
        assert np.max(np.abs(ml - whole_l)) <= 1e-12
    # the sink may also enter as its own block in the merge
    po, pl = [], []
    for kb in range(nsplit):
        begin = np.array([bd[kb] for bd in bounds], dtype=np.int32)
        end = np.array([bd[kb + 1] for bd in bounds], dtype=np.int32)
        o, l = _oracle_prefill(oracle_lib, c, kv_begin=begin, kv_end=end, use_sink=False)
        po.append(o)
        pl.append(l)
    mo, ml = oracle_lib.merge(np.stack(po), np.stack(pl), sinks=c.sinks)
    assert np.max(np.abs(mo - whole_o)) <= 1e-12
    assert np.max(np.abs(ml - whole_l)) <= 1e-12


def test_oracle_sink_counted_twice_is_detected(oracle_lib):
    """Guard for pin 6: a sink entered in two blocks must NOT reproduce the whole."""
    c = S.make_prefill("split2", [4], [12], 2, 1, seed=29, causal=True,
                       head_dim=4, scale=0.5)
    whole_o, _ = _oracle_prefill(oracle_lib, c)
    o0, l0 = _oracle_prefill(oracle_lib, c, kv_begin=np.array([0], np.int32),
                             kv_end=np.array([6], np.int32), use_sink=True)
    o1, l1 = _oracle_prefill(oracle_lib, c, kv_begin=np.array([6], np.int32),
                             kv_end=np.array([12], np.int32), use_sink=True)
    mo, _ = oracle_lib.merge(np.stack([o0, o1]), np.stack([l0, l1]))
    assert np.max(np.abs(mo - whole_o)) > 1e-6


# ---------------------------------------------- 7. degenerate masks -------

def test_oracle_degenerate_masks(oracle_lib):
    c = S.make_prefill("deg", [5, 8], [9, 8], 4, 2, seed=23, causal=True, head_dim=8,
                       scale=0.5)
    full_o, full_l = _oracle_prefill(oracle_lib, c)
    wide_o, wide_l = _oracle_prefill(oracle_lib, c, window=9)
    assert np.array_equal(full_o, wide_o) and np.array_equal(full_l, wide_l)
    # one query at the end of its context: causal == non-causal
    d = S.make_decode("deg_dec", [1, 7, 40], 4, 2, seed=24, head_dim=8)
    cu_q = torch.arange(0, 4, dtype=torch.int32)
    a = oracle_lib.attention(d.q, d.k, d.v, cu_q, d.kv_indptr, hq=4, hkv=2, head_dim=8,
                             sinks=d.sinks, causal=True, scale=d.scale)
    b = oracle_lib.attention(d.q, d.k, d.v, cu_q, d.kv_indptr, hq=4, hkv=2, head_dim=8,
                             sinks=d.sinks, causal=False, scale=d.scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_oracle_rows_match_full(oracle_lib):
    c = S.make_prefill("rows", [10, 4], [10, 30], 4, 2, seed=31, causal=True,
                       window=5, head_dim=8, scale=0.5)
    full_o, full_l = _oracle_prefill(oracle_lib, c)
    rows = np.array([[0, 0, 0], [0, 3, 9], [1, 2, 3], [1, 1, 0]], dtype=np.int32)
    o, l = oracle_lib.attention_rows(rows, c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                     hq=4, hkv=2, head_dim=8, sinks=c.sinks, causal=True,
                                     window=5, scale=c.scale)
    for n, (b, h, i) in enumerate(rows):
        r = int(c.cu_seqlens_q[b]) + i
        assert np.array_equal(o[n], full_o[r, h]) and l[n] == full_l[r, h]

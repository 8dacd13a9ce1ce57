"""Float64 CPU oracle for the backward pass of sink attention.

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg use this module; the library's product path never imports
it, and it shares no code with the CUDA sources.

The pages describe only the forward pass (page "GPT-OSS on day 0", sections
"Attention: GQA with Attention Sinks" and "Kernels for GPT-OSS / Sink
Attention": one trained sink logit per head, inside the softmax denominator,
with no value row). The gradients below follow from that definition by the
chain rule; they are pinned by finite differences of `forward` in the tests.

For query row i of head h (KV head g = h / (Hq / Hkv)) with visible keys J,
scores s_j = scale * q_i . k_j and sink logit c_h:

  P_j = e^{s_j} / Z,   P_c = e^{c_h} / Z,   Z = e^{c_h} + sum_{j in J} e^{s_j}
  o_i = sum_j P_j v_j
  dP_j = dO_i . v_j              (the sink has no value row: dP_c = 0)
  D_i = sum_j P_j dP_j  (= dO_i . o_i)
  dS_j = P_j (dP_j - D_i)        (softmax Jacobian over [sink, scores])
  dq_i    = scale * sum_j dS_j k_j
  dk_j   += scale * dS_j q_i     (summed over the group's query heads)
  dv_j   += P_j dO_i
  dc_h   += P_c (0 - D_i)        (summed over every row of head h)

Everything is float64: inputs are taken at their exact values (bf16 inputs
convert exactly), one explicit score matrix per (sequence, head).
"""
import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def _visible(lq, lk, causal, window):
    """Boolean [lq, lk]: key j visible from query i (queries are the last lq
    of the lk positions: p_i = lk - lq + i)."""
    pos = (lk - lq) + np.arange(lq)[:, None]
    j = np.arange(lk)[None, :]
    vis = np.ones((lq, lk), dtype=bool)
    if causal:
        vis &= j <= pos
    if window > 0:
        vis &= j > pos - window
    return vis


def _probs(q, k, vis, sink, scale):
    """P [lq, lk] over the visible keys and the sink's share P_c [lq], from
    the definition: softmax over [sink, scores]. Rows with nothing visible and
    no sink get all zeros."""
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    z = np.maximum(s.max(axis=1, initial=-np.inf), sink)
    live = np.isfinite(z)
    zz = np.where(live, z, 0.0)
    e = np.where(vis, np.exp(s - zz[:, None]), 0.0)
    ec = np.where(live, np.exp(sink - zz), 0.0) if np.isfinite(sink) else np.zeros_like(zz)
    den = ec + e.sum(axis=1)
    den_safe = np.where(live, den, 1.0)
    p = np.where(live[:, None], e / den_safe[:, None], 0.0)
    pc = np.where(live, ec / den_safe, 0.0)
    lse = np.where(live, zz + np.log(den_safe), -np.inf)
    return p, pc, lse


def forward(q, k, v, cu_seqlens_q, cu_seqlens_k, *, hq, hkv, sinks=None, causal=True,
            window=0, scale):
    """Float64 forward (out [total_q, hq, d], lse [total_q, hq]) on float64
    inputs; the same definition as the C oracle, written with matrices."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck = _i64(cu_seqlens_q), _i64(cu_seqlens_k)
    sk = _f64(sinks)
    group = hq // hkv
    out = np.zeros(q.shape, dtype=np.float64)
    lse = np.full(q.shape[:2], -np.inf)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        lq, lk = q1 - q0, k1 - k0
        if lq == 0:
            continue
        vis = _visible(lq, lk, causal, window)
        for h in range(hq):
            g = h // group
            sink = sk[h] if sk is not None else -np.inf
            p, _, l = _probs(q[q0:q1, h], k[k0:k1, g], vis, sink, scale)
            out[q0:q1, h] = p @ v[k0:k1, g]
            lse[q0:q1, h] = l
    return out, lse


def backward(q, k, v, cu_seqlens_q, cu_seqlens_k, dout, *, hq, hkv, sinks=None, causal=True,
             window=0, scale, seqs=None):
    """Gradients of sum(dout * out) with respect to q, k, v and the sinks.

    Returns float64 (dq [total_q, hq, d], dk [total_k, hkv, d],
    dv [total_k, hkv, d], dsinks [hq] or None without sinks). `seqs` limits
    the work to those sequences: their rows of dq/dk/dv are exact, other rows
    stay zero, and dsinks sums over those sequences only.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    cq, ck = _i64(cu_seqlens_q), _i64(cu_seqlens_k)
    sk = _f64(sinks)
    group = hq // hkv
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    dsink = np.zeros(hq, dtype=np.float64)
    for b in (range(len(cq) - 1) if seqs is None else seqs):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        lq, lk = q1 - q0, k1 - k0
        if lq == 0:
            continue
        vis = _visible(lq, lk, causal, window)
        for h in range(hq):
            g = h // group
            sink = sk[h] if sk is not None else -np.inf
            qh, kg, vg, doh = q[q0:q1, h], k[k0:k1, g], v[k0:k1, g], do[q0:q1, h]
            p, pc, _ = _probs(qh, kg, vis, sink, scale)
            dp = doh @ vg.T
            d_row = (p * dp).sum(axis=1)
            ds = p * (dp - d_row[:, None])
            dq[q0:q1, h] = scale * (ds @ kg)
            dk[k0:k1, g] += scale * (ds.T @ qh)
            dv[k0:k1, g] += p.T @ doh
            dsink[h] += -(pc * d_row).sum()
    return dq, dk, dv, (dsink if sk is not None else None)

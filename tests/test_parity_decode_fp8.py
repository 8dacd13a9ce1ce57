"""GPU decode over an fp8 e4m3 KV cache against the float64 oracle.

The oracle decodes the same e4m3 codes exactly (oracle/fp8.py), applies the
per-KV-head scales and runs the float64 forward on the values."""
import numpy as np
import pytest
import torch

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import synthetic as S
from helpers import check_close, cuda
from oracle import backward as OB
from oracle import fp8 as F

pytestmark = pytest.mark.gpu


def run(c, num_splits=0, scales=True):
    ks = cuda(c.k_scale) if scales else None
    vs = cuda(c.v_scale) if scales else None
    if c.paged:
        return sa.sinkattn_decode_fp8(c.q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(), k_scale=ks,
                                      v_scale=vs, block_table=c.block_table.cuda(),
                                      seqlens_k=c.seqlens_k_t.cuda(), max_seqlen_k=c.max_seqlen_k,
                                      sinks=cuda(c.sinks), window=c.window, scale=c.scale,
                                      num_splits=num_splits)
    return sa.sinkattn_decode_fp8(c.q.cuda(), c.k.cuda(), c.v.cuda(), k_scale=ks, v_scale=vs,
                                  kv_indptr=c.kv_indptr.cuda(), max_seqlen_k=c.max_seqlen_k,
                                  sinks=cuda(c.sinks), window=c.window, scale=c.scale,
                                  num_splits=num_splits)


def reference(c, seqs=None, scales=True):
    """float64 forward over the decoded cache (contiguous per sequence)."""
    seqs = list(range(c.batch)) if seqs is None else seqs
    ks = c.k_scale if scales else torch.ones(c.hkv)
    vs = c.v_scale if scales else torch.ones(c.hkv)
    kd, vd = [], []
    for b in seqs:
        L = c.seqlens_k[b]
        if c.paged:
            j = np.arange(L)
            pages = c.block_table[b].numpy()[j // c.page_size]
            kc = c.k_cache.numpy()[pages, :, j % c.page_size]
            vc = c.v_cache.numpy()[pages, :, j % c.page_size]
        else:
            k0 = int(c.kv_indptr[b])
            kc, vc = c.k.numpy()[k0:k0 + L], c.v.numpy()[k0:k0 + L]
        kd.append(F.dequantize(kc.reshape(L, c.hkv, c.head_dim), ks, 1))
        vd.append(F.dequantize(vc.reshape(L, c.hkv, c.head_dim), vs, 1))
    lens = [c.seqlens_k[b] for b in seqs]
    cu_k = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    cu_q = np.arange(len(seqs) + 1)
    return OB.forward(c.q[seqs], np.concatenate(kd), np.concatenate(vd), cu_q, cu_k, hq=c.hq,
                      hkv=c.hkv, sinks=c.sinks, causal=True, window=c.window, scale=c.scale)


LENS = [1, 31, 32, 33, 127, 128, 129, 511, 512, 513, 1000, 1537, 2048, 3001, 0, 77]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (64, 8), (24, 3), (32, 2)])
@pytest.mark.parametrize("window", [0, 1, 100])
def test_decode_fp8_contiguous(hq, hkv, window):
    c = S.make_decode("fp8", LENS, hq, hkv, seed=141 + hq + window, window=window,
                      sink_std=1.5, kv_dtype="fp8")
    out, lse = run(c)
    ro, rl = reference(c)
    check_close(out, lse, ro, rl, "decode fp8 hq=%d hkv=%d w=%d" % (hq, hkv, window))


@pytest.mark.parametrize("page_size", [16, 24])
@pytest.mark.parametrize("window", [0, 200])
def test_decode_fp8_paged(page_size, window):
    c = S.make_decode("fp8p", LENS, 64, 8, seed=143 + window, window=window, paged=True,
                      page_size=page_size, sink_std=2.0, kv_dtype="fp8")
    out, lse = run(c)
    ro, rl = reference(c)
    check_close(out, lse, ro, rl, "decode fp8 paged ps=%d w=%d" % (page_size, window))


@pytest.mark.parametrize("num_splits", [1, 3, 17])
def test_decode_fp8_splits_and_unit_scales(num_splits):
    c = S.make_decode("fp8s", [5000, 4097, 1, 300], 64, 8, seed=145, kv_dtype="fp8")
    vmax = float(np.abs(F.dequantize(c.v, torch.ones(8), 1)).max())  # unscaled codes
    for scales in (True, False):  # NULL scales mean 1
        out, lse = run(c, num_splits=num_splits, scales=scales)
        ro, rl = reference(c, scales=scales)
        check_close(out, lse, ro, rl, "fp8 splits=%d scales=%s" % (num_splits, scales),
                    v_absmax=None if scales else vmax)


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("window", [0, 100])
def test_decode_fp8_head_dim_128(paged, window):
    c = S.make_decode("fp8d128", LENS, 64, 8, seed=151 + window, window=window, paged=paged,
                      page_size=16, sink_std=1.5, kv_dtype="fp8", head_dim=128)
    for ns in (0, 7):
        out, lse = run(c, num_splits=ns)
        ro, rl = reference(c)
        check_close(out, lse, ro, rl, "fp8 d=128 paged=%s w=%d ns=%d" % (paged, window, ns))


def test_decode_fp8_without_sinks_and_empty():
    c = S.make_decode("fp8n", [0, 700, 33], 16, 2, seed=147, with_sinks=False, kv_dtype="fp8")
    out, lse = run(c)
    ro, rl = reference(c)
    check_close(out, lse, ro, rl, "fp8 no sinks")
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_decode_fp8_contig_full_config():
    """64 sequences, KV lengths uniform in [1024, 8192], 64 q / 8 kv heads, fp8
    cache: every output against the oracle."""
    c = S.decode_contig_fp8()
    out, lse = run(c)
    ro, rl = reference(c)
    check_close(out, lse, ro, rl, "decode_contig_fp8")


def test_decode_fp8_matches_bf16_of_the_same_values():
    """The fp8 call on codes equals the bf16 call on the decoded values (every
    scaled e4m3 value with scale 1 is a bf16 value) within the parity bar."""
    c = S.make_decode("fp8eq", [700, 2000, 64], 64, 8, seed=149, kv_dtype="fp8")
    kb = torch.tensor(F.dequantize(c.k, torch.ones(8), 1)).to(torch.bfloat16)
    vb = torch.tensor(F.dequantize(c.v, torch.ones(8), 1)).to(torch.bfloat16)
    a = run(c, scales=False)
    b = sa.sinkattn_decode(c.q.cuda(), kb.cuda(), vb.cuda(), kv_indptr=c.kv_indptr.cuda(),
                           max_seqlen_k=c.max_seqlen_k, sinks=c.sinks.cuda())
    ro, rl = reference(c, scales=False)
    vmax = float(vb.float().abs().max())  # unscaled codes: values up to a few hundred
    check_close(a[0], a[1], ro, rl, "fp8 vs oracle", v_absmax=vmax)
    check_close(b[0], b[1], ro, rl, "bf16 of the decoded values vs oracle", v_absmax=vmax)

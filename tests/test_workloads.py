"""The seeded synthetic workloads have the shapes, lengths, value
distributions and page structure their recipes state (the five benchmark
configurations and the extra workloads). CPU only: the largest caches are
checked through the same recipe at a smaller batch."""
import numpy as np
import pytest
import torch

from attention_learned_sinks_gb300 import synthetic as S


def _stats(t, n=1 << 20):
    x = t.reshape(-1)[:n].float().numpy().astype(np.float64)
    return float(x.mean()), float(x.std())


def _check_normal(t, std=1.0):
    """bf16 N(0, std^2): mean and spread of the first million draws."""
    mean, sd = _stats(t)
    assert abs(mean) < 0.01 * std and abs(sd / std - 1.0) < 0.01, (mean, sd)


def test_uniform_lengths_cover_both_ends():
    x = S.uniform_lengths(20000, 3, 7, seed=11)
    assert min(x) == 3 and max(x) == 7
    assert S.uniform_lengths(50, 512, 4096, seed=5) == S.uniform_lengths(50, 512, 4096, seed=5)


def test_bf16_normal_is_rounded_fp32_normal():
    t = S.bf16_normal((1 << 20,), seed=7, std=2.0)
    assert t.dtype == torch.bfloat16
    _check_normal(t, 2.0)
    # chunked drawing gives the same values as one draw of the same generator
    a = S.bf16_normal((3000, 5), seed=9, chunk_elems=1 << 26)
    b = S.bf16_normal((3000, 5), seed=9, chunk_elems=15000)
    assert torch.equal(a, b)


def test_tiny_prefill():
    c = S.tiny_prefill()
    assert c.seqlens_q == [64] and c.seqlens_k == [64]
    assert (c.hq, c.hkv, c.head_dim, c.causal, c.window) == (4, 1, 64, True, 0)
    assert c.scale == 1.0 / 8.0
    assert c.q.shape == (64, 4, 64) and c.k.shape == (64, 1, 64) and c.v.shape == (64, 1, 64)
    assert c.sinks.dtype == torch.float32 and c.sinks.shape == (4,)


def test_decode_contig():
    c = S.decode_contig()
    assert len(c.seqlens_k) == 64 and all(1024 <= l <= 8192 for l in c.seqlens_k)
    assert (c.hq, c.hkv, c.head_dim, c.window) == (64, 8, 64, 0)
    assert c.q.shape == (64, 64, 64)
    assert c.k.shape == (sum(c.seqlens_k), 8, 64) and c.v.shape == c.k.shape
    assert torch.equal(c.kv_indptr, S.offsets(c.seqlens_k))
    _check_normal(c.k)
    _check_normal(c.v)
    assert c.sinks.shape == (64,) and abs(float(c.sinks.std()) - 1.0) < 0.3
    # the head_dim 128 and fp8 variants keep the lengths and heads
    assert S.uniform_lengths(64, 1024, 8192, seed=2000) == c.seqlens_k


@pytest.mark.parametrize("window", [0, 128])
def test_varlen_prefill(window):
    c = S.varlen_prefill(window=window)
    assert len(c.seqlens_q) == 16 and c.seqlens_q == c.seqlens_k
    assert all(512 <= l <= 4096 for l in c.seqlens_q)
    assert (c.hq, c.hkv, c.head_dim, c.causal, c.window) == (64, 8, 64, True, window)
    assert c.q.shape == (sum(c.seqlens_q), 64, 64)
    assert torch.equal(c.cu_seqlens_q, S.offsets(c.seqlens_q))
    _check_normal(c.q)


def test_paged_decode_recipe():
    """paged_decode's recipe at batch 16: contexts in [1024, 32768], 16-token
    pages, every page referenced once through a permuted table, sinks with
    std 2."""
    c = S.paged_decode(batch=16)
    assert all(1024 <= l <= 32768 for l in c.seqlens_k)
    assert (c.hq, c.hkv, c.head_dim, c.page_size) == (64, 8, 64, 16)
    pages = [(l + 15) // 16 for l in c.seqlens_k]
    num_pages = c.k_cache.shape[0]
    assert num_pages == sum(pages)
    assert c.k_cache.shape == (num_pages, 8, 16, 64) and c.v_cache.shape == c.k_cache.shape
    used = torch.cat([c.block_table[b, :n] for b, n in enumerate(pages)])
    assert sorted(used.tolist()) == list(range(num_pages))
    # permuted: consecutive pages of a sequence are not laid out in order
    assert not torch.equal(used, torch.arange(num_pages, dtype=used.dtype))
    _check_normal(c.k_cache)
    assert c.sinks.shape == (64,) and 1.5 < float(c.sinks.std()) < 2.5
    # the full workload draws its 256 lengths from the same recipe
    full = S.uniform_lengths(256, 1024, 32768, seed=4000)
    assert len(full) == 256 and min(full) >= 1024 and max(full) <= 32768


def test_chunked_prefill():
    """4096 queries at positions 126976..131071 of a 131072-token context."""
    c = S.chunked_prefill()
    assert c.seqlens_q == [4096] and c.seqlens_k == [131072]
    assert (c.hq, c.hkv, c.head_dim, c.causal, c.window) == (64, 8, 64, True, 0)
    assert c.k.shape == (131072, 8, 64)
    lc = S.long_context_prefill(lk=4096)
    assert lc.seqlens_q == [256] and lc.causal


def test_paged_prefill_batch_recipe():
    c = S.paged_prefill_batch(nseq=4)
    new = S.uniform_lengths(4, 256, 2048, seed=6000)
    cached = S.uniform_lengths(4, 1024, 32768, seed=6001)
    assert c.seqlens_q == new and c.seqlens_k == [n + k for n, k in zip(new, cached)]
    assert c.page_size == 16 and c.k_cache.shape[1:] == (8, 16, 64)


def test_fp8_scales_recipe():
    s = S.fp8_scales(4096, seed=3)
    assert float(s.min()) >= 0.5 / 16 and float(s.max()) <= 2.0 / 16
    c = S.make_decode("f8", [100, 37], 16, 2, seed=5, kv_dtype="fp8")
    assert c.k.dtype == torch.uint8 and c.k_scale.shape == (2,)  # e4m3 codes as bytes
    # codes times their KV head's scale are N(0, 1) values
    x = c.k.view(torch.float8_e4m3fn).float() * c.k_scale.view(1, 2, 1)
    assert abs(float(x.std()) - 1.0) < 0.1


def test_workload_table_is_complete():
    assert set(S.WORKLOADS) >= {"tiny_prefill", "decode_contig", "varlen_prefill",
                                "paged_decode", "chunked_prefill"}

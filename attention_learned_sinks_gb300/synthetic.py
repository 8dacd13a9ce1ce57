"""Seeded synthetic inputs for sink attention.

This module is the one piece both the CUDA path's tests/benchmark and the
float64 oracle consume. It draws shapes, lengths and values only; it holds no
part of the attention arithmetic.

Workloads (gpt-oss-like head geometry: 64 query heads sharing 8 KV heads,
head_dim 64; the pages evaluate on real weights and an evaluation set that
are not available here, so seeded normal values stand in for them):

  tiny_prefill     1 sequence of 64 tokens, causal, 4 q / 1 kv heads, scale 1/8
  decode_contig    batch 64, one query each, KV lengths uniform in [1024, 8192]
  varlen_prefill   16 sequences, lengths uniform in [512, 4096], causal,
                   full or sliding window 128
  paged_decode     batch 256, contexts uniform in [1024, 32768], 16-token pages,
                   randomly permuted block table, sinks ~N(0, 2), full or window 128
  chunked_prefill  4096 new query tokens at positions 126976..131071 of a
                   131072-token causal context
  long_context_prefill   256 new query tokens at the end of a 131072-token
                   causal context (few query tiles: the split-KV case)
  decode_contig_d128 decode_contig's lengths and heads with head_dim 128
  varlen_prefill_d128  varlen_prefill's lengths and heads with head_dim 128
  varlen_prefill_g3    varlen_prefill's lengths with 24 q / 8 kv heads (groups
                   of 3: one head per work item)
  decode_contig_fp8  decode_contig's lengths and geometry over an fp8 e4m3 KV
                   cache with per-KV-head scales 2^-4 * U(0.5, 2)
  paged_chunked_prefill  the same as chunked_prefill, with K/V in 16-token pages and a randomly
                   permuted block table
  paged_prefill_batch    16 sequences, new chunks uniform in [256, 2048] after
                   cached contexts uniform in [1024, 32768], 16-token pages
  paged_chunked_prefill_fp8  paged_chunked_prefill over an fp8 e4m3 cache with
                   decode_contig_fp8's scale recipe

Conventions: "uniform in [a, b]" draws integers with both ends included; values
are float32 normal samples rounded to bf16 (round to nearest even); sinks stay
float32. Lengths use their own seed so that shapes do not depend on value draws.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import torch

HEAD_DIM = 64
PAGE_SIZE = 16


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> List[int]:
    """n integers drawn uniformly from [lo, hi], both ends included."""
    g = _gen(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def bf16_normal(shape, seed: int, std: float = 1.0, device="cpu",
                chunk_elems: int = 1 << 26) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) samples, drawn in float32 then rounded.

    Large tensors are drawn in chunks along dim 0 so the float32 staging
    stays small; the result depends only on (shape, seed, std, device).
    """
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    g = _gen(seed, device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        x = torch.randn(e - s, generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            x.mul_(std)
        flat[s:e].copy_(x)
    return out


def normal_f32(n: int, seed: int, std: float = 1.0) -> torch.Tensor:
    g = _gen(seed, "cpu")
    x = torch.randn(n, generator=g, dtype=torch.float32)
    return x * std if std != 1.0 else x


def offsets(lengths: List[int]) -> torch.Tensor:
    """int32 [len+1] start offsets of packed sequences (0, l0, l0+l1, ...)."""
    o = [0]
    for l in lengths:
        o.append(o[-1] + int(l))
    return torch.tensor(o, dtype=torch.int32)


@dataclass
class PrefillCase:
    name: str
    q: torch.Tensor            # bf16 [total_q, hq, D]
    k: torch.Tensor            # bf16 [total_k, hkv, D]
    v: torch.Tensor            # bf16 [total_k, hkv, D]
    cu_seqlens_q: torch.Tensor  # int32 [batch+1]
    cu_seqlens_k: torch.Tensor  # int32 [batch+1]
    seqlens_q: List[int]
    seqlens_k: List[int]
    hq: int
    hkv: int
    sinks: Optional[torch.Tensor]  # f32 [hq]
    causal: bool
    window: int
    scale: float
    head_dim: int = HEAD_DIM
    # paged K/V (k, v and cu_seqlens_k are None then)
    k_cache: Optional[torch.Tensor] = None      # bf16 [num_pages, hkv, page, D]
    v_cache: Optional[torch.Tensor] = None
    block_table: Optional[torch.Tensor] = None  # int32 [batch, max_pages]
    seqlens_k_t: Optional[torch.Tensor] = None  # int32 [batch]
    page_size: int = PAGE_SIZE
    # fp8 paged cache: k_cache/v_cache hold e4m3 codes as uint8; the value of
    # a code c of KV head g is k_scale[g] * e4m3(c)
    kv_dtype: str = "bf16"
    k_scale: Optional[torch.Tensor] = None  # f32 [hkv]
    v_scale: Optional[torch.Tensor] = None

    @property
    def batch(self):
        return len(self.seqlens_q)

    @property
    def paged(self):
        return self.block_table is not None

    @property
    def max_seqlen_q(self):
        return max(self.seqlens_q) if self.seqlens_q else 0

    @property
    def max_seqlen_k(self):
        return max(self.seqlens_k) if self.seqlens_k else 0


@dataclass
class DecodeCase:
    name: str
    q: torch.Tensor            # bf16 [batch, hq, D]
    seqlens_k: List[int]
    hq: int
    hkv: int
    sinks: Optional[torch.Tensor]
    window: int
    scale: float
    # contiguous layout
    k: Optional[torch.Tensor] = None        # bf16 [total_k, hkv, D]
    v: Optional[torch.Tensor] = None
    kv_indptr: Optional[torch.Tensor] = None  # int32 [batch+1]
    # paged layout
    k_cache: Optional[torch.Tensor] = None  # bf16 [num_pages, hkv, page, D]
    v_cache: Optional[torch.Tensor] = None
    block_table: Optional[torch.Tensor] = None  # int32 [batch, max_pages]
    seqlens_k_t: Optional[torch.Tensor] = None  # int32 [batch]
    page_size: int = PAGE_SIZE
    head_dim: int = HEAD_DIM
    # fp8 cache: k/v (or k_cache/v_cache) hold e4m3 codes as uint8; the value
    # of a code c of KV head g is k_scale[g] * e4m3(c)
    kv_dtype: str = "bf16"
    k_scale: Optional[torch.Tensor] = None  # f32 [hkv]
    v_scale: Optional[torch.Tensor] = None

    @property
    def batch(self):
        return len(self.seqlens_k)

    @property
    def max_seqlen_k(self):
        return max(self.seqlens_k) if self.seqlens_k else 0

    @property
    def paged(self):
        return self.block_table is not None


def make_prefill(name, seqlens_q, seqlens_k, hq, hkv, *, seed, causal=True,
                 window=0, sink_std=1.0, with_sinks=True, scale=None,
                 device="cpu", head_dim=HEAD_DIM) -> PrefillCase:
    tq = sum(seqlens_q)
    tk = sum(seqlens_k)
    q = bf16_normal((tq, hq, head_dim), seed * 10 + 1, device=device)
    k = bf16_normal((tk, hkv, head_dim), seed * 10 + 2, device=device)
    v = bf16_normal((tk, hkv, head_dim), seed * 10 + 3, device=device)
    sinks = normal_f32(hq, seed * 10 + 4, sink_std) if with_sinks else None
    return PrefillCase(name=name, q=q, k=k, v=v,
                       cu_seqlens_q=offsets(seqlens_q),
                       cu_seqlens_k=offsets(seqlens_k),
                       seqlens_q=list(seqlens_q), seqlens_k=list(seqlens_k),
                       hq=hq, hkv=hkv, sinks=sinks, causal=causal,
                       window=window,
                       scale=scale if scale is not None else head_dim ** -0.5,
                       head_dim=head_dim)


def _page_table(seqlens_k, page_size, seed, spare_pages=0):
    """Block table over randomly permuted pages: sequence b gets
    ceil(Lk_b / page_size) pages; spare_pages extra pages are never referenced."""
    pages_per_seq = [(l + page_size - 1) // page_size for l in seqlens_k]
    num_pages = max(1, sum(pages_per_seq) + spare_pages)
    max_pages = max(1, max(pages_per_seq) if pages_per_seq else 1)
    g = _gen(seed, "cpu")
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    table = torch.zeros((len(seqlens_k), max_pages), dtype=torch.int32)
    at = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[at:at + n]
        at += n
    return table, num_pages


def make_prefill_paged(name, seqlens_q, seqlens_k, hq, hkv, *, seed, causal=True,
                       window=0, sink_std=1.0, with_sinks=True, scale=None,
                       page_size=PAGE_SIZE, spare_pages=0, device="cpu",
                       head_dim=HEAD_DIM, kv_dtype="bf16") -> PrefillCase:
    """Packed queries against K/V in pages; the queries of sequence b are the
    last Lq_b of its Lk_b positions. kv_dtype "fp8": e4m3 codes with
    per-KV-head scales, as make_decode draws them."""
    tq = sum(seqlens_q)
    q = bf16_normal((tq, hq, head_dim), seed * 10 + 1, device=device)
    table, num_pages = _page_table(seqlens_k, page_size, seed * 10 + 5, spare_pages)
    sinks = normal_f32(hq, seed * 10 + 4, sink_std) if with_sinks else None
    shape = (num_pages, hkv, page_size, head_dim)
    k_scale = v_scale = None
    if kv_dtype == "fp8":
        k_scale = fp8_scales(hkv, seed * 10 + 6)
        v_scale = fp8_scales(hkv, seed * 10 + 7)
        k_cache = e4m3_codes(shape, seed * 10 + 2, k_scale, 1, device=device)
        v_cache = e4m3_codes(shape, seed * 10 + 3, v_scale, 1, device=device)
    else:
        k_cache = bf16_normal(shape, seed * 10 + 2, device=device)
        v_cache = bf16_normal(shape, seed * 10 + 3, device=device)
    return PrefillCase(name=name, q=q, k=None, v=None, cu_seqlens_q=offsets(seqlens_q),
                       cu_seqlens_k=None, seqlens_q=list(seqlens_q),
                       seqlens_k=list(seqlens_k), hq=hq, hkv=hkv, sinks=sinks,
                       causal=causal, window=window,
                       scale=scale if scale is not None else head_dim ** -0.5,
                       head_dim=head_dim, k_cache=k_cache, v_cache=v_cache,
                       block_table=table,
                       seqlens_k_t=torch.tensor(seqlens_k, dtype=torch.int32),
                       page_size=page_size, kv_dtype=kv_dtype, k_scale=k_scale,
                       v_scale=v_scale)


def fp8_scales(hkv: int, seed: int) -> torch.Tensor:
    """Per-KV-head fp8 scales 2^-4 * U(0.5, 2): codes of N(0, 1) values then
    reach magnitudes near 2^4 * 4 sigma, well inside e4m3's 448."""
    g = _gen(seed, "cpu")
    return (torch.rand(hkv, generator=g, dtype=torch.float32) * 1.5 + 0.5) / 16.0


def e4m3_codes(shape, seed: int, scale: torch.Tensor, head_axis: int,
               device="cpu") -> torch.Tensor:
    """uint8 e4m3 codes of N(0, 1) samples divided by the per-head scale
    (rounded to nearest even by torch's float8_e4m3fn conversion)."""
    x = torch.empty(shape, dtype=torch.float32, device=device)
    g = _gen(seed, device)
    flat = x.view(-1)
    step = 1 << 26
    for s in range(0, flat.numel(), step):
        e = min(flat.numel(), s + step)
        flat[s:e].copy_(torch.randn(e - s, generator=g, dtype=torch.float32, device=device))
    view = [1] * len(shape)
    view[head_axis] = shape[head_axis]
    x.div_(scale.to(device).view(view))
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def make_decode(name, seqlens_k, hq, hkv, *, seed, window=0, sink_std=1.0,
                with_sinks=True, paged=False, page_size=PAGE_SIZE, scale=None,
                device="cpu", head_dim=HEAD_DIM, kv_dtype="bf16") -> DecodeCase:
    batch = len(seqlens_k)
    q = bf16_normal((batch, hq, head_dim), seed * 10 + 1, device=device)
    sinks = normal_f32(hq, seed * 10 + 4, sink_std) if with_sinks else None
    case = DecodeCase(name=name, q=q, seqlens_k=list(seqlens_k), hq=hq,
                      hkv=hkv, sinks=sinks, window=window,
                      scale=scale if scale is not None else head_dim ** -0.5,
                      page_size=page_size, head_dim=head_dim, kv_dtype=kv_dtype)
    if kv_dtype == "fp8":
        case.k_scale = fp8_scales(hkv, seed * 10 + 6)
        case.v_scale = fp8_scales(hkv, seed * 10 + 7)

        def values(shape, s, which):
            sc = case.k_scale if which == "k" else case.v_scale
            return e4m3_codes(shape, s, sc, 1, device=device)
    else:
        def values(shape, s, which):
            return bf16_normal(shape, s, device=device)
    if not paged:
        tk = sum(seqlens_k)
        case.k = values((tk, hkv, head_dim), seed * 10 + 2, "k")
        case.v = values((tk, hkv, head_dim), seed * 10 + 3, "v")
        case.kv_indptr = offsets(seqlens_k)
        return case
    table, num_pages = _page_table(seqlens_k, page_size, seed * 10 + 5)
    case.k_cache = values((num_pages, hkv, page_size, head_dim), seed * 10 + 2, "k")
    case.v_cache = values((num_pages, hkv, page_size, head_dim), seed * 10 + 3, "v")
    case.block_table = table
    case.seqlens_k_t = torch.tensor(seqlens_k, dtype=torch.int32)
    return case


# ---- the named workloads ----------------------------------------------------

def tiny_prefill(device="cpu") -> PrefillCase:
    return make_prefill("tiny_prefill", [64], [64], 4, 1, seed=1, causal=True,
                        scale=1.0 / 8.0, device=device)


def decode_contig(device="cpu", batch=64) -> DecodeCase:
    lens = uniform_lengths(batch, 1024, 8192, seed=2000)
    return make_decode("decode_contig", lens, 64, 8, seed=2, device=device)


def varlen_prefill(window=0, device="cpu", nseq=16) -> PrefillCase:
    lens = uniform_lengths(nseq, 512, 4096, seed=3000)
    return make_prefill("varlen_prefill" + ("_w%d" % window if window else ""),
                        lens, lens, 64, 8, seed=3, causal=True, window=window,
                        device=device)


def decode_contig_d128(device="cpu", batch=64) -> DecodeCase:
    lens = uniform_lengths(batch, 1024, 8192, seed=2000)
    return make_decode("decode_contig_d128", lens, 64, 8, seed=10, device=device, head_dim=128)


def varlen_prefill_d128(device="cpu", nseq=16) -> PrefillCase:
    lens = uniform_lengths(nseq, 512, 4096, seed=3000)
    return make_prefill("varlen_prefill_d128", lens, lens, 64, 8, seed=11, causal=True,
                        device=device, head_dim=128)


def varlen_prefill_g3(device="cpu", nseq=16) -> PrefillCase:
    lens = uniform_lengths(nseq, 512, 4096, seed=3000)
    return make_prefill("varlen_prefill_g3", lens, lens, 24, 8, seed=13, causal=True,
                        device=device)


def decode_contig_fp8(device="cpu", batch=64) -> DecodeCase:
    lens = uniform_lengths(batch, 1024, 8192, seed=2000)
    return make_decode("decode_contig_fp8", lens, 64, 8, seed=9, device=device, kv_dtype="fp8")


def paged_decode(window=0, device="cpu", batch=256) -> DecodeCase:
    lens = uniform_lengths(batch, 1024, 32768, seed=4000)
    return make_decode("paged_decode" + ("_w%d" % window if window else ""),
                       lens, 64, 8, seed=4, window=window, sink_std=2.0,
                       paged=True, device=device)


def chunked_prefill(device="cpu", lq=4096, lk=131072) -> PrefillCase:
    return make_prefill("chunked_prefill", [lq], [lk], 64, 8, seed=5,
                        causal=True, device=device)


def long_context_prefill(device="cpu", lq=256, lk=131072) -> PrefillCase:
    return make_prefill("long_context_prefill", [lq], [lk], 64, 8, seed=8, causal=True,
                        device=device)


def paged_chunked_prefill(device="cpu", lq=4096, lk=131072) -> PrefillCase:
    return make_prefill_paged("paged_chunked_prefill", [lq], [lk], 64, 8, seed=6,
                              causal=True, device=device)


def paged_chunked_prefill_fp8(device="cpu", lq=4096, lk=131072) -> PrefillCase:
    return make_prefill_paged("paged_chunked_prefill_fp8", [lq], [lk], 64, 8, seed=12,
                              causal=True, device=device, kv_dtype="fp8")


def paged_prefill_batch(device="cpu", nseq=16) -> PrefillCase:
    new = uniform_lengths(nseq, 256, 2048, seed=6000)
    cached = uniform_lengths(nseq, 1024, 32768, seed=6001)
    return make_prefill_paged("paged_prefill_batch", new,
                              [n + c for n, c in zip(new, cached)], 64, 8, seed=7,
                              causal=True, device=device)


WORKLOADS = {
    "tiny_prefill": tiny_prefill,
    "decode_contig": decode_contig,
    "varlen_prefill": varlen_prefill,
    "paged_decode": paged_decode,
    "decode_contig_fp8": decode_contig_fp8,
    "decode_contig_d128": decode_contig_d128,
    "varlen_prefill_d128": varlen_prefill_d128,
    "varlen_prefill_g3": varlen_prefill_g3,
    "chunked_prefill": chunked_prefill,
    "long_context_prefill": long_context_prefill,
    "paged_chunked_prefill": paged_chunked_prefill,
    "paged_prefill_batch": paged_prefill_batch,
    "paged_chunked_prefill_fp8": paged_chunked_prefill_fp8,
}

"""Thin ctypes binding of libsinkattn.so (C ABI in include/sinkattn.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the launch stream, missing outputs/workspace are allocated with
torch. Every step of the computation runs in the library's CUDA kernels; there
is no fallback. If the library is missing or cannot be loaded, every call
raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsinkattn.so")

SINKATTN_OK = 0
SINKATTN_ERR_INVALID_ARGUMENT = 1
SINKATTN_ERR_UNSUPPORTED = 2
SINKATTN_ERR_WORKSPACE_TOO_SMALL = 3
SINKATTN_ERR_CUDA = 4
# size of the fixed scratch array behind sinkattn_decode_noalloc (as in the header)
SINKATTN_NOALLOC_SCRATCH_BYTES = 32 << 20

EXPORTED = (
    "sinkattn_status_string",
    "sinkattn_last_cuda_error",
    "sinkattn_prefill_workspace_size",
    "sinkattn_prefill",
    "sinkattn_prefill_paged_workspace_size",
    "sinkattn_prefill_paged",
    "sinkattn_prefill_backward_workspace_size",
    "sinkattn_prefill_backward",
    "sinkattn_decode_workspace_size",
    "sinkattn_decode",
    "sinkattn_decode_fp8",
    "sinkattn_decode_noalloc",
    "sinkattn_prefill_paged_fp8",
    "sinkattn_merge",
    "sinkattn_get_device_error",
    "sinkattn_debug_stall_waits",
)


class SinkAttnError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = "%s: %s (status %d)" % (what, _status_string(status), status)
        if status == SINKATTN_ERR_CUDA:
            try:
                msg += ": " + load().sinkattn_last_cuda_error().decode()
            except Exception:  # library missing: the status alone
                pass
        super().__init__(msg)


class Mask(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int), ("window", ctypes.c_int), ("scale", ctypes.c_float)]


_LIB = None


def load(path: str = LIB_PATH):
    """Load the library (once) and declare its signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError("libsinkattn.so not built at %s: run "
                           "`python -m attention_learned_sinks_gb300.build`" % path)
    lib = ctypes.CDLL(path)
    P, I, L, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.sinkattn_status_string.argtypes = [I]
    lib.sinkattn_status_string.restype = ctypes.c_char_p
    lib.sinkattn_last_cuda_error.argtypes = []
    lib.sinkattn_last_cuda_error.restype = ctypes.c_char_p
    lib.sinkattn_prefill_workspace_size.argtypes = [I, L, L, I, I, I, I, I, I, I]
    lib.sinkattn_prefill_workspace_size.restype = S
    lib.sinkattn_prefill.argtypes = [P, P, P, P, P, I, L, L, I, I, I, I, I, P, Mask, I,
                                     P, P, P, S, P]
    lib.sinkattn_prefill.restype = I
    lib.sinkattn_prefill_paged_workspace_size.argtypes = [I, L, I, I, I, I, I, I, I]
    lib.sinkattn_prefill_paged_workspace_size.restype = S
    lib.sinkattn_prefill_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, L, I, I, I, I, I, P,
                                           Mask, I, P, P, P, S, P]
    lib.sinkattn_prefill_paged.restype = I
    lib.sinkattn_prefill_paged_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, L, I, I, I,
                                               I, I, P, Mask, I, P, P, P, S, P]
    lib.sinkattn_prefill_paged_fp8.restype = I
    lib.sinkattn_prefill_backward_workspace_size.argtypes = [I, L, L, I, I, I]
    lib.sinkattn_prefill_backward_workspace_size.restype = S
    lib.sinkattn_prefill_backward.argtypes = [P, P, P, P, P, P, P, P, I, L, L, I, I, I, I, I, P,
                                              Mask, P, P, P, P, P, S, P]
    lib.sinkattn_prefill_backward.restype = I
    lib.sinkattn_decode_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.sinkattn_decode_workspace_size.restype = S
    lib.sinkattn_decode.argtypes = [P, P, P, P, P, P, L, I, I, I, I, I, I, I, P, Mask, I,
                                    P, P, P, S, P]
    lib.sinkattn_decode.restype = I
    lib.sinkattn_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, L, I, I, I, I, I, I, I, P, Mask,
                                        I, P, P, P, S, P]
    lib.sinkattn_decode_fp8.restype = I
    lib.sinkattn_decode_noalloc.argtypes = [P, P, P, P, P, P, L, I, I, I, I, I, I, I, P, Mask,
                                            I, P, P, P]
    lib.sinkattn_decode_noalloc.restype = I
    lib.sinkattn_merge.argtypes = [P, P, I, L, I, I, P, P, P, P]
    lib.sinkattn_merge.restype = I
    lib.sinkattn_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
    lib.sinkattn_get_device_error.restype = I
    lib.sinkattn_debug_stall_waits.argtypes = [ctypes.c_uint64]
    lib.sinkattn_debug_stall_waits.restype = I
    _LIB = lib
    return lib


def _status_string(status):
    try:
        return load().sinkattn_status_string(status).decode()
    except Exception:  # library missing: still report the number
        return "status"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != SINKATTN_OK:
        raise SinkAttnError(status, what)


def _req(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))


def sinkattn_prefill_workspace_size(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, hq,
                                    hkv, head_dim=64, window=0, num_splits=0):
    return load().sinkattn_prefill_workspace_size(int(batch), int(total_q), int(total_k),
                                                  int(max_seqlen_q), int(max_seqlen_k), hq, hkv,
                                                  head_dim, int(window), int(num_splits))


def sinkattn_decode_workspace_size(batch, max_seqlen_k, hq, hkv, head_dim=64, window=0,
                                   num_splits=0):
    return load().sinkattn_decode_workspace_size(batch, max_seqlen_k, hq, hkv, head_dim,
                                                 window, num_splits)


def sinkattn_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *,
                     sinks=None, causal=True, window=0, scale=None, num_splits=0, out=None,
                     lse=None, return_lse=True, workspace=None, total_q=None, total_k=None,
                     stream=None):
    """Sink-attention prefill over packed sequences. Returns (out, lse)."""
    lib = load()
    _req(q, torch.bfloat16, "q")
    _req(k, torch.bfloat16, "k")
    _req(v, torch.bfloat16, "v")
    _req(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _req(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=q.device)
    if sinks is not None:
        _req(sinks, torch.float32, "sinks")
    tk_ = tk if total_k is None else total_k
    tq_ = tq if total_q is None else total_q
    batch = cu_seqlens_q.numel() - 1
    if workspace is None:
        need = lib.sinkattn_prefill_workspace_size(batch, tq_, tk_, int(max_seqlen_q),
                                                   int(max_seqlen_k), hq, hkv, d, int(window),
                                                   int(num_splits))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask = Mask(1 if causal else 0, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                              batch, tq_, tk_, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
                              _ptr(sinks), mask, int(num_splits), _ptr(out), _ptr(lse),
                              _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sinkattn_prefill")
    return out, lse


def sinkattn_prefill_paged_workspace_size(batch, total_q, max_seqlen_q, max_seqlen_k, hq, hkv,
                                          head_dim=64, window=0, num_splits=0):
    return load().sinkattn_prefill_paged_workspace_size(int(batch), int(total_q),
                                                        int(max_seqlen_q), int(max_seqlen_k), hq,
                                                        hkv, head_dim, int(window),
                                                        int(num_splits))


def sinkattn_prefill_paged(q, cu_seqlens_q, k_cache, v_cache, block_table, seqlens_k,
                           max_seqlen_q, max_seqlen_k, *, sinks=None, causal=True, window=0,
                           scale=None, num_splits=0, out=None, lse=None, return_lse=True,
                           workspace=None, stream=None):
    """Sink-attention prefill of packed queries against a paged KV cache
    [num_pages, hkv, page_size, head_dim] addressed by block_table / seqlens_k.
    Returns (out, lse)."""
    lib = load()
    _req(q, torch.bfloat16, "q")
    _req(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _req(k_cache, torch.bfloat16, "k_cache")
    _req(v_cache, torch.bfloat16, "v_cache")
    _req(block_table, torch.int32, "block_table")
    _req(seqlens_k, torch.int32, "seqlens_k")
    tq, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_cache.shape
    batch = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=q.device)
    if sinks is not None:
        _req(sinks, torch.float32, "sinks")
    if workspace is None:
        need = lib.sinkattn_prefill_paged_workspace_size(batch, tq, int(max_seqlen_q),
                                                         int(max_seqlen_k), hq, hkv, d,
                                                         int(window), int(num_splits))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask = Mask(1 if causal else 0, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_prefill_paged(_ptr(q), _ptr(cu_seqlens_q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_table), _ptr(seqlens_k), num_pages,
                                    block_table.shape[1], page_size, batch, tq,
                                    int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
                                    _ptr(sinks), mask, int(num_splits), _ptr(out), _ptr(lse),
                                    _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sinkattn_prefill_paged")
    return out, lse


def sinkattn_prefill_paged_fp8(q, cu_seqlens_q, k_cache, v_cache, block_table, seqlens_k,
                               max_seqlen_q, max_seqlen_k, *, k_scale=None, v_scale=None,
                               sinks=None, causal=True, window=0, scale=None, num_splits=0,
                               out=None, lse=None, return_lse=True, workspace=None,
                               stream=None):
    """sinkattn_prefill_paged over an fp8 e4m3 cache: k_cache / v_cache hold
    uint8 codes [num_pages, hkv, page_size, head_dim]; k_scale / v_scale are
    float32 [hkv] (None = 1). Returns (out, lse)."""
    lib = load()
    _req(q, torch.bfloat16, "q")
    _req(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _req(k_cache, torch.uint8, "k_cache")
    _req(v_cache, torch.uint8, "v_cache")
    _req(block_table, torch.int32, "block_table")
    _req(seqlens_k, torch.int32, "seqlens_k")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale"), (sinks, "sinks")):
        if t is not None:
            _req(t, torch.float32, n)
    tq, hq, d = q.shape
    num_pages, hkv, page_size, _ = k_cache.shape
    batch = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = lib.sinkattn_prefill_paged_workspace_size(batch, tq, int(max_seqlen_q),
                                                         int(max_seqlen_k), hq, hkv, d,
                                                         int(window), int(num_splits))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask = Mask(1 if causal else 0, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_prefill_paged_fp8(_ptr(q), _ptr(cu_seqlens_q), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                        _ptr(block_table), _ptr(seqlens_k), num_pages,
                                        block_table.shape[1], page_size, batch, tq,
                                        int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
                                        _ptr(sinks), mask, int(num_splits), _ptr(out), _ptr(lse),
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sinkattn_prefill_paged_fp8")
    return out, lse


def sinkattn_prefill_backward_workspace_size(batch, total_q, total_k, hq, hkv, head_dim=64):
    return load().sinkattn_prefill_backward_workspace_size(int(batch), int(total_q),
                                                           int(total_k), hq, hkv, head_dim)


def sinkattn_prefill_backward(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                              max_seqlen_k, *, sinks=None, causal=True, window=0, scale=None,
                              dq=None, dk=None, dv=None, dsinks=None, workspace=None,
                              stream=None):
    """Gradients of sinkattn_prefill with respect to q, k, v and the sinks,
    given the forward's out and lse and the output gradient dout.
    Returns (dq, dk, dv, dsinks); dsinks is None without sinks."""
    lib = load()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _req(t, torch.bfloat16, name)
    _req(lse, torch.float32, "lse")
    _req(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _req(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    if sinks is not None:
        _req(sinks, torch.float32, "sinks")
        if dsinks is None:
            dsinks = torch.empty(hq, dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        need = lib.sinkattn_prefill_backward_workspace_size(batch, tq, tk, hq, hkv, d)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask = Mask(1 if causal else 0, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                       _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch,
                                       tq, tk, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
                                       _ptr(sinks), mask, _ptr(dq), _ptr(dk), _ptr(dv),
                                       _ptr(dsinks if sinks is not None else None),
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sinkattn_prefill_backward")
    return dq, dk, dv, (dsinks if sinks is not None else None)


def sinkattn_decode(q, k_cache, v_cache, *, kv_indptr=None, block_table=None, seqlens_k=None,
                    max_seqlen_k, sinks=None, window=0, scale=None, num_splits=0, out=None,
                    lse=None, return_lse=True, workspace=None, stream=None):
    """Sink-attention decode over a contiguous (kv_indptr) or paged
    (block_table + seqlens_k) KV cache. Returns (out, lse)."""
    lib = load()
    _req(q, torch.bfloat16, "q")
    _req(k_cache, torch.bfloat16, "k_cache")
    _req(v_cache, torch.bfloat16, "v_cache")
    batch, hq, d = q.shape
    hkv = k_cache.shape[1]
    if block_table is not None:
        _req(block_table, torch.int32, "block_table")
        _req(seqlens_k, torch.int32, "seqlens_k")
        kv_rows, page_size, max_pages = k_cache.shape[0], k_cache.shape[2], block_table.shape[1]
    else:
        _req(kv_indptr, torch.int32, "kv_indptr")
        kv_rows, page_size, max_pages = k_cache.shape[0], 0, 0
    if sinks is not None:
        _req(sinks, torch.float32, "sinks")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((batch, hq), dtype=torch.float32, device=q.device)
    need = lib.sinkattn_decode_workspace_size(batch, int(max_seqlen_k), hq, hkv, d, int(window),
                                              int(num_splits))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask = Mask(1, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_indptr),
                             _ptr(block_table), _ptr(seqlens_k), kv_rows, max_pages, page_size,
                             batch, int(max_seqlen_k), hq, hkv, d, _ptr(sinks), mask,
                             int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(st, "sinkattn_decode")
    return out, lse


def sinkattn_decode_fp8(q, k_cache, v_cache, *, k_scale=None, v_scale=None, kv_indptr=None,
                        block_table=None, seqlens_k=None, max_seqlen_k, sinks=None, window=0,
                        scale=None, num_splits=0, out=None, lse=None, return_lse=True,
                        workspace=None, stream=None):
    """sinkattn_decode over an fp8 e4m3 cache (uint8 codes, same layouts) with
    optional per-KV-head scales. Returns (out, lse)."""
    lib = load()
    _req(q, torch.bfloat16, "q")
    _req(k_cache, torch.uint8, "k_cache")
    _req(v_cache, torch.uint8, "v_cache")
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale"), (sinks, "sinks")):
        if t is not None:
            _req(t, torch.float32, name)
    batch, hq, d = q.shape
    hkv = k_cache.shape[1]
    if block_table is not None:
        _req(block_table, torch.int32, "block_table")
        _req(seqlens_k, torch.int32, "seqlens_k")
        kv_rows, page_size, max_pages = k_cache.shape[0], k_cache.shape[2], block_table.shape[1]
    else:
        _req(kv_indptr, torch.int32, "kv_indptr")
        kv_rows, page_size, max_pages = k_cache.shape[0], 0, 0
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((batch, hq), dtype=torch.float32, device=q.device)
    need = lib.sinkattn_decode_workspace_size(batch, int(max_seqlen_k), hq, hkv, d, int(window),
                                              int(num_splits))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask = Mask(1, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                 _ptr(v_scale), _ptr(kv_indptr), _ptr(block_table),
                                 _ptr(seqlens_k), kv_rows, max_pages, page_size, batch,
                                 int(max_seqlen_k), hq, hkv, d, _ptr(sinks), mask,
                                 int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(st, "sinkattn_decode_fp8")
    return out, lse


def sinkattn_decode_noalloc(q, k_cache, v_cache, *, kv_indptr=None, block_table=None,
                            seqlens_k=None, max_seqlen_k, sinks=None, window=0, scale=None,
                            num_splits=0, out, lse=None, stream=None):
    """sinkattn_decode without a workspace: the library's fixed scratch array is
    used instead (for callers that may not allocate device memory). `out` (and
    `lse`, if wanted) must be given; nothing is allocated here."""
    lib = load()
    batch, hq, d = q.shape
    hkv = k_cache.shape[1]
    if block_table is not None:
        kv_rows, page_size, max_pages = k_cache.shape[0], k_cache.shape[2], block_table.shape[1]
    else:
        kv_rows, page_size, max_pages = k_cache.shape[0], 0, 0
    mask = Mask(1, int(window), float(d ** -0.5 if scale is None else scale))
    st = lib.sinkattn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_indptr),
                                     _ptr(block_table), _ptr(seqlens_k), kv_rows, max_pages,
                                     page_size, batch, int(max_seqlen_k), hq, hkv, d, _ptr(sinks),
                                     mask, int(num_splits), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "sinkattn_decode_noalloc")
    return out, lse


def sinkattn_merge(partial_o, partial_lse, *, sinks=None, out=None, lse=None, return_lse=True,
                   stream=None):
    """Merge split-KV partials [S, rows, hq, D] / [S, rows, hq] by log-sum-exp (D 64 or 128)."""
    lib = load()
    _req(partial_o, torch.float32, "partial_o")
    _req(partial_lse, torch.float32, "partial_lse")
    ns, rows, hq, d = partial_o.shape
    if out is None:
        out = torch.empty((rows, hq, d), dtype=torch.bfloat16, device=partial_o.device)
    if lse is None and return_lse:
        lse = torch.empty((rows, hq), dtype=torch.float32, device=partial_o.device)
    if sinks is not None:
        _req(sinks, torch.float32, "sinks")
    st = lib.sinkattn_merge(_ptr(partial_o), _ptr(partial_lse), ns, rows, hq, d, _ptr(sinks),
                            _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "sinkattn_merge")
    return out, lse


def sinkattn_get_device_error(stream=None) -> int:
    """Synchronise, read and clear the device error word (0 = no error)."""
    code = ctypes.c_int(0)
    _check(load().sinkattn_get_device_error(_stream(stream), ctypes.byref(code)),
           "sinkattn_get_device_error")
    return code.value


def sinkattn_debug_stall_waits(limit_ns: int) -> None:
    """Testing hook: later prefill / backward calls make one wait of at most
    limit_ns on a barrier nothing completes, so every CTA takes its timeout
    path (0 turns it off)."""
    _check(load().sinkattn_debug_stall_waits(int(limit_ns)), "sinkattn_debug_stall_waits")

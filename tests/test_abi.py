"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/sinkattn.h declares, and rejects bad arguments before
it touches the device (all cases below return before any CUDA call)."""
import ctypes
import os
import re

import pytest

import attention_learned_sinks_gb300 as sa
from attention_learned_sinks_gb300 import build as sbuild
from attention_learned_sinks_gb300 import sinkattn as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sbuild.build()
    return sa.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sinkattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sinkattn_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(B.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(5):
        assert lib.sinkattn_status_string(code)
    assert lib.sinkattn_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: every call below fails validation
M = B.Mask(1, 0, 0.125)


def prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cuq=FAKE, cuk=FAKE, batch=2, tq=10, tk=10, mq=5, mk=5,
             hq=8, hkv=2, d=64, sinks=None, mask=M, ns=0, out=FAKE, lse=None)
    a.update(kw)
    return lib.sinkattn_prefill(a["q"], a["k"], a["v"], a["cuq"], a["cuk"], a["batch"], a["tq"],
                                a["tk"], a["mq"], a["mk"], a["hq"], a["hkv"], a["d"], a["sinks"],
                                a["mask"], a["ns"], a["out"], a["lse"], a.get("ws"),
                                a.get("wsb", 0), None)


def decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, indptr=FAKE, table=None, seqlens=None, rows=100, maxp=0,
             page=0, batch=2, mk=50, hq=8, hkv=2, d=64, sinks=None, mask=M, ns=0, out=FAKE,
             lse=None, ws=None, wsb=0)
    a.update(kw)
    return lib.sinkattn_decode(a["q"], a["k"], a["v"], a["indptr"], a["table"], a["seqlens"],
                               a["rows"], a["maxp"], a["page"], a["batch"], a["mk"], a["hq"],
                               a["hkv"], a["d"], a["sinks"], a["mask"], a["ns"], a["out"],
                               a["lse"], a["ws"], a["wsb"], None)


def test_prefill_rejects_bad_arguments(lib):
    assert prefill(lib, d=96) == B.SINKATTN_ERR_UNSUPPORTED
    assert prefill(lib, d=256) == B.SINKATTN_ERR_UNSUPPORTED
    assert prefill(lib, hq=6, hkv=4) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, hkv=0) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, mask=B.Mask(1, 0, 0.0)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, mask=B.Mask(1, -1, 0.1)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, mask=B.Mask(1, 0, float("nan"))) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, q=None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, out=ctypes.c_void_p((1 << 20) + 2)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, batch=-1) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill(lib, ns=-1) == B.SINKATTN_ERR_INVALID_ARGUMENT
    need = lib.sinkattn_prefill_workspace_size(2, 10, 10, 5, 5, 8, 2, 64, 0, 0)
    assert need >= 10 * 2 * 64 * 2
    assert prefill(lib) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert prefill(lib, ws=FAKE, wsb=need - 1) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert prefill(lib, ws=ctypes.c_void_p((1 << 20) + 16), wsb=need) == \
        B.SINKATTN_ERR_INVALID_ARGUMENT
    # nothing to do: returns before any launch
    assert prefill(lib, batch=0) == B.SINKATTN_OK
    assert prefill(lib, tq=0) == B.SINKATTN_OK
    # head_dim 128 is accepted and needs twice the V copy
    need128 = lib.sinkattn_prefill_workspace_size(2, 10, 10, 5, 5, 8, 2, 128, 0, 0)
    assert need128 >= 10 * 2 * 128 * 2 and need128 > need
    assert prefill(lib, d=128, ws=FAKE, wsb=need) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert prefill(lib, d=128, batch=0) == B.SINKATTN_OK


def prefill_paged(lib, **kw):
    a = dict(q=FAKE, cuq=FAKE, k=FAKE, v=FAKE, table=FAKE, seqlens=FAKE, npages=8, maxp=4,
             page=16, batch=2, tq=10, mq=5, mk=64, hq=8, hkv=2, d=64, sinks=None, mask=M, ns=0,
             out=FAKE, lse=None)
    a.update(kw)
    return lib.sinkattn_prefill_paged(a["q"], a["cuq"], a["k"], a["v"], a["table"], a["seqlens"],
                                      a["npages"], a["maxp"], a["page"], a["batch"], a["tq"],
                                      a["mq"], a["mk"], a["hq"], a["hkv"], a["d"], a["sinks"],
                                      a["mask"], a["ns"], a["out"], a["lse"], a.get("ws"),
                                      a.get("wsb", 0), None)


def test_prefill_paged_rejects_bad_arguments(lib):
    assert prefill_paged(lib, d=80) == B.SINKATTN_ERR_UNSUPPORTED
    assert prefill_paged(lib, hq=6, hkv=4) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, page=0) == B.SINKATTN_ERR_INVALID_ARGUMENT
    # the block table must be able to address max_seqlen_k keys
    assert prefill_paged(lib, mk=65) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, table=None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, seqlens=None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, npages=0) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, k=ctypes.c_void_p((1 << 20) + 8)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, mask=B.Mask(0, -3, 0.1)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, ns=-2) == B.SINKATTN_ERR_INVALID_ARGUMENT
    need = lib.sinkattn_prefill_paged_workspace_size(2, 10, 5, 64, 8, 2, 64, 0, 0)
    # K and V staging for batch * max_seqlen_k rows plus a 128-row tail
    assert need >= 2 * (2 * 64 + 128) * 2 * 64 * 2
    assert prefill_paged(lib) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert prefill_paged(lib, ws=FAKE, wsb=need - 1) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert prefill_paged(lib, ws=ctypes.c_void_p((1 << 20) + 16), wsb=need) == \
        B.SINKATTN_ERR_INVALID_ARGUMENT
    assert prefill_paged(lib, batch=0) == B.SINKATTN_OK
    assert prefill_paged(lib, tq=0) == B.SINKATTN_OK
    assert lib.sinkattn_prefill_paged_workspace_size(2, 10, 5, 64, 8, 2, 96, 0, 0) == 0
    assert lib.sinkattn_prefill_paged_workspace_size(2, 10, 5, 128, 8, 2, 64, 0, 0) > need
    need128 = lib.sinkattn_prefill_paged_workspace_size(2, 10, 5, 64, 8, 2, 128, 0, 0)
    assert need128 >= 2 * (2 * 64 + 128) * 2 * 128 * 2
    assert prefill_paged(lib, d=128, ws=FAKE, wsb=need) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL


def test_prefill_paged_fp8_rejects_bad_arguments(lib):
    def f(**kw):
        a = dict(q=FAKE, cuq=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, table=FAKE, seqlens=FAKE,
                 npages=8, maxp=4, page=16, batch=2, tq=10, mq=5, mk=64, hq=8, hkv=2, d=64,
                 sinks=None, mask=M, ns=0, out=FAKE, lse=None, ws=None, wsb=0)
        a.update(kw)
        return lib.sinkattn_prefill_paged_fp8(
            a["q"], a["cuq"], a["k"], a["v"], a["ks"], a["vs"], a["table"], a["seqlens"],
            a["npages"], a["maxp"], a["page"], a["batch"], a["tq"], a["mq"], a["mk"], a["hq"],
            a["hkv"], a["d"], a["sinks"], a["mask"], a["ns"], a["out"], a["lse"], a["ws"],
            a["wsb"], None)
    assert f(d=96) == B.SINKATTN_ERR_UNSUPPORTED
    assert f(hq=6, hkv=4) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert f(ks=ctypes.c_void_p((1 << 20) + 2)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert f(mk=65) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert f() == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert f(ks=FAKE, vs=FAKE) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert f(batch=0) == B.SINKATTN_OK


def backward(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, dout=FAKE, lse=FAKE, cuq=FAKE, cuk=FAKE, batch=2,
             tq=10, tk=10, mq=5, mk=5, hq=8, hkv=2, d=64, sinks=None, mask=M, dq=FAKE, dk=FAKE,
             dv=FAKE, dsinks=None)
    a.update(kw)
    return lib.sinkattn_prefill_backward(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"],
                                         a["cuq"], a["cuk"], a["batch"], a["tq"], a["tk"],
                                         a["mq"], a["mk"], a["hq"], a["hkv"], a["d"], a["sinks"],
                                         a["mask"], a["dq"], a["dk"], a["dv"], a["dsinks"],
                                         a.get("ws"), a.get("wsb", 0), None)


def test_backward_rejects_bad_arguments(lib):
    assert backward(lib, d=96) == B.SINKATTN_ERR_UNSUPPORTED
    # head_dim 128 is accepted; its workspace holds twice the fp16 copies
    need64 = lib.sinkattn_prefill_backward_workspace_size(2, 10, 10, 8, 2, 64)
    need128 = lib.sinkattn_prefill_backward_workspace_size(2, 10, 10, 8, 2, 128)
    assert need128 > need64 and lib.sinkattn_prefill_backward_workspace_size(2, 10, 10, 8, 2, 96) == 0
    assert backward(lib, d=128, batch=0) == B.SINKATTN_OK
    assert backward(lib, hq=6, hkv=4) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert backward(lib, lse=None) == B.SINKATTN_ERR_INVALID_ARGUMENT   # lse is required
    assert backward(lib, out=None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert backward(lib, dv=ctypes.c_void_p((1 << 20) + 4)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert backward(lib, mask=B.Mask(1, 0, -2.0)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    need = lib.sinkattn_prefill_backward_workspace_size(2, 10, 10, 8, 2, 64)
    # fp16 copies of q, dout (10 x 8 x 64) and k, v (10 x 2 x 64), two fp32 per (row, head)
    assert need >= 2 * 10 * 8 * 128 + 2 * 10 * 2 * 128 + 2 * 10 * 8 * 4
    assert backward(lib) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert backward(lib, ws=FAKE, wsb=need - 1) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert backward(lib, ws=ctypes.c_void_p((1 << 20) + 64), wsb=need) == \
        B.SINKATTN_ERR_INVALID_ARGUMENT
    assert backward(lib, batch=0) == B.SINKATTN_OK
    assert backward(lib, tq=0, tk=0) == B.SINKATTN_OK
    assert lib.sinkattn_prefill_backward_workspace_size(2, 10, 10, 8, 2, 96) == 0


def test_decode_rejects_bad_arguments(lib):
    assert decode(lib, d=80) == B.SINKATTN_ERR_UNSUPPORTED
    # groups above 8 run in tiles of 8 query heads, each with its own counter
    n16 = lib.sinkattn_decode_workspace_size(2, 5000, 32, 2, 64, 0, 0)
    n8 = lib.sinkattn_decode_workspace_size(2, 5000, 16, 2, 64, 0, 0)
    assert n16 > n8 > 0
    assert decode(lib, hq=32, hkv=2, batch=0) == B.SINKATTN_OK
    assert decode(lib, hq=9, hkv=2) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert decode(lib, table=FAKE, seqlens=FAKE, page=16, maxp=4) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert decode(lib, indptr=None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert decode(lib, indptr=None, table=FAKE, seqlens=None, page=16, maxp=4) == \
        B.SINKATTN_ERR_INVALID_ARGUMENT
    assert decode(lib, seqlens=FAKE) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert decode(lib, ns=-1) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert decode(lib, mask=B.Mask(1, 0, -1.0)) == B.SINKATTN_ERR_INVALID_ARGUMENT
    # long contexts are split: the workspace must be big enough
    need = lib.sinkattn_decode_workspace_size(2, 5000, 8, 2, 64, 0, 0)
    assert need > 0
    assert decode(lib, mk=5000, ws=None, wsb=0) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert decode(lib, mk=5000, ws=FAKE, wsb=need - 1) == B.SINKATTN_ERR_WORKSPACE_TOO_SMALL
    assert decode(lib, batch=0) == B.SINKATTN_OK


def test_merge_rejects_bad_arguments(lib):
    f = lib.sinkattn_merge
    assert f(FAKE, FAKE, 2, 4, 8, 32, None, FAKE, None, None) == B.SINKATTN_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, 2, 0, 8, 128, None, FAKE, None, None) == B.SINKATTN_OK
    assert f(None, FAKE, 2, 4, 8, 64, None, FAKE, None, None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert f(FAKE, FAKE, -1, 4, 8, 64, None, FAKE, None, None) == B.SINKATTN_ERR_INVALID_ARGUMENT
    assert f(FAKE, FAKE, 2, 0, 8, 64, None, FAKE, None, None) == B.SINKATTN_OK


def test_workspace_sizes_follow_the_split_plan(lib):
    ws = lambda b, mk, w=0, ns=0: lib.sinkattn_decode_workspace_size(b, mk, 64, 8, 64, w, ns)
    assert ws(64, 8192, ns=16) >= 16 * 64 * 64 * 64 * 4    # 16 blocks of 512
    assert ws(64, 8192) > 0
    assert ws(64, 8192, ns=2) < ws(64, 8192, ns=16)
    assert ws(64, 8192, w=128) < ws(64, 8192)               # window: one block
    assert lib.sinkattn_decode_workspace_size(0, 10, 8, 2, 64, 0, 0) == 0
    pws = lambda *a: lib.sinkattn_prefill_workspace_size(*a)
    assert pws(3, 1000, 1000, 500, 500, 64, 8, 64, 0, 1) >= 1000 * 8 * 64 * 2 + 256
    assert pws(3, 1000, 1000, 500, 500, 64, 8, 96, 0, 1) == 0
    assert pws(3, 1000, 1000, 500, 500, 64, 8, 128, 0, 1) >= 1000 * 8 * 128 * 2 + 256
    assert pws(3, 1000, 1000, 500, 500, 64, 8, 64, -1, 0) == 0
    # explicit splits add fp32 partials: splits * total_q * hq * (64 + 1) * 4 bytes
    one = pws(3, 1000, 1000, 500, 500, 64, 8, 64, 0, 1)
    assert pws(3, 1000, 1000, 500, 500, 64, 8, 64, 0, 4) >= one + 4 * 1000 * 64 * 260
    # automatic: a few hundred queries over a long context are split ...
    long_ctx = pws(1, 256, 131072, 256, 131072, 64, 8, 64, 0, 0)
    assert long_ctx > pws(1, 256, 131072, 256, 131072, 64, 8, 64, 0, 1)
    # ... many query tiles or short contexts are not
    assert pws(1, 4096, 131072, 4096, 131072, 64, 8, 64, 0, 0) == \
        pws(1, 4096, 131072, 4096, 131072, 64, 8, 64, 0, 1)
    assert pws(1, 256, 2048, 256, 2048, 64, 8, 64, 0, 0) == \
        pws(1, 256, 2048, 256, 2048, 64, 8, 64, 0, 1)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "_LIB", None)
    with pytest.raises(RuntimeError):
        B.load(str(tmp_path / "missing.so"))

"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/pgd.h declares, and rejects bad arguments on the host before any CUDA
call."""
import ctypes
import os
import re

import pytest

import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgd.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pgd_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from paged_gqa_decode_kv_gb300 import build
    build.build()
    return pgd.lib()


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("pgd_kv_append", "pgd_paged_decode_attention", "pgd_attention_workspace_size",
              "pgd_alloc_create", "pgd_copy_blocks", "pgd_decode_step"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_symbols() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_symbols()) <= set(_native.SIGNATURES)


def test_status_strings(L):
    for s in range(7):
        assert L.pgd_status_string(s)
    assert L.pgd_version() >= 100


def _attn(L, **kw):
    a = dict(out=16, q=16, k=16, v=16, t=16, c=16, B=2, n_q=8, n_kv=2, d=128, bs=16, MB=4, NB=8,
             scale=0.1, splits=0, ws=None, wsb=0)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.pgd_paged_decode_attention(P(a["out"]), P(a["q"]), P(a["k"]), P(a["v"]), P(a["t"]),
                                        P(a["c"]), a["B"], a["n_q"], a["n_kv"], a["d"], a["bs"],
                                        a["MB"], a["NB"], a["scale"], a["splits"], P(a["ws"]),
                                        a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=64), _native.ERR_UNSUPPORTED),
    (dict(bs=8), _native.ERR_UNSUPPORTED),
    (dict(n_q=6, n_kv=2), _native.ERR_UNSUPPORTED),      # G = 3
    (dict(n_q=32, n_kv=2), _native.ERR_UNSUPPORTED),     # G = 16
    (dict(n_q=7, n_kv=2), _native.ERR_INVALID_ARG),
    (dict(B=-1), _native.ERR_INVALID_ARG),
    (dict(B=5000), _native.ERR_UNSUPPORTED),
    (dict(B=2049), _native.ERR_UNSUPPORTED),              # one past PGD_MAX_BATCH
    (dict(scale=0.0), _native.ERR_INVALID_ARG),
    (dict(scale=float("inf")), _native.ERR_INVALID_ARG),
    (dict(q=None), _native.ERR_INVALID_ARG),
    (dict(q=24), _native.ERR_INVALID_ARG),                # misaligned
    (dict(NB=0), _native.ERR_INVALID_ARG),
    (dict(splits=-1), _native.ERR_INVALID_ARG),
    (dict(ws=None, wsb=0), _native.ERR_WORKSPACE),
    (dict(ws=256, wsb=16), _native.ERR_WORKSPACE),
    (dict(ws=264, wsb=1 << 30), _native.ERR_WORKSPACE),   # misaligned workspace
])
def test_attention_rejects_on_host(L, kw, status):
    assert _attn(L, **kw) == status
    assert L.pgd_last_error_detail()


def _attn_noalloc(L, **kw):
    a = dict(out=16, q=16, k=16, v=16, t=16, c=16, B=2, n_q=8, n_kv=2, d=128, bs=16, MB=4, NB=8,
             scale=0.1, splits=0)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.pgd_paged_decode_attention_noalloc(P(a["out"]), P(a["q"]), P(a["k"]), P(a["v"]),
                                                P(a["t"]), P(a["c"]), a["B"], a["n_q"], a["n_kv"],
                                                a["d"], a["bs"], a["MB"], a["NB"], a["scale"],
                                                a["splits"], None)


@pytest.mark.parametrize("kw", [
    dict(d=64), dict(bs=8), dict(n_q=6, n_kv=2), dict(n_q=32, n_kv=2), dict(n_q=7, n_kv=2),
    dict(B=-1), dict(B=5000), dict(scale=0.0), dict(scale=float("inf")), dict(q=None),
    dict(q=24), dict(out=None), dict(t=18), dict(NB=0), dict(splits=-1),
], ids=lambda kw: "-".join("%s=%s" % i for i in kw.items()))
def test_noalloc_rejects_like_the_regular_entry_point(L, kw):
    """Every argument set the workspace entry point refuses on the host is
    refused by the allocation-free one with the same status, before it looks
    up, clears or sizes its scratch (no CUDA call is made here: there is no
    GPU)."""
    want = _attn(L, ws=256, wsb=1 << 30, **kw)
    assert want != 0
    assert _attn_noalloc(L, **kw) == want
    assert L.pgd_last_error_detail()


def test_noalloc_empty_batch_is_a_noop(L):
    assert _attn_noalloc(L, B=0, out=None, q=None, k=None, v=None, t=None, c=None) == 0


def test_empty_batch_is_a_noop(L):
    assert _attn(L, B=0, out=None, q=None, k=None, v=None, t=None, c=None) == 0


def test_kv_append_rejects_on_host(L):
    P = ctypes.c_void_p
    assert L.pgd_kv_append(P(16), P(16), P(16), P(16), P(16), P(16), 2, 2, 64, 16, 4, 8,
                           None) == _native.ERR_UNSUPPORTED
    assert L.pgd_kv_append(P(16), P(16), P(16), P(16), P(16), P(16), 2, 2, 128, 12, 4, 8,
                           None) == _native.ERR_UNSUPPORTED
    assert L.pgd_kv_append(None, P(16), P(16), P(16), P(16), P(16), 2, 2, 128, 16, 4, 8,
                           None) == _native.ERR_INVALID_ARG
    assert L.pgd_kv_append(P(18), P(16), P(16), P(16), P(16), P(16), 2, 2, 128, 16, 4, 8,
                           None) == _native.ERR_INVALID_ARG
    assert L.pgd_kv_append(None, None, None, None, None, None, 0, 2, 128, 16, 4, 8, None) == 0


def test_workspace_size_grows_with_splits(L):
    assert pgd.workspace_size(16, 32, 8, 0) > 0
    a = pgd.workspace_size(16, 32, 8, 1)
    b = pgd.workspace_size(16, 32, 8, 64)
    assert 0 < a < b
    assert pgd.workspace_size(16, 32, 8, 0, d=64) == 0


def test_read_stream_rejects_on_host(L):
    P = ctypes.c_void_p
    assert L.pgd_read_stream(P(16), 4096, 2, None) == _native.ERR_INVALID_ARG   # mode
    assert L.pgd_read_stream(None, 4096, 0, None) == _native.ERR_INVALID_ARG
    assert L.pgd_read_stream(P(24), 4096, 0, None) == _native.ERR_INVALID_ARG   # misaligned
    assert L.pgd_read_stream(P(16), 40, 0, None) == _native.ERR_INVALID_ARG     # not 16 B units
    assert L.pgd_read_stream(P(16), 8192 + 16, 1, None) == _native.ERR_INVALID_ARG  # not 4 KiB
    assert L.pgd_read_stream(None, 0, 1, None) == 0                              # no-op


def test_wait_limit_setting(L):
    """The bounded waits' limit: 4 s by default, set and restored process-wide
    (a host-side setting; no GPU call)."""
    assert pgd.wait_limit_ns() == 4_000_000_000
    try:
        pgd.set_wait_limit_ns(1234)
        assert pgd.wait_limit_ns() == 1234
    finally:
        pgd.set_wait_limit_ns(0)
    assert pgd.wait_limit_ns() == 4_000_000_000


def test_short_context_setting(L):
    prev = pgd.set_short_context_tokens(256)
    try:
        assert prev == 1024
        assert pgd.set_short_context_tokens(0) == 256
    finally:
        pgd.set_short_context_tokens(-1)
    assert pgd.set_short_context_tokens(-1) == 1024
    assert pgd.uses_short_path(8, 8, 16, 40) and not pgd.uses_short_path(8, 8, 16, 41)
    assert not pgd.uses_short_path(9, 8, 16, 8) and not pgd.uses_short_path(1, 8, 16, 65)


def test_prepare_checks_arguments_on_the_host(L):
    """pgd.prepare runs the binding's checks once, before any C call: a CPU
    tensor, a wrong dtype or an unknown operation are refused at once."""
    import torch
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16)
    pool = torch.zeros(2, 2, 2, 16, 8, 8, dtype=torch.bfloat16)
    tables = torch.zeros(1, 1, dtype=torch.int32)
    lens = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        pgd.prepare("paged_decode_attention", None, q, pool, pool, tables, lens, 0.1,
                    workspace=torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(TypeError):
        pgd.prepare("paged_decode_attention", None, q.float(), pool, pool, tables, lens, 0.1)
    with pytest.raises(ValueError):
        pgd.prepare("no_such_call")


def _verify_call(L, fn, **kw):
    a = dict(out=16, q=16, kn=16, vn=16, k=16, v=16, t=16, c=16, B=2, T=2, n_q=8, n_kv=2,
             d=128, bs=16, MB=4, NB=8, scale=0.1, splits=0, ws=None, wsb=0)
    a.update(kw)
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    if fn == "append_verify":
        return L.pgd_append_verify_attention(
            P(a["out"]), P(a["q"]), P(a["kn"]), P(a["vn"]), P(a["k"]), P(a["v"]), P(a["t"]),
            P(a["c"]), a["B"], a["T"], a["n_q"], a["n_kv"], a["d"], a["bs"], a["MB"], a["NB"],
            a["scale"], a["splits"], P(a["ws"]), a["wsb"], None)
    # verify_step: host buffers 32 bytes apart from the device ones
    h = lambda x: None if x is None else x + 4096
    return L.pgd_verify_step(
        P(h(a["out"])), P(h(a["q"])), P(h(a["kn"])), P(h(a["vn"])), P(h(a["c"])), P(a["out"]),
        P(a["q"]), P(a["kn"]), P(a["vn"]), P(a["c"]), P(a["k"]), P(a["v"]), P(a["t"]), a["B"],
        a["T"], a["n_q"], a["n_kv"], a["d"], a["bs"], a["MB"], a["NB"], a["scale"], a["splits"],
        P(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("fn", ["append_verify", "verify_step"])
@pytest.mark.parametrize("kw,status", [
    (dict(T=0), _native.ERR_INVALID_ARG),
    (dict(T=5, n_q=8, n_kv=2), _native.ERR_UNSUPPORTED),   # 20 query rows per KV head
    (dict(d=64), _native.ERR_UNSUPPORTED),
    (dict(q=None), _native.ERR_INVALID_ARG),
    (dict(kn=None), _native.ERR_INVALID_ARG),
    (dict(vn=24), _native.ERR_INVALID_ARG),                 # misaligned
    (dict(B=0, out=None, q=None, kn=None, vn=None, k=None, v=None, t=None, c=None), 0),
])
def test_verify_step_calls_reject_on_host(L, fn, kw, status):
    """The one-call and host-buffer verify steps run their checks before any
    copy or launch (no CUDA call is made here: there is no GPU)."""
    assert _verify_call(L, fn, **kw) == status
    if status:
        assert L.pgd_last_error_detail()


def test_verify_step_rejects_null_host_buffers(L):
    P = ctypes.c_void_p
    args = [P(16)] * 13 + [2, 2, 8, 2, 128, 16, 4, 8, 0.1, 0, None, 0, None]
    for i in range(5):  # out_h, q_h, k_new_h, v_new_h, context_lens_h
        a = list(args)
        a[i] = None
        assert L.pgd_verify_step(*a) == _native.ERR_INVALID_ARG


def test_mla_step_rejects_on_host(L):
    P = ctypes.c_void_p
    def call(d=576, bs=32, c_new_d=16, B=2):
        return L.pgd_mla_step(P(4112), P(4112), P(4112), P(4112), P(16), P(16),
                              None if c_new_d is None else P(c_new_d), P(16), P(16), P(16), B,
                              16, d, 512, bs, 4, 8, 0.1, 0, None, 0, None)
    assert call(d=512) == _native.ERR_UNSUPPORTED
    assert call(bs=8) == _native.ERR_UNSUPPORTED
    assert call(c_new_d=None) == _native.ERR_INVALID_ARG
    assert call(c_new_d=24) == _native.ERR_INVALID_ARG
    assert call(B=-1) == _native.ERR_INVALID_ARG

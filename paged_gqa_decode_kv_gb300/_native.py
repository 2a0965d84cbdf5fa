"""ctypes binding of libpgd (include/pgd.h).  Argument marshalling only: every
step of the path runs in the library's CUDA kernels; there is no fallback.
The library is loaded on first use and a missing build is an error."""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

import torch

from . import build as _build

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

HEAD_DIM = 128

# status codes (pgd_status)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OUT_OF_BLOCKS, ERR_WORKSPACE, ERR_CUDA, \
    ERR_BLOCK_STATE = range(7)
# device error bits (PGD_DEVERR_*)
DEVERR_BAD_BLOCK_ID, DEVERR_BAD_CONTEXT, DEVERR_BAD_POSITION, DEVERR_TIMEOUT = 1, 2, 4, 8

#: every symbol include/pgd.h declares, with (argtypes, restype)
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "pgd_status_string": ([_I], ctypes.c_char_p),
    "pgd_last_error_detail": ([], ctypes.c_char_p),
    "pgd_version": ([], _I),
    "pgd_kv_append": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "pgd_attention_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "pgd_paged_decode_attention": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                    _P, _Z, _P], _I),
    "pgd_attention_grid": ([_I, _I, _I, _I, _I], _I),
    "pgd_paged_decode_attention_noalloc": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                            _F, _I, _P], _I),
    "pgd_append_decode_attention": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     _F, _I, _P, _Z, _P], _I),
    "pgd_kv_append_tokens": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P], _I),
    "pgd_verify_workspace_size": ([_I, _I, _I, _I, _I, _I], _Z),
    "pgd_paged_verify_attention": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                    _I, _P, _Z, _P], _I),
    "pgd_append_verify_attention": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     _I, _F, _I, _P, _Z, _P], _I),
    "pgd_verify_step": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                         _I, _I, _I, _F, _I, _P, _Z, _P], _I),
    "pgd_mla_workspace_size": ([_I, _I, _I], _Z),
    "pgd_mla_append": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "pgd_mla_decode_attention": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z,
                                  _P], _I),
    "pgd_mla_append_decode_attention": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                         _I, _P, _Z, _P], _I),
    "pgd_mla_step": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                      _P, _Z, _P], _I),
    "pgd_cascade_workspace_size": ([_I, _I, _I, _I, _I, _I, _I, _I], _Z),
    "pgd_cascade_decode_attention": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                      _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P], _I),
    "pgd_kv_append_fp8": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "pgd_paged_decode_attention_fp8": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                        _I, _P, _Z, _P], _I),
    "pgd_append_decode_attention_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                         _I, _F, _I, _P, _Z, _P], _I),
    "pgd_decode_step": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                         _I, _I, _F, _I, _P, _Z, _P], _I),
    "pgd_decode_step_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                             _I, _I, _I, _F, _I, _P, _Z, _P], _I),
    "pgd_copy_blocks": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "pgd_device_errors": ([_P, _I, _P], _I),
    "pgd_read_stream": ([_P, _Z, _I, _P], _I),
    "pgd_set_wait_limit_ns": ([ctypes.c_uint64], None),
    "pgd_wait_limit_ns": ([], ctypes.c_uint64),
    "pgd_set_short_context_tokens": ([_I], _I),
    "pgd_short_path": ([_I, _I, _I, _I, _I], _I),
    "pgd_alloc_create": ([_I, _P], _I),
    "pgd_alloc_destroy": ([_P], None),
    "pgd_alloc_allocate": ([_P, _I, _P], _I),
    "pgd_alloc_share": ([_P, _P, _I], _I),
    "pgd_alloc_release": ([_P, _P, _I], _I),
    "pgd_alloc_refcount": ([_P, _I], _I),
    "pgd_alloc_num_free": ([_P], _I),
    "pgd_alloc_num_blocks": ([_P], _I),
    "pgd_alloc_append_slot": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "pgd_alloc_fork": ([_P, _P, _I, _I, _P, _I], _I),
    "pgd_validate_tables": ([_P, _P, _I, _I, _I, _I], _I),
}


class PGDError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__("pgd status %d: %s" % (status, detail))
        self.status = status
        self.detail = detail


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libpgd.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    "libpgd.so is not built (%s); run paged_gqa_decode_kv_gb300.build.build() "
                    "or __graft_entry__.build()" % path)
            L = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
        return _lib


def _check(status: int) -> None:
    if status != OK:
        L = lib()
        raise PGDError(status, "%s: %s" % (L.pgd_status_string(status).decode(),
                                           L.pgd_last_error_detail().decode()))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype: torch.dtype, name: str, cuda: bool = True) -> None:
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if cuda and not t.is_cuda:
        raise ValueError("%s must be on a CUDA device" % name)


def _cache_dims(k_cache: torch.Tensor) -> Tuple[int, int, int, int]:
    """(NB, n_kv, bs, d) of a pool [NB][n_kv][bs/8][d/8][8][8] (each (block,
    head) tile stored as 8x8 core matrices)."""
    if k_cache.dim() != 6 or tuple(k_cache.shape[4:]) != (8, 8):
        raise ValueError("cache must be [NB][n_kv][bs/8][d/8][8][8]")
    NB, n_kv, rg, nc = k_cache.shape[:4]
    return NB, n_kv, rg * 8, nc * 8


# --------------------------------------------------------------------- GPU ops
def kv_append(k_new, v_new, k_cache, v_cache, block_tables, positions, stream=None) -> None:
    """Write k_new/v_new [B][n_kv][d] at logical positions[b] of every sequence."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(positions, torch.int32, "positions")
    NB, n_kv, bs, d = _cache_dims(k_cache)
    B, MB = block_tables.shape
    _check(lib().pgd_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                               _ptr(block_tables), _ptr(positions), B, n_kv, d, bs, MB, NB,
                               _stream(stream)))


def workspace_size(B: int, n_q: int, n_kv: int, num_splits: int = 0, d: int = HEAD_DIM) -> int:
    return int(lib().pgd_attention_workspace_size(B, n_q, n_kv, d, num_splits))


def make_workspace(B: int, n_q: int, n_kv: int, num_splits: int = 0, device=None) -> torch.Tensor:
    """A zero-filled workspace for these shapes (torch allocations are
    256-byte aligned)."""
    n = max(1, workspace_size(B, n_q, n_kv, num_splits))
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def attention_grid(B: int, n_q: int, n_kv: int, bs: int, num_splits: int = 0) -> int:
    return int(lib().pgd_attention_grid(B, n_q, n_kv, bs, num_splits))


def _attention_call(fp8, out, q, k_cache, v_cache, block_tables, context_lens, scale,
                    num_splits=0, workspace=None, stream=None):
    _need(q, torch.bfloat16, "q")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.uint8 if fp8 else torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, n_q, d = q.shape
    NB, n_kv, bs, _ = _cache8_dims(k_cache) if fp8 else _cache_dims(k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = make_workspace(B, n_q, n_kv, num_splits, q.device)
    MB = block_tables.shape[1]
    name = "pgd_paged_decode_attention_fp8" if fp8 else "pgd_paged_decode_attention"
    return name, (
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, n_q, n_kv, d, bs, MB, NB, float(scale), int(num_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), out


def paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """out[B][n_q][d] (bf16) = paged decode attention of q over the cache."""
    name, args, out = _attention_call(False, out, q, k_cache, v_cache, block_tables,
                                      context_lens, scale, num_splits, workspace, stream)
    _check(getattr(lib(), name)(*args))
    return out


def paged_decode_attention_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                   scale: float, num_splits: int = 0, stream=None) -> torch.Tensor:
    """paged_decode_attention without a workspace argument, for callers that
    cannot allocate device memory: the library keeps the scratch in its own
    fixed device array (shared by every call on a device; calls that overlap
    on one GPU race).  `out` must be given -- this call allocates nothing."""
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, n_q, d = q.shape
    NB, n_kv, bs, _ = _cache_dims(k_cache)
    MB = block_tables.shape[1]
    _check(lib().pgd_paged_decode_attention_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, n_q, n_kv, d, bs, MB, NB, float(scale), int(num_splits), _stream(stream)))
    return out


def _append_attention_call(fp8, out, q, k_new, v_new, k_cache, v_cache, block_tables,
                           context_lens, scale, num_splits=0, workspace=None, stream=None):
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, n)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.uint8 if fp8 else torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, n_q, d = q.shape
    NB, n_kv, bs, _ = _cache8_dims(k_cache) if fp8 else _cache_dims(k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = make_workspace(B, n_q, n_kv, num_splits, q.device)
    MB = block_tables.shape[1]
    name = "pgd_append_decode_attention_fp8" if fp8 else "pgd_append_decode_attention"
    return name, (
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(context_lens), B, n_q, n_kv, d, bs, MB, NB, float(scale),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), out


def append_decode_attention(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                            scale: float, num_splits: int = 0,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """kv_append of k_new/v_new at context_lens - 1, then paged decode
    attention over the updated cache (one call; two kernels, the attention
    prologue overlapping the append, or one short-context kernel that
    appends itself)."""
    name, args, out = _append_attention_call(False, out, q, k_new, v_new, k_cache, v_cache,
                                             block_tables, context_lens, scale, num_splits,
                                             workspace, stream)
    _check(getattr(lib(), name)(*args))
    return out


def _decode_step_call(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d,
                      v_new_d, context_lens_d, k_cache, v_cache, block_tables, scale, num_splits,
                      workspace, stream=None):
    for t, n in ((out_h, "out_h"), (q_h, "q_h"), (k_new_h, "k_new_h"), (v_new_h, "v_new_h")):
        _need(t, torch.bfloat16, n, cuda=False)
    _need(context_lens_h, torch.int32, "context_lens_h", cuda=False)
    B, n_q, d = q_h.shape
    fp8 = k_cache.dtype == torch.uint8
    NB, n_kv, bs, _ = _cache8_dims(k_cache) if fp8 else _cache_dims(k_cache)
    MB = block_tables.shape[1]
    name = "pgd_decode_step_fp8" if fp8 else "pgd_decode_step"
    return name, (
        _ptr(out_h), _ptr(q_h), _ptr(k_new_h), _ptr(v_new_h), _ptr(context_lens_h), _ptr(out_d),
        _ptr(q_d), _ptr(k_new_d), _ptr(v_new_d), _ptr(context_lens_d), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), B, n_q, n_kv, d, bs, MB, NB, float(scale),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), None


def decode_step(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d, v_new_d,
                context_lens_d, k_cache, v_cache, block_tables, scale: float, num_splits: int,
                workspace: torch.Tensor, stream=None) -> None:
    """One decode step with host inputs/outputs: append at context_lens - 1,
    then attention, all on `stream`.  Page-locked (pinned) host tensors are
    read and written in place by the kernels; pageable ones go through the
    given device tensors and a copy each.  An 8-bit pool (uint8) selects the
    FP8 path."""
    name, args, _ = _decode_step_call(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d,
                                      k_new_d, v_new_d, context_lens_d, k_cache, v_cache,
                                      block_tables, scale, num_splits, workspace, stream)
    _check(getattr(lib(), name)(*args))


class PreparedCall:
    """One C-ABI call whose arguments were checked and marshalled once;
    calling the object enqueues the same call again (same buffers, same
    stream) and returns its output tensor.  The Python side of a regular
    binding call -- a dozen tensor checks and pointer conversions -- takes
    about 10 us, longer than a short-context decode step on the GPU; a
    prepared call leaves only the C call (a few us).  The buffers must stay
    alive and unchanged in shape while the object is used."""
    __slots__ = ("name", "_fn", "_args", "out")

    def __init__(self, name: str, args: tuple, out=None):
        self.name = name
        self._fn = getattr(lib(), name)
        self._args = args
        self.out = out

    def __call__(self):
        s = self._fn(*self._args)
        if s != OK:
            _check(s)
        return self.out


def prepare(op: str, *args, **kwargs) -> PreparedCall:
    """A PreparedCall of one of the step calls, with the arguments that call
    takes: "paged_decode_attention", "paged_decode_attention_fp8",
    "append_decode_attention", "append_decode_attention_fp8", "decode_step",
    "append_verify_attention" or "verify_step"."""
    if op == "paged_decode_attention":
        return PreparedCall(*_attention_call(False, *args, **kwargs))
    if op == "paged_decode_attention_fp8":
        return PreparedCall(*_attention_call(True, *args, **kwargs))
    if op == "append_decode_attention":
        return PreparedCall(*_append_attention_call(False, *args, **kwargs))
    if op == "append_decode_attention_fp8":
        return PreparedCall(*_append_attention_call(True, *args, **kwargs))
    if op == "decode_step":
        return PreparedCall(*_decode_step_call(*args, **kwargs))
    if op == "append_verify_attention":
        return PreparedCall(*_append_verify_call(*args, **kwargs))
    if op == "verify_step":
        return PreparedCall(*_verify_step_call(*args, **kwargs))
    raise ValueError("no prepared form of %r" % op)


# ---------------------------------------------------------------- cascade
def kv_append_tokens(k_new, v_new, k_cache, v_cache, block_tables, positions,
                     stream=None) -> None:
    """Write k_new/v_new [B][T][n_kv][d]: token j of sequence b at logical
    position positions[b] + j."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(positions, torch.int32, "positions")
    NB, n_kv, bs, d = _cache_dims(k_cache)
    B, MB = block_tables.shape
    T = k_new.shape[1]
    _check(lib().pgd_kv_append_tokens(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(block_tables), _ptr(positions), B, T, n_kv, d, bs, MB,
                                      NB, _stream(stream)))


def verify_workspace_size(B: int, T: int, n_q: int, n_kv: int, num_splits: int = 0,
                          d: int = HEAD_DIM) -> int:
    return int(lib().pgd_verify_workspace_size(B, T, n_q, n_kv, d, num_splits))


def paged_verify_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """out[B][T][n_q][d] (bf16): each of the T new query tokens of a sequence
    attends to its cached context up to and including its own position."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, T, n_q, d = q.shape
    NB, n_kv, bs, d2 = _cache_dims(k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        n = max(1, verify_workspace_size(B, T, n_q, n_kv, num_splits))
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    MB = block_tables.shape[1]
    _check(lib().pgd_paged_verify_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, T, n_q, n_kv, d, bs, MB, NB, float(scale), int(num_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def _verify_workspace(workspace, B, T, n_q, n_kv, num_splits, device):
    if workspace is None:
        n = max(1, verify_workspace_size(B, T, n_q, n_kv, num_splits))
        workspace = torch.zeros(n, dtype=torch.uint8, device=device)
    return workspace


def _append_verify_call(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                        scale, num_splits=0, workspace=None, stream=None):
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"),
                 (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, T, n_q, d = q.shape
    NB, n_kv, bs, _ = _cache_dims(k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    workspace = _verify_workspace(workspace, B, T, n_q, n_kv, num_splits, q.device)
    MB = block_tables.shape[1]
    return "pgd_append_verify_attention", (
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(context_lens), B, T, n_q, n_kv, d, bs, MB, NB, float(scale),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), out


def append_verify_attention(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                            scale: float, num_splits: int = 0,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One verify step in one call: the T new tokens of every sequence
    (k_new/v_new [B][T][n_kv][d]) appended at context_lens - T + j, then
    paged_verify_attention over the updated caches (its prologue overlapping
    the append)."""
    name, args, out = _append_verify_call(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                          context_lens, scale, num_splits, workspace, stream)
    _check(getattr(lib(), name)(*args))
    return out


def _verify_step_call(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d,
                      v_new_d, context_lens_d, k_cache, v_cache, block_tables, scale, num_splits,
                      workspace, stream=None):
    for t, n in ((out_h, "out_h"), (q_h, "q_h"), (k_new_h, "k_new_h"), (v_new_h, "v_new_h")):
        _need(t, torch.bfloat16, n, cuda=False)
    _need(context_lens_h, torch.int32, "context_lens_h", cuda=False)
    _need(k_cache, torch.bfloat16, "k_cache")
    B, T, n_q, d = q_h.shape
    NB, n_kv, bs, _ = _cache_dims(k_cache)
    MB = block_tables.shape[1]
    return "pgd_verify_step", (
        _ptr(out_h), _ptr(q_h), _ptr(k_new_h), _ptr(v_new_h), _ptr(context_lens_h), _ptr(out_d),
        _ptr(q_d), _ptr(k_new_d), _ptr(v_new_d), _ptr(context_lens_d), _ptr(k_cache),
        _ptr(v_cache), _ptr(block_tables), B, T, n_q, n_kv, d, bs, MB, NB, float(scale),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), None


def verify_step(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d, k_new_d, v_new_d,
                context_lens_d, k_cache, v_cache, block_tables, scale: float, num_splits: int,
                workspace: torch.Tensor, stream=None) -> None:
    """One verify step with host inputs/outputs (q and out [B][T][n_q][d],
    k_new/v_new [B][T][n_kv][d]): append at context_lens - T + j, then verify
    attention, all on `stream`.  Page-locked (pinned) host tensors are read
    and written in place by the kernels; pageable ones go through the given
    device tensors and a copy each."""
    name, args, _ = _verify_step_call(out_h, q_h, k_new_h, v_new_h, context_lens_h, out_d, q_d,
                                      k_new_d, v_new_d, context_lens_d, k_cache, v_cache,
                                      block_tables, scale, num_splits, workspace, stream)
    _check(getattr(lib(), name)(*args))


def _mla_pool_dims(pool: torch.Tensor) -> Tuple[int, int, int]:
    """(NB, bs, D) of a latent pool bf16 [NB][bs/8][D/8][8][8]."""
    if pool.dim() != 5 or tuple(pool.shape[3:]) != (8, 8):
        raise ValueError("latent pool must be [NB][bs/8][D/8][8][8]")
    return pool.shape[0], pool.shape[1] * 8, pool.shape[2] * 8


def mla_append(c_new, cache, block_tables, positions, stream=None) -> None:
    """Write c_new[b] ([B][576] bf16) at logical position positions[b]."""
    _need(c_new, torch.bfloat16, "c_new")
    _need(cache, torch.bfloat16, "cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(positions, torch.int32, "positions")
    NB, bs, D = _mla_pool_dims(cache)
    B, MB = block_tables.shape
    _check(lib().pgd_mla_append(_ptr(c_new), _ptr(cache), _ptr(block_tables), _ptr(positions),
                                B, D, bs, MB, NB, _stream(stream)))


def mla_workspace_size(B: int, H: int, num_splits: int = 0) -> int:
    return int(lib().pgd_mla_workspace_size(B, H, num_splits))


def mla_decode_attention(out, q, cache, block_tables, context_lens, scale: float,
                         num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """out[B][H][512] (bf16) = decode attention of the absorbed queries q
    ([B][H][576]) over the latent cache."""
    _need(q, torch.bfloat16, "q")
    _need(cache, torch.bfloat16, "cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, H, D = q.shape
    NB, bs, D2 = _mla_pool_dims(cache)
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = torch.empty(max(256, mla_workspace_size(B, H, num_splits)), dtype=torch.uint8,
                                device=q.device)
    MB = block_tables.shape[1]
    _check(lib().pgd_mla_decode_attention(
        _ptr(out), _ptr(q), _ptr(cache), _ptr(block_tables), _ptr(context_lens), B, H, D, 512,
        bs, MB, NB, float(scale), int(num_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def mla_append_decode_attention(out, q, c_new, cache, block_tables, context_lens, scale: float,
                                num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """mla_append of c_new at context_lens - 1, then mla_decode_attention over
    the updated cache (one call, two kernels and the merge; the attention
    prologue overlaps the append)."""
    _need(q, torch.bfloat16, "q")
    _need(c_new, torch.bfloat16, "c_new")
    _need(cache, torch.bfloat16, "cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, H, D = q.shape
    NB, bs, D2 = _mla_pool_dims(cache)
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = torch.empty(max(256, mla_workspace_size(B, H, num_splits)), dtype=torch.uint8,
                                device=q.device)
    MB = block_tables.shape[1]
    _check(lib().pgd_mla_append_decode_attention(
        _ptr(out), _ptr(q), _ptr(c_new), _ptr(cache), _ptr(block_tables), _ptr(context_lens), B,
        H, D, 512, bs, MB, NB, float(scale), int(num_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def mla_step(out_h, q_h, c_new_h, context_lens_h, out_d, q_d, c_new_d, context_lens_d, cache,
             block_tables, scale: float, num_splits: int, workspace: torch.Tensor,
             stream=None) -> None:
    """One MLA decode step with host inputs/outputs (q [B][H][576], c_new
    [B][576], out [B][H][512]): q copied to q_d, page-locked c_new, context
    lengths and out read and written in place (pageable ones through the
    given device tensors and a copy), then mla_append_decode_attention, all
    on `stream`."""
    for t, n in ((out_h, "out_h"), (q_h, "q_h"), (c_new_h, "c_new_h")):
        _need(t, torch.bfloat16, n, cuda=False)
    _need(context_lens_h, torch.int32, "context_lens_h", cuda=False)
    _need(cache, torch.bfloat16, "cache")
    B, H, D = q_h.shape
    NB, bs, _ = _mla_pool_dims(cache)
    MB = block_tables.shape[1]
    _check(lib().pgd_mla_step(
        _ptr(out_h), _ptr(q_h), _ptr(c_new_h), _ptr(context_lens_h), _ptr(out_d), _ptr(q_d),
        _ptr(c_new_d), _ptr(context_lens_d), _ptr(cache), _ptr(block_tables), B, H, D, 512, bs,
        MB, NB, float(scale), int(num_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def cascade_workspace_size(B: int, n_q: int, n_kv: int, bs: int, max_group_size: int,
                           max_group_blocks: int, num_splits: int = 0, d: int = HEAD_DIM) -> int:
    return int(lib().pgd_cascade_workspace_size(B, n_q, n_kv, d, bs, num_splits, max_group_size,
                                                max_group_blocks))


def cascade_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens,
                             seq_prefix_blocks, group_first, group_size, group_blocks,
                             max_group_size: int, max_group_blocks: int, scale: float,
                             num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """Paged decode attention with shared prefixes read once per group (see
    pgd_cascade_decode_attention); group arrays are device int32."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    for t, n in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                 (seq_prefix_blocks, "seq_prefix_blocks"), (group_first, "group_first"),
                 (group_size, "group_size"), (group_blocks, "group_blocks")):
        _need(t, torch.int32, n)
    B, n_q, d = q.shape
    NB, n_kv, bs, _ = _cache_dims(k_cache)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        n = cascade_workspace_size(B, n_q, n_kv, bs, max_group_size, max_group_blocks, num_splits)
        workspace = torch.zeros(max(1, n), dtype=torch.uint8, device=q.device)
    MB = block_tables.shape[1]
    _check(lib().pgd_cascade_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(seq_prefix_blocks), _ptr(group_first), _ptr(group_size), _ptr(group_blocks),
        group_first.numel(), int(max_group_size), int(max_group_blocks), B, n_q, n_kv, d, bs, MB,
        NB, float(scale), int(num_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


# ------------------------------------------------------------ 8-bit KV cache
def _cache8_dims(pool: torch.Tensor) -> Tuple[int, int, int, int]:
    """(NB, n_kv, bs, d) of an 8-bit pool uint8 [NB][n_kv][bs/8][8*d + 32]."""
    if pool.dim() != 4 or pool.dtype != torch.uint8 or (pool.shape[3] - 32) % 8:
        raise ValueError("8-bit cache must be uint8 [NB][n_kv][bs/8][8*d + 32]")
    NB, n_kv, ng, gb = pool.shape
    return NB, n_kv, ng * 8, (gb - 32) // 8


def kv_append_fp8(k_new, v_new, k_cache, v_cache, block_tables, positions, stream=None) -> None:
    """Quantise k_new/v_new [B][n_kv][d] (bf16) per (token, head) and write
    codes and scales at logical positions[b] of the 8-bit pools."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(k_cache, torch.uint8, "k_cache")
    _need(v_cache, torch.uint8, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(positions, torch.int32, "positions")
    NB, n_kv, bs, d = _cache8_dims(k_cache)
    B, MB = block_tables.shape
    _check(lib().pgd_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_tables), _ptr(positions), B, n_kv, d, bs, MB, NB,
                                   _stream(stream)))


def paged_decode_attention_fp8(out, q, k_cache, v_cache, block_tables, context_lens,
                               scale: float, num_splits: int = 0,
                               workspace: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """out[B][n_q][d] (bf16) = paged decode attention of q over the 8-bit cache."""
    name, args, out = _attention_call(True, out, q, k_cache, v_cache, block_tables, context_lens,
                                      scale, num_splits, workspace, stream)
    _check(getattr(lib(), name)(*args))
    return out


def append_decode_attention_fp8(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                context_lens, scale: float, num_splits: int = 0,
                                workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """kv_append_fp8 at context_lens - 1, then attention over the 8-bit cache."""
    name, args, out = _append_attention_call(True, out, q, k_new, v_new, k_cache, v_cache,
                                             block_tables, context_lens, scale, num_splits,
                                             workspace, stream)
    _check(getattr(lib(), name)(*args))
    return out


def copy_blocks(k_cache, v_cache, src_ids, dst_ids, stream=None) -> None:
    """Copy whole physical blocks src_ids[i] -> dst_ids[i] (device int32)."""
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(src_ids, torch.int32, "src_ids")
    _need(dst_ids, torch.int32, "dst_ids")
    NB, n_kv, bs, d = _cache_dims(k_cache)
    _check(lib().pgd_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_ids), _ptr(dst_ids),
                                 src_ids.numel(), n_kv, d, bs, NB, _stream(stream)))


def device_errors(clear: bool = True, stream=None) -> int:
    """Wait for `stream` and return (then clear) the device error bits."""
    v = ctypes.c_int32(0)
    _check(lib().pgd_device_errors(ctypes.addressof(v), 1 if clear else 0, _stream(stream)))
    return int(v.value)


def read_stream(src: torch.Tensor, mode: int = 0, stream=None) -> None:
    """Read every byte of the CUDA tensor `src` once and discard it (the
    read-only streaming calibration pass; mode 0: 16-byte loads, mode 1:
    4 KiB bulk copies into shared memory)."""
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    _check(lib().pgd_read_stream(_ptr(src), src.numel() * src.element_size(), int(mode),
                                 _stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' bounded waits for launches made after this call
    (0 restores the 4 s default).  A short limit makes waits run out on
    purpose: for tests of the timeout exit only."""
    lib().pgd_set_wait_limit_ns(int(ns))


def wait_limit_ns() -> int:
    return int(lib().pgd_wait_limit_ns())


def set_short_context_tokens(max_tokens: int) -> int:
    """Largest MB * bs (at most 1024) for which an automatic single-query
    call may run the short-context kernel (0: never; negative: the default
    1024).  Returns the previous limit."""
    return int(lib().pgd_set_short_context_tokens(int(max_tokens)))


def uses_short_path(B: int, n_kv: int, bs: int, MB: int, num_splits: int = 0) -> bool:
    """Whether a call with these sizes (B sequences, n_kv KV heads, block size
    bs, table width MB) runs the short-context kernel now (pgd_short_path)."""
    return bool(lib().pgd_short_path(int(B), int(n_kv), int(bs), int(MB), int(num_splits)))


# ------------------------------------------------------------ host allocator
class BlockAllocator:
    """Host pool of physical block ids with reference counts (pgd_alloc_*)."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        _check(lib().pgd_alloc_create(int(num_blocks), ctypes.addressof(h)))
        self._h = h

    def close(self) -> None:
        if self._h:
            lib().pgd_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _arr(ids: Sequence[int]):
        return (ctypes.c_int32 * max(1, len(ids)))(*ids)

    def allocate(self, n: int) -> list:
        buf = (ctypes.c_int32 * max(1, n))()
        _check(lib().pgd_alloc_allocate(self._h, int(n), buf))
        return list(buf[:n])

    def share(self, ids: Sequence[int]) -> None:
        _check(lib().pgd_alloc_share(self._h, self._arr(ids), len(ids)))

    def release(self, ids: Sequence[int]) -> None:
        _check(lib().pgd_alloc_release(self._h, self._arr(ids), len(ids)))

    def refcount(self, i: int) -> int:
        return int(lib().pgd_alloc_refcount(self._h, int(i)))

    @property
    def num_free(self) -> int:
        return int(lib().pgd_alloc_num_free(self._h))

    @property
    def num_blocks(self) -> int:
        return int(lib().pgd_alloc_num_blocks(self._h))

    def append_slot(self, row: list, pos: int, block_size: int) -> Tuple[int, int]:
        """Make position `pos` of table `row` writable (row updated in place);
        returns the (src, dst) copy-on-write pair or (-1, -1)."""
        buf = (ctypes.c_int32 * len(row))(*row)
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        _check(lib().pgd_alloc_append_slot(self._h, buf, len(row), int(block_size), int(pos),
                                           ctypes.addressof(src), ctypes.addressof(dst)))
        row[:] = list(buf)
        return int(src.value), int(dst.value)

    def fork(self, src_row: Sequence[int], n_tokens: int, block_size: int, dst_row: list) -> None:
        s = (ctypes.c_int32 * len(src_row))(*src_row)
        d = (ctypes.c_int32 * len(dst_row))(*dst_row)
        _check(lib().pgd_alloc_fork(self._h, s, int(n_tokens), int(block_size), d, len(dst_row)))
        dst_row[:] = list(d)


def validate_tables(block_tables_h: torch.Tensor, context_lens_h: torch.Tensor, num_blocks: int,
                    block_size: int) -> None:
    """Host check of host copies of the tables and lengths (raises PGDError)."""
    t = block_tables_h.contiguous().to(torch.int32).cpu()
    c = context_lens_h.contiguous().to(torch.int32).cpu()
    B, MB = t.shape
    _check(lib().pgd_validate_tables(_ptr(t), _ptr(c), B, MB, int(num_blocks), int(block_size)))

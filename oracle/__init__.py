"""The oracle: plain, slow, float64 CPU statements of what the paged GQA decode
path computes.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it; both sides only share the seeded
input generators, which hold none of the method's arithmetic.

Contents
  * ``paged_attention`` / ``attention_weights`` / ``attention_part`` /
    ``lse_merge`` / ``kv_append`` -- ctypes wrappers over ``pgd_oracle.c``
    (plain C, float64, pthreads over (sequence, query head) rows).
  * ``e4m3_decode`` / ``e4m3_encode`` / ``quantize_rows`` /
    ``kv_append_fp8`` / ``paged_attention_fp8`` -- the 8-bit (FP8 E4M3,
    per-(token, head) scale) cache, over ``pgd_oracle_fp8.c``.
  * ``paged_verify_attention`` / ``kv_append_tokens`` -- multi-query
    (speculative verify) attention, T new query tokens per sequence with the
    causal mask among them, and appending T tokens, over
    ``pgd_oracle_verify.c``.
  * ``mla_attention`` / ``mla_append`` -- decode attention over an MLA
    latent cache (576 values per token shared by all heads; absorbed query;
    512-d latent output), over ``pgd_oracle_mla.c``.
  * ``kv_formula`` -- the KV-cache byte count in closed form.
  * ``block_model`` -- a plain-Python model of block tables, reference counts
    and copy-on-write.

Every function cites the page section it restates; see the C source header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import kv_formula  # noqa: F401  (re-exported)
from . import block_model  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "pgd_oracle.c"), os.path.join(_HERE, "pgd_oracle_fp8.c"),
         os.path.join(_HERE, "pgd_oracle_verify.c"), os.path.join(_HERE, "pgd_oracle_mla.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpgd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C sources with gcc into ``oracle/_build/``.  Plain
    -O2, no fast-math: the oracle's arithmetic must stay IEEE."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-o", tmp] + _SRCS + [
           "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_kv_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I]
        lib.oracle_kv_append.restype = I
        lib.oracle_paged_attention.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, D, I, I]
        lib.oracle_paged_attention.restype = I
        lib.oracle_attention_weights.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, D]
        lib.oracle_attention_weights.restype = I
        lib.oracle_attention_part.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, D]
        lib.oracle_attention_part.restype = I
        lib.oracle_lse_merge.argtypes = [P, P, P, P, I, I]
        lib.oracle_lse_merge.restype = I
        lib.oracle_threads_used.argtypes = [I, ctypes.c_long]
        lib.oracle_threads_used.restype = I
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = D
        lib.oracle_e4m3_encode_mode.argtypes = [ctypes.c_float, I]
        lib.oracle_e4m3_encode_mode.restype = ctypes.c_uint8
        lib.oracle_quantize_row.argtypes = [P, I, P, P, I]
        lib.oracle_quantize_row.restype = None
        lib.oracle_kv_append_fp8.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I]
        lib.oracle_kv_append_fp8.restype = I
        lib.oracle_paged_attention_fp8.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, D, I, I]
        lib.oracle_paged_attention_fp8.restype = I
        lib.oracle_kv_append_tokens.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I]
        lib.oracle_kv_append_tokens.restype = I
        lib.oracle_paged_verify_attention.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, D,
                                                      I, I]
        lib.oracle_paged_verify_attention.restype = I
        lib.oracle_mla_append.argtypes = [P, P, P, P, I, I, I, I, I]
        lib.oracle_mla_append.restype = I
        lib.oracle_mla_attention.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, D, I, I]
        lib.oracle_mla_attention.restype = I
        _lib = lib
        return lib


def _u16(a) -> np.ndarray:
    """bf16 data as its uint16 bit patterns (accepts torch bf16 tensors or
    uint16 numpy arrays)."""
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16, got %s" % a.dtype)
        return np.ascontiguousarray(a)
    import torch  # local: the oracle itself does not need torch
    if a.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor, got %s" % a.dtype)
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _tile_dims(cache: np.ndarray):
    """(NB, n_kv, bs, d) of a pool stored as [NB][n_kv][bs/8][d/8][8][8]."""
    if cache.ndim != 6 or cache.shape[4:] != (8, 8):
        raise ValueError("cache must be [NB][n_kv][bs/8][d/8][8][8] (8x8 core-matrix tiles)")
    NB, n_kv, rg, nc = cache.shape[:4]
    return NB, n_kv, rg * 8, nc * 8


def _i32(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a, dtype=np.int32)
    return np.ascontiguousarray(a.detach().cpu().numpy().astype(np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def threads_used(n_threads: int, rows: int) -> int:
    return int(_load().oracle_threads_used(int(n_threads), int(rows)))


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                    n_threads: int = 0, mutation: int = 0) -> np.ndarray:
    """float64 out[B][n_q][d] of single-token decode attention over the paged
    cache.  q: [B][n_q][d] bf16; k_cache, v_cache: [NB][n_kv][bs/8][d/8][8][8]
    bf16 (each (block, head) tile as 8x8 core matrices);
    block_tables: [B][MB] int32; context_lens: [B] int32 (includes the token
    just appended).  Raises ValueError on an invalid length or block id."""
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    ta, ca = _i32(block_tables), _i32(context_lens)
    B, n_q, d = qa.shape
    NB, n_kv, bs, d2 = _tile_dims(ka)
    assert d2 == d and va.shape == ka.shape and ta.shape[0] == B and ca.shape == (B,)
    MB = ta.shape[1]
    out = np.zeros((B, n_q, d), dtype=np.float64)
    st = _load().oracle_paged_attention(_p(out), _p(qa), _p(ka), _p(va), _p(ta), _p(ca), B, n_q,
                                        n_kv, d, bs, MB, NB, float(scale), int(n_threads),
                                        int(mutation))
    if st:
        raise ValueError("oracle: invalid context length or block id (status %d)" % st)
    return out


def attention_weights(q, k_cache, block_tables, context_lens, b: int, h: int,
                      scale: float) -> np.ndarray:
    """Softmax weights w[t], t < context_lens[b], of row (b, h)."""
    qa, ka = _u16(q), _u16(k_cache)
    ta, ca = _i32(block_tables), _i32(context_lens)
    B, n_q, d = qa.shape
    NB, n_kv, bs, _ = _tile_dims(ka)
    w = np.zeros(int(ca[b]), dtype=np.float64)
    st = _load().oracle_attention_weights(_p(w), _p(qa), _p(ka), _p(ta), _p(ca), int(b), int(h),
                                          n_q, n_kv, d, bs, ta.shape[1], NB, float(scale))
    if st:
        raise ValueError("oracle: invalid context length or block id")
    return w


def attention_part(q, k_cache, v_cache, block_tables, b: int, h: int, t0: int, t1: int,
                   scale: float):
    """Local state (m, l, o[d]) of row (b, h) over tokens [t0, t1)."""
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    ta = _i32(block_tables)
    B, n_q, d = qa.shape
    NB, n_kv, bs, _ = _tile_dims(ka)
    m = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    o = np.zeros(d, dtype=np.float64)
    st = _load().oracle_attention_part(_p(m), _p(l), _p(o), _p(qa), _p(ka), _p(va), _p(ta),
                                       int(b), int(h), int(t0), int(t1), n_q, n_kv, d, bs,
                                       ta.shape[1], NB, float(scale))
    if st:
        raise ValueError("oracle: invalid block id")
    return float(m[0]), float(l[0]), o


def lse_merge(m, l, o) -> np.ndarray:
    """Merge local states (m_i, l_i, o_i[d]) into the normalised row."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    n, d = o.shape
    out = np.zeros(d, dtype=np.float64)
    st = _load().oracle_lse_merge(_p(out), _p(m), _p(l), _p(o), n, d)
    if st:
        raise ValueError("oracle: every part is empty")
    return out


def kv_append(k_cache, v_cache, k_new, v_new, block_tables, positions):
    """Return copies of (k_cache, v_cache) as uint16 bit patterns with one new
    token per sequence written at logical position positions[b]."""
    kc = _u16(k_cache).copy()
    vc = _u16(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    ta, pa = _i32(block_tables), _i32(positions)
    NB, n_kv, bs, d = _tile_dims(kc)
    B = kn.shape[0]
    st = _load().oracle_kv_append(_p(kc), _p(vc), _p(kn), _p(vn), _p(ta), _p(pa), B, n_kv, d, bs,
                                  ta.shape[1], NB)
    if st:
        raise ValueError("oracle: position or block id out of range")
    return kc, vc


# ------------------------------------------------------------------ 8-bit KV
def _u8(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint8:
            raise TypeError("expected uint8 codes, got %s" % a.dtype)
        return np.ascontiguousarray(a)
    import torch
    if a.dtype != torch.uint8:
        raise TypeError("expected a uint8 tensor, got %s" % a.dtype)
    return np.ascontiguousarray(a.detach().cpu().contiguous().numpy())


def _pool8_dims(cache: np.ndarray, bs: int):
    """(NB, n_kv, d) of an 8-bit pool stored as [NB][n_kv][bs/8][8*d + 32]
    (per 8-token group: codes as 8 x 16-byte core matrices, then 8 fp32
    scales)."""
    if cache.ndim != 4 or cache.shape[2] * 8 != bs or (cache.shape[3] - 32) % 8:
        raise ValueError("8-bit cache must be [NB][n_kv][bs/8][8*d + 32] uint8")
    return cache.shape[0], cache.shape[1], (cache.shape[3] - 32) // 8


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of E4M3 codes (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def e4m3_encode(x, truncate: bool = False) -> np.ndarray:
    """Nearest E4M3 codes of binary32 values (ties to even, saturating)."""
    a = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.oracle_e4m3_encode_mode(float(v), 1 if truncate else 0)
                     for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def quantize_rows(x, mutation: int = 0):
    """Per-row quantisation of bf16 rows x[..., d]: (codes uint8 [..., d],
    scales float32 [...])."""
    xa = _u16(x)
    d = xa.shape[-1]
    rows = xa.reshape(-1, d)
    codes = np.zeros(rows.shape, dtype=np.uint8)
    scales = np.zeros(rows.shape[0], dtype=np.float32)
    lib = _load()
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        out = np.zeros(d, dtype=np.uint8)
        sc = np.zeros(1, dtype=np.float32)
        lib.oracle_quantize_row(_p(row), d, _p(out), _p(sc), int(mutation))
        codes[r] = out
        scales[r] = sc[0]
    return codes.reshape(xa.shape), scales.reshape(xa.shape[:-1])


def kv_append_fp8(k_cache, v_cache, k_new, v_new, block_tables, positions, block_size: int,
                  mutation: int = 0):
    """Return copies of the 8-bit pools (k_cache, v_cache) with one new token
    per sequence quantised and written, codes and scale, at logical position
    positions[b]."""
    kc, vc = _u8(k_cache).copy(), _u8(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    ta, pa = _i32(block_tables), _i32(positions)
    NB, n_kv, d = _pool8_dims(kc, block_size)
    B = kn.shape[0]
    st = _load().oracle_kv_append_fp8(_p(kc), _p(vc), _p(kn), _p(vn), _p(ta), _p(pa), B, n_kv, d,
                                      block_size, ta.shape[1], NB, int(mutation))
    if st:
        raise ValueError("oracle: position or block id out of range")
    return kc, vc


def paged_attention_fp8(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                        block_size: int, n_threads: int = 0, mutation: int = 0) -> np.ndarray:
    """float64 out[B][n_q][d] of decode attention over the 8-bit cache: the
    definition of ``paged_attention`` applied to the dequantised K and V.
    k_cache, v_cache: uint8 [NB][n_kv][bs/8][8*d + 32]."""
    qa, ka, va = _u16(q), _u8(k_cache), _u8(v_cache)
    ta, ca = _i32(block_tables), _i32(context_lens)
    B, n_q, d = qa.shape
    NB, n_kv, d2 = _pool8_dims(ka, block_size)
    assert d2 == d and va.shape == ka.shape
    out = np.zeros((B, n_q, d), dtype=np.float64)
    st = _load().oracle_paged_attention_fp8(_p(out), _p(qa), _p(ka), _p(va), _p(ta), _p(ca), B,
                                            n_q, n_kv, d, block_size, ta.shape[1], NB,
                                            float(scale), int(n_threads), int(mutation))
    if st:
        raise ValueError("oracle: invalid context length or block id (status %d)" % st)
    return out


def kv_append_tokens(k_cache, v_cache, k_new, v_new, block_tables, positions):
    """Return copies of the tiled bf16 pools with T new tokens per sequence
    (k_new / v_new [B][T][n_kv][d]) written at positions[b] + j."""
    kc, vc = _u16(k_cache).copy(), _u16(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    ta, pa = _i32(block_tables), _i32(positions)
    NB, n_kv, bs, d = _tile_dims(kc)
    B, T = kn.shape[0], kn.shape[1]
    st = _load().oracle_kv_append_tokens(_p(kc), _p(vc), _p(kn), _p(vn), _p(ta), _p(pa), B, T,
                                         n_kv, d, bs, ta.shape[1], NB)
    if st:
        raise ValueError("oracle: position or block id out of range")
    return kc, vc


def paged_verify_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           n_threads: int = 0, mutation: int = 0) -> np.ndarray:
    """float64 out[B][T][n_q][d]: query token i of sequence b attends to its
    cached positions 0 .. context_lens[b] - T + i (the T new tokens are the
    last T cached positions)."""
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    ta, ca = _i32(block_tables), _i32(context_lens)
    B, T, n_q, d = qa.shape
    NB, n_kv, bs, d2 = _tile_dims(ka)
    assert d2 == d and va.shape == ka.shape
    out = np.zeros((B, T, n_q, d), dtype=np.float64)
    st = _load().oracle_paged_verify_attention(_p(out), _p(qa), _p(ka), _p(va), _p(ta), _p(ca),
                                               B, T, n_q, n_kv, d, bs, ta.shape[1], NB,
                                               float(scale), int(n_threads), int(mutation))
    if st:
        raise ValueError("oracle: invalid context length or block id (status %d)" % st)
    return out


def _mla_dims(cache: np.ndarray):
    """(NB, bs, D) of a latent pool stored as [NB][bs/8][D/8][8][8]."""
    if cache.ndim != 5 or cache.shape[3:] != (8, 8):
        raise ValueError("latent pool must be [NB][bs/8][D/8][8][8] (8x8 core-matrix tiles)")
    NB, rg, nc = cache.shape[:3]
    return NB, rg * 8, nc * 8


def mla_append(cache, c_new, block_tables, positions):
    """Return a copy of the latent pool with c_new[b] ([B][D] bf16) written at
    logical position positions[b]."""
    ca = _u16(cache).copy()
    cn = _u16(c_new)
    ta, pa = _i32(block_tables), _i32(positions)
    NB, bs, D = _mla_dims(ca)
    st = _load().oracle_mla_append(_p(ca), _p(cn), _p(ta), _p(pa), cn.shape[0], D, bs,
                                   ta.shape[1], NB)
    if st:
        raise ValueError("oracle: position or block id out of range")
    return ca


def mla_attention(q, cache, block_tables, context_lens, scale: float, dv: int = 512,
                  n_threads: int = 0, mutation: int = 0) -> np.ndarray:
    """float64 out[B][H][dv]: softmax over t < context_lens[b] of
    scale * q[b][h] . c_t (all D cached values of token t), weighting the
    first dv values of each c_t."""
    qa, ca = _u16(q), _u16(cache)
    ta, la = _i32(block_tables), _i32(context_lens)
    B, H, D = qa.shape
    NB, bs, D2 = _mla_dims(ca)
    assert D2 == D
    out = np.zeros((B, H, dv), dtype=np.float64)
    st = _load().oracle_mla_attention(_p(out), _p(qa), _p(ca), _p(ta), _p(la), B, H, D, dv, bs,
                                      ta.shape[1], NB, float(scale), int(n_threads),
                                      int(mutation))
    if st:
        raise ValueError("oracle: invalid argument, context length or block id (status %d)" % st)
    return out

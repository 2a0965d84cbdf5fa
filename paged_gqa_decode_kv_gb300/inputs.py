"""Seeded synthetic inputs for the paged decode path.

This module is shared by the tests, the benchmark and the oracle's callers.
It holds none of the method's arithmetic: it only draws bf16 tensors, builds
block tables (random permutations of a physical pool) and poisons every slot
that must never be read with NaN.

Workloads (all single layer, d_head = 128, scale 1/sqrt(128)):

=====================  ====  =========  ===============================  ====  ==========
name                   B     n_q/n_kv   context                          bs    K/V
=====================  ====  =========  ===============================  ====  ==========
single_ctx512          1     32/8       512                              16    N(0, 1)
batch16_ctx8192        16    32/8       8192                             16    N(0, 1)
mha40_batch4_ctx8192   4     40/40      8192                             16    N(0, 1)
ragged64_g8            64    64/8       L ~ U[128, 32768], +1 appended   32    N(0, 0.5^2)
shared_prefix32        32    32/8       4000 shared + U[1, 2000]         16    N(0, 1)
single_ctx131072       1     32/8       131072                           16    N(0, 1)
=====================  ====  =========  ===============================  ====  ==========

Q is N(0, 1) everywhere.  Data seed 1234, table seed 4321.  The physical pool
holds every needed block plus 5 % spare blocks; the table is a random
permutation of it.  Spare blocks, unused tail slots and (when a workload
appends) the slot of the token about to be appended are NaN, and unused table
entries are -1, so any read outside the valid range shows up in the output.

Pool layout: bf16 [NB][n_kv][bs/8][d/8][8][8] -- each (block, KV head) tile of
bs tokens x d dims is stored as 8 x 8 core matrices, element (slot s, dim i)
at ((s/8)*(d/8) + i/8)*64 + (s%8)*8 + i%8.  ``tile_pool`` / ``untile_pool``
convert from / to the row-major view [NB][n_kv][bs][d].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

HEAD_DIM = 128
DATA_SEED = 1234
TABLE_SEED = 4321


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q: int
    n_kv: int
    block_size: int
    ctx: Optional[int] = None           # fixed context (all sequences)
    ragged: Optional[tuple] = None      # (lo, hi) inclusive, drawn per sequence
    shared_prefix: int = 0              # tokens shared by every sequence
    suffix: Optional[tuple] = None      # (lo, hi) inclusive unique suffix
    kv_std: float = 1.0
    q_std: float = 1.0
    append: bool = False                # one new token appended before attention
    head_dim: int = HEAD_DIM

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("single_ctx512", 1, 32, 8, 16, ctx=512),
        Workload("batch16_ctx8192", 16, 32, 8, 16, ctx=8192),
        Workload("mha40_batch4_ctx8192", 4, 40, 40, 16, ctx=8192),
        Workload("ragged64_g8", 64, 64, 8, 32, ragged=(128, 32768), kv_std=0.5, append=True),
        Workload("shared_prefix32", 32, 32, 8, 16, shared_prefix=4000, suffix=(1, 2000)),
        Workload("single_ctx131072", 1, 32, 8, 16, ctx=131072),
    ]
}


def context_lengths(w: Workload, seed: int = DATA_SEED) -> List[int]:
    """Context length of every sequence after the append (if any)."""
    g = torch.Generator().manual_seed(seed)
    if w.ctx is not None:
        return [w.ctx] * w.batch
    if w.ragged is not None:
        lo, hi = w.ragged
        drawn = torch.randint(lo, hi + 1, (w.batch,), generator=g).tolist()
        return [x + 1 for x in drawn] if w.append else drawn
    if w.suffix is not None:
        lo, hi = w.suffix
        suf = torch.randint(lo, hi + 1, (w.batch,), generator=g).tolist()
        return [w.shared_prefix + s for s in suf]
    raise ValueError("workload %s has no length rule" % w.name)


def tile_pool(x: torch.Tensor) -> torch.Tensor:
    """Row-major pool [NB][n_kv][bs][d] -> tiled [NB][n_kv][bs/8][d/8][8][8]."""
    NB, n_kv, bs, d = x.shape
    return x.reshape(NB, n_kv, bs // 8, 8, d // 8, 8).permute(0, 1, 2, 4, 3, 5).contiguous()


def untile_pool(x: torch.Tensor) -> torch.Tensor:
    """Tiled pool [NB][n_kv][bs/8][d/8][8][8] -> row-major [NB][n_kv][bs][d]."""
    NB, n_kv, rg, nc = x.shape[:4]
    return x.permute(0, 1, 2, 4, 3, 5).reshape(NB, n_kv, rg * 8, nc * 8)


def pool_shape(num_blocks: int, n_kv: int, block_size: int, head_dim: int = HEAD_DIM):
    return (num_blocks, n_kv, block_size // 8, head_dim // 8, 8, 8)


def pack_pool8(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """Row-major E4M3 codes [NB][n_kv][bs][d] (uint8) and fp32 scales
    [NB][n_kv][bs] -> the 8-bit pool [NB][n_kv][bs/8][8*d + 32]: per 8-token
    group, the codes as 8-row x 16-byte core matrices, then the 8 scales."""
    NB, n_kv, bs, d = codes.shape
    c = codes.reshape(NB, n_kv, bs // 8, 8, d // 16, 16).permute(0, 1, 2, 4, 3, 5)
    c = c.reshape(NB, n_kv, bs // 8, 8 * d)
    sc = scales.contiguous().reshape(NB, n_kv, bs // 8, 8).view(torch.uint8)
    return torch.cat([c, sc], dim=3).contiguous()


def unpack_pool8(pool: torch.Tensor):
    """The 8-bit pool -> (codes [NB][n_kv][bs][d] uint8, scales [NB][n_kv][bs] fp32)."""
    NB, n_kv, ng, gb = pool.shape
    d = (gb - 32) // 8
    c = pool[..., :8 * d].reshape(NB, n_kv, ng, d // 16, 8, 16).permute(0, 1, 2, 4, 3, 5)
    codes = c.reshape(NB, n_kv, ng * 8, d)
    scales = pool[..., 8 * d:].contiguous().view(torch.float32).reshape(NB, n_kv, ng * 8)
    return codes, scales


def pool_shape8(num_blocks: int, n_kv: int, block_size: int, head_dim: int = HEAD_DIM):
    return (num_blocks, n_kv, block_size // 8, 8 * head_dim + 32)


@dataclasses.dataclass
class PagedBatch:
    """Inputs of one decode step.  Tensors live on `device`.  With
    kv_format "fp8" the pools are uint8 [NB][n_kv][bs/8][8*d + 32]: E4M3
    codes and per-(token, head) fp32 scales (see pack_pool8)."""
    q: torch.Tensor              # bf16 [B][n_q][d] (verify steps: [B][T][n_q][d])
    k_cache: torch.Tensor        # bf16 [NB][n_kv][bs/8][d/8][8][8] (tiled), or uint8 codes
    v_cache: torch.Tensor        # same layout
    block_tables: torch.Tensor   # int32 [B][MB], -1 where unused
    context_lens: torch.Tensor   # int32 [B]
    k_new: Optional[torch.Tensor]  # bf16 [B][n_kv][d] when appending
    v_new: Optional[torch.Tensor]
    positions: Optional[torch.Tensor]  # int32 [B] = context_lens - 1 when appending
    scale: float
    n_kv: int
    block_size: int
    unique_blocks: int           # physical blocks referenced by the tables
    shared_blocks: int           # blocks referenced by more than one sequence
    kv_format: str = "bf16"      # "bf16" or "fp8" (E4M3 codes + scales)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def n_q(self) -> int:
        return self.q.shape[-2]  # (q may carry a token axis: [B][T][n_q][d])

    @property
    def head_dim(self) -> int:
        return self.q.shape[-1]

    def token(self, cache: torch.Tensor, block: int, head: int, slot: int) -> torch.Tensor:
        """The d-vector of one cached token (bf16 pools)."""
        t = cache[block, head, slot // 8, :, slot % 8, :]
        return t.reshape(-1)

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]


def _randn_bf16(shape, std: float, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, std^2) rounded to bf16, drawn in chunks to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    chunk = 1 << 26
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        t = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        flat[s:e].copy_(t)
    return out


def make_batch(batch: int, n_q: int, n_kv: int, block_size: int, ctx_lens: List[int], *,
               head_dim: int = HEAD_DIM, kv_std: float = 1.0, q_std: float = 1.0,
               shared_prefix: int = 0, append: bool = False, spare_frac: float = 0.05,
               max_blocks: Optional[int] = None, seed: int = DATA_SEED,
               table_seed: int = TABLE_SEED, device="cpu", poison: bool = True,
               scale: Optional[float] = None, kv_format: str = "bf16") -> PagedBatch:
    """Build one decode step's inputs.

    Every sequence b holds ctx_lens[b] tokens.  The first `shared_prefix`
    tokens of every sequence live in the same physical blocks (shared_prefix
    must then be a multiple of block_size, or the partial block is private).
    With append=True, the last token of every sequence is returned as
    k_new/v_new and its cache slot is left NaN.  The pool is drawn row-major,
    poisoned, then tiled.

    kv_format="fp8": the pools hold E4M3 codes drawn as N(0, 110^2) values
    clamped to +-448 and cast to float8_e4m3fn, with per-(token, head) scales
    uniform in kv_std * [0.5, 1.5] / 110 (so the dequantised values are about
    N(0, kv_std^2)), packed by pack_pool8; poisoned slots hold the NaN code
    and a NaN scale.  The appended token's k_new/v_new are fresh bf16
    N(0, kv_std^2) draws."""
    assert kv_format in ("bf16", "fp8")
    assert len(ctx_lens) == batch and n_q % n_kv == 0 and block_size % 8 == 0
    bs = block_size
    nblk = [(c + bs - 1) // bs for c in ctx_lens]
    n_shared = shared_prefix // bs if batch > 1 else 0
    if n_shared:
        assert all(c >= n_shared * bs for c in ctx_lens)
    private = [n - n_shared for n in nblk]
    needed = n_shared + sum(private)
    NB = max(1, needed + int(math.ceil(needed * spare_frac)))
    MB = max(nblk) if max_blocks is None else max_blocks
    assert MB >= max(nblk)

    tgen = torch.Generator().manual_seed(table_seed)
    perm = torch.randperm(NB, generator=tgen).to(torch.int32)
    tables = torch.full((batch, MB), -1, dtype=torch.int32)
    cursor = n_shared
    shared_ids = perm[:n_shared]
    for b in range(batch):
        if n_shared:
            tables[b, :n_shared] = shared_ids
        tables[b, n_shared:nblk[b]] = perm[cursor:cursor + private[b]]
        cursor += private[b]
    used_ids = perm[:needed]
    spare_ids = perm[needed:]

    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn_bf16((batch, n_q, head_dim), q_std, gen, device)
    fp8 = kv_format == "fp8"
    k_scale = v_scale = None
    if fp8:
        k_cache = _codes_e4m3((NB, n_kv, bs, head_dim), gen, device)
        v_cache = _codes_e4m3((NB, n_kv, bs, head_dim), gen, device)
        k_scale = _scales((NB, n_kv, bs), kv_std, gen, device)
        v_scale = _scales((NB, n_kv, bs), kv_std, gen, device)
    else:
        k_cache = _randn_bf16((NB, n_kv, bs, head_dim), kv_std, gen, device)
        v_cache = _randn_bf16((NB, n_kv, bs, head_dim), kv_std, gen, device)

    k_new = v_new = positions = None
    if append:
        positions = torch.tensor([c - 1 for c in ctx_lens], dtype=torch.int32)
        blk = tables[torch.arange(batch), positions // bs].long().to(device)
        slot = (positions % bs).long().to(device)
        if fp8:
            k_new = _randn_bf16((batch, n_kv, head_dim), kv_std, gen, device)
            v_new = _randn_bf16((batch, n_kv, head_dim), kv_std, gen, device)
        else:
            k_new = k_cache[blk, :, slot, :].clone()
            v_new = v_cache[blk, :, slot, :].clone()

    if poison and fp8:
        _poison8(k_cache, v_cache, k_scale, v_scale, tables, ctx_lens, bs, nblk, spare_ids,
                 (blk, slot) if append else None, device)
    elif poison:
        nan = float("nan")
        if spare_ids.numel():
            sid = spare_ids.long().to(device)
            k_cache[sid] = nan
            v_cache[sid] = nan
        for b in range(batch):
            tail = ctx_lens[b] % bs
            if tail:
                last = int(tables[b, nblk[b] - 1])
                k_cache[last, :, tail:, :] = nan
                v_cache[last, :, tail:, :] = nan
        if append:
            k_cache[blk, :, slot, :] = nan
            v_cache[blk, :, slot, :] = nan
    del used_ids
    if fp8:
        k_cache = pack_pool8(k_cache, k_scale)
        v_cache = pack_pool8(v_cache, v_scale)
    else:
        k_cache = tile_pool(k_cache)
        v_cache = tile_pool(v_cache)

    return PagedBatch(
        q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=tables.to(device), context_lens=torch.tensor(ctx_lens, dtype=torch.int32).to(device),
        k_new=k_new, v_new=v_new,
        positions=None if positions is None else positions.to(device),
        scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale,
        n_kv=n_kv, block_size=bs, unique_blocks=needed,
        shared_blocks=n_shared, kv_format=kv_format)


@dataclasses.dataclass
class VerifyBatch:
    """Inputs of one speculative-verify step: T new tokens per sequence (the
    pending token and T - 1 draft proposals) whose K/V are still to be
    appended at positions .. positions + T - 1 (their cache slots are NaN
    until then); context_lens of `paged` already count them."""
    paged: PagedBatch
    q: torch.Tensor          # bf16 [B][T][n_q][d]
    k_new: torch.Tensor      # bf16 [B][T][n_kv][d]
    v_new: torch.Tensor
    positions: torch.Tensor  # int32 [B] = context_lens - T

    @property
    def T(self) -> int:
        return self.q.shape[1]


def make_verify_batch(batch: int, n_q: int, n_kv: int, block_size: int, ctx_lens: List[int],
                      T: int, *, seed: int = DATA_SEED, table_seed: int = TABLE_SEED,
                      device="cpu", kv_std: float = 1.0, poison: bool = True) -> VerifyBatch:
    """make_batch's cache and tables for contexts of ctx_lens[b] tokens (the
    last T of them new), fresh N(0, 1) queries [B][T][n_q][d], and the new
    tokens' K/V taken from the drawn cache before their slots are poisoned."""
    assert T >= 1 and all(c >= T for c in ctx_lens)
    pb = make_batch(batch, n_q, n_kv, block_size, ctx_lens, seed=seed, table_seed=table_seed,
                    device=device, kv_std=kv_std, poison=poison)
    gen = torch.Generator(device=device).manual_seed(seed + 17)
    q = _randn_bf16((batch, T, n_q, pb.head_dim), 1.0, gen, device)
    bs = block_size
    pos = torch.tensor([c - T for c in ctx_lens], dtype=torch.int64)
    P = pos[:, None] + torch.arange(T)[None, :]
    blk = pb.block_tables.cpu().long()[torch.arange(batch)[:, None], P // bs].to(device)
    slot = (P % bs).to(device)
    kr, vr = untile_pool(pb.k_cache), untile_pool(pb.v_cache)
    k_new = kr[blk, :, slot, :].clone()  # [B][T][n_kv][d]
    v_new = vr[blk, :, slot, :].clone()
    if poison:
        kr[blk, :, slot, :] = float("nan")
        vr[blk, :, slot, :] = float("nan")
    pb.k_cache = tile_pool(kr)
    pb.v_cache = tile_pool(vr)
    return VerifyBatch(paged=pb, q=q, k_new=k_new, v_new=v_new,
                       positions=pos.to(torch.int32).to(device))


def make_verify_workload(name: str, T: int, device="cpu") -> VerifyBatch:
    """A named workload's batch, tables and context lengths (which then
    count the T new tokens of every sequence) as a verify step."""
    w = WORKLOADS[name]
    return make_verify_batch(w.batch, w.n_q, w.n_kv, w.block_size, context_lengths(w), T,
                             device=device, kv_std=w.kv_std)


# ---------------------------------------------------------------- MLA latent cache
MLA_D, MLA_DV = 576, 512  # cached values per token (latent 512 + RoPE key 64); value dims


def tile_latent(x: torch.Tensor) -> torch.Tensor:
    """Row-major latent rows [NB][bs][576] -> the latent pool's tiled layout
    [NB][bs/8][72][8][8] (8x8 core matrices per 8 tokens)."""
    NB, bs, D = x.shape
    return x.reshape(NB, bs // 8, 8, D // 8, 8).permute(0, 1, 3, 2, 4).contiguous()


def untile_latent(x: torch.Tensor) -> torch.Tensor:
    NB, rg, nc = x.shape[:3]
    return x.permute(0, 1, 3, 2, 4).reshape(NB, rg * 8, nc * 8)


@dataclasses.dataclass
class MlaBatch:
    """One decode step over an MLA latent cache: absorbed queries [B][H][576],
    the tiled latent pool, tables and lengths; with append, the newest
    token's row (c_new [B][576]) still to be written at `positions`."""
    q: torch.Tensor
    cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    c_new: Optional[torch.Tensor]
    positions: Optional[torch.Tensor]
    scale: float
    block_size: int
    unique_blocks: int

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def heads(self) -> int:
        return self.q.shape[1]


def make_mla_batch(batch: int, heads: int, block_size: int, ctx_lens: List[int], *,
                   append: bool = False, kv_std: float = 1.0, spare_frac: float = 0.05,
                   seed: int = DATA_SEED, table_seed: int = TABLE_SEED, device="cpu",
                   poison: bool = True, scale: Optional[float] = None) -> MlaBatch:
    """Latent rows N(0, kv_std^2) and queries N(0, 1), bf16; a pool of the
    needed blocks plus 5 % spare under a random permutation; spare blocks,
    tail slots and (append) the newest slot NaN; scale 1/sqrt(128 + 64) by
    default (the query-key width of the heads the latent stands for)."""
    bs = block_size
    nblk = [(c + bs - 1) // bs for c in ctx_lens]
    needed = sum(nblk)
    NB = max(1, needed + int(math.ceil(needed * spare_frac)))
    MB = max(nblk)
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(table_seed)).to(torch.int32)
    tables = torch.full((batch, MB), -1, dtype=torch.int32)
    cur = 0
    for b in range(batch):
        tables[b, :nblk[b]] = perm[cur:cur + nblk[b]]
        cur += nblk[b]
    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn_bf16((batch, heads, MLA_D), 1.0, gen, device)
    rows = _randn_bf16((NB, bs, MLA_D), kv_std, gen, device)
    c_new = positions = None
    if append:
        positions = torch.tensor([c - 1 for c in ctx_lens], dtype=torch.int32)
        blk = tables[torch.arange(batch), positions // bs].long().to(device)
        slot = (positions % bs).long().to(device)
        c_new = rows[blk, slot].clone()
    if poison:
        nan = float("nan")
        spare = perm[needed:].long().to(device)
        if spare.numel():
            rows[spare] = nan
        for b in range(batch):
            tail = ctx_lens[b] % bs
            if tail:
                rows[int(tables[b, nblk[b] - 1]), tail:] = nan
        if append:
            rows[blk, slot] = nan
    return MlaBatch(q=q, cache=tile_latent(rows), block_tables=tables.to(device),
                    context_lens=torch.tensor(ctx_lens, dtype=torch.int32).to(device),
                    c_new=c_new, positions=None if positions is None else positions.to(device),
                    scale=(1.0 / math.sqrt(192.0)) if scale is None else scale,
                    block_size=bs, unique_blocks=needed)


# Latent-cache workloads: (batch, heads, block size, context)
MLA_WORKLOADS = {
    "mla128_batch16_ctx8192": (16, 128, 64, 8192),
    "mla128_batch64_ctx4096": (64, 128, 64, 4096),
}


def make_mla_workload(name: str, device="cpu", append: bool = True) -> MlaBatch:
    B, H, bs, ctx = MLA_WORKLOADS[name]
    return make_mla_batch(B, H, bs, [ctx] * B, append=append, device=device)


def mla_bytes_read(batch: MlaBatch) -> int:
    """Algorithmic bytes of one latent decode call: every cached token's 576
    bf16 values, read once for all heads."""
    return int(batch.context_lens.sum().item()) * MLA_D * 2


NAN_CODE = 0x7F  # E4M3 S.1111.111


def _codes_e4m3(shape, gen: torch.Generator, device) -> torch.Tensor:
    """E4M3 codes (uint8): N(0, 110^2) draws clamped to the largest finite
    code and cast by torch's float8_e4m3fn conversion."""
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    flat = out.view(-1)
    n = flat.numel()
    chunk = 1 << 26
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        t = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        t.mul_(110.0).clamp_(-448.0, 448.0)
        flat[s:e].copy_(t.to(torch.float8_e4m3fn).view(torch.uint8))
    return out


def _scales(shape, kv_std: float, gen: torch.Generator, device) -> torch.Tensor:
    u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    return (u + 0.5) * (kv_std / 110.0)


def _poison8(k8, v8, ks, vs, tables, ctx_lens, bs, nblk, spare_ids, appended, device):
    """NaN codes and NaN scales wherever nothing valid is cached."""
    nan = float("nan")
    if spare_ids.numel():
        sid = spare_ids.long().to(device)
        k8[sid] = NAN_CODE
        v8[sid] = NAN_CODE
        ks[sid] = nan
        vs[sid] = nan
    for b in range(len(ctx_lens)):
        tail = ctx_lens[b] % bs
        if tail:
            last = int(tables[b, nblk[b] - 1])
            k8[last, :, tail:, :] = NAN_CODE
            v8[last, :, tail:, :] = NAN_CODE
            ks[last, :, tail:] = nan
            vs[last, :, tail:] = nan
    if appended is not None:
        blk, slot = appended
        k8[blk, :, slot, :] = NAN_CODE
        v8[blk, :, slot, :] = NAN_CODE
        ks[blk, :, slot] = nan
        vs[blk, :, slot] = nan


def make_workload(name: str, device="cpu", seed: int = DATA_SEED, kv_format: str = "bf16",
                  **overrides) -> PagedBatch:
    w = WORKLOADS[name]
    if overrides:
        w = dataclasses.replace(w, **overrides)
    lens = context_lengths(w, seed)
    return make_batch(w.batch, w.n_q, w.n_kv, w.block_size, lens, head_dim=w.head_dim,
                      kv_std=w.kv_std, q_std=w.q_std, shared_prefix=w.shared_prefix,
                      append=w.append, seed=seed, device=device, scale=w.scale,
                      kv_format=kv_format)


def kv_bytes_read(batch: PagedBatch, unique: bool = False) -> int:
    """Algorithmic K+V bytes one attention call must read: every cached token
    of every sequence, all KV heads, K and V (logical), or each physical block
    once (unique; only differs when blocks are shared).  bf16: 2 bytes per
    element; fp8: 1 byte per element plus the token's fp32 scale."""
    per_head = batch.head_dim * batch.k_cache.element_size()
    if batch.kv_format == "fp8":
        per_head += 4
    per_token = 2 * batch.n_kv * per_head
    assert batch.k_cache.dim() == (4 if batch.kv_format == "fp8" else 6)
    if not unique:
        return int(batch.context_lens.sum().item()) * per_token
    bs = batch.block_size
    lens = batch.context_lens.tolist()
    shared_tokens = batch.shared_blocks * bs
    total = shared_tokens + sum(c - shared_tokens for c in lens) if batch.shared_blocks else sum(lens)
    return total * per_token


def prefix_groups(batch: PagedBatch, groups):
    """Group arrays for cascade attention, as int32 tensors on the batch's
    device.  groups: list of (first sequence, number of sequences, shared
    blocks); the listed sequences must share those leading table entries
    (true of any sequences of a batch built with shared_prefix, up to its
    shared block count).  Returns (seq_prefix_blocks [B], group_first,
    group_size, group_blocks, max_group_size, max_group_blocks)."""
    dev = batch.q.device
    seq = [0] * batch.batch
    for first, size, blocks in groups:
        for b in range(first, first + size):
            seq[b] = blocks
    t = lambda v: torch.tensor(v, dtype=torch.int32, device=dev)
    firsts = [g[0] for g in groups]
    sizes = [g[1] for g in groups]
    blocks = [g[2] for g in groups]
    return (t(seq), t(firsts), t(sizes), t(blocks), max(sizes, default=0),
            max(blocks, default=0))

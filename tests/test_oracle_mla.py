"""Pins of the MLA latent-cache oracle (oracle/pgd_oracle_mla.c), CPU only.

  * the pages' absorption identities ("LLM inference systems engineering",
    2.8.2; "The math of Transformer inference", MLA section): per-head
    attention with explicit keys [W_h^UK c_t ; k_t^R] against queries
    [q_h^C ; q_h^R] and explicit values W_h^UV c_t, computed in float64,
    equals W_h^UV applied to the oracle's latent output for the absorbed
    query [W_h^{UK T} q_h^C ; q_h^R];
  * a library routine: torch SDPA in float64 with the cached row as the key
    (all 576 values), its first 512 values as the value, one KV head
    repeated for every query head (MQA with G = n_h);
  * the cache byte count per token the pages print (36 KiB; 70,272 B);
  * planted mistakes (RoPE part dropped, value read from the wrong dims, no
    scale) each make a pin fail.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import kv_formula

DC, DR = 512, 64
D = DC + DR


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def page_latent(C, bs, seed, spare=2):
    """Scatter contiguous per-sequence latent rows C[b] ([T][D] bf16) through a
    random block table into a tiled pool [NB][bs/8][D/8][8][8] (built
    row-major here, then tiled); unused slots NaN, unused entries -1."""
    B = len(C)
    nblk = [(c.shape[0] + bs - 1) // bs for c in C]
    NB = sum(nblk) + spare
    perm = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    MB = max(nblk) + 1
    tables = np.full((B, MB), -1, dtype=np.int32)
    pool = torch.full((NB, bs, D), float("nan"), dtype=torch.bfloat16)
    cur = 0
    for b in range(B):
        for j in range(nblk[b]):
            pid = int(perm[cur]); cur += 1
            tables[b, j] = pid
            t0, t1 = j * bs, min((j + 1) * bs, C[b].shape[0])
            pool[pid, : t1 - t0] = C[b][t0:t1]
    tiled = pool.reshape(NB, bs // 8, 8, D // 8, 8).permute(0, 1, 3, 2, 4).contiguous()
    return tiled, tables


def case(B, H, lens, seed):
    g = torch.Generator().manual_seed(seed)
    C = [bf16(torch.randn(T, D, generator=g)) for T in lens]
    q = bf16(torch.randn(B, H, D, generator=g))
    return q, C


def pin_absorbed_identity(mutation=0):
    B, H, dh, lens, bs = 2, 4, 32, [37, 70], 16
    g = torch.Generator().manual_seed(5)
    C = [bf16(torch.randn(T, D, generator=g)) for T in lens]
    pool, tab = page_latent(C, bs, seed=6)
    W_uk = torch.randn(H, dh, DC, generator=g, dtype=torch.float64) / math.sqrt(DC)
    W_uv = torch.randn(H, dh, DC, generator=g, dtype=torch.float64) / math.sqrt(DC)
    qc = torch.randn(B, H, dh, generator=g, dtype=torch.float64)
    qr = bf16(torch.randn(B, H, DR, generator=g)).double()
    # absorbed latent query, rounded to bf16; W_uk is then nudged (in float64)
    # so that W_uk^T qc equals the rounded vector, keeping the identity exact
    q_lat = torch.einsum("bhk,hkc->bhc", qc, W_uk)
    q_lat_r = bf16(q_lat).double()
    W = W_uk.unsqueeze(0).repeat(B, 1, 1, 1)  # per (b, h)
    u = qc / (qc * qc).sum(-1, keepdim=True)
    W = W + u.unsqueeze(-1) * (q_lat_r - q_lat).unsqueeze(-2)
    q_abs = torch.cat([q_lat_r, qr], dim=-1).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(dh + DR)
    lat = oracle.mla_attention(q_abs, pool, tab, np.array(lens, np.int32), scale,
                               mutation=mutation)
    for b in range(B):
        c = C[b].double()
        for h in range(H):
            k = torch.cat([c[:, :DC] @ W[b, h].T, c[:, DC:]], dim=1)        # [T][dh + DR]
            v = c[:, :DC] @ W_uv[h].T                                       # [T][dh]
            qq = torch.cat([qc[b, h], qr[b, h]])
            ref = F.scaled_dot_product_attention(qq[None, None, None], k[None, None],
                                                 v[None, None], scale=scale)[0, 0, 0]
            got = W_uv[h] @ torch.from_numpy(lat[b, h])
            err = (got - ref).abs().max().item()
            assert err < 1e-10, "absorbed vs explicit (b=%d h=%d): %.3g" % (b, h, err)


def pin_sdpa_mqa(mutation=0):
    for i, (B, H, lens, bs) in enumerate([(1, 8, [1], 16), (2, 16, [33, 64], 16),
                                          (3, 4, [100, 7, 129], 32), (2, 128, [65, 300], 64)]):
        q, C = case(B, H, lens, seed=20 + i)
        pool, tab = page_latent(C, bs, seed=30 + i)
        scale = 1.0 / math.sqrt(192)
        got = oracle.mla_attention(q, pool, tab, np.array(lens, np.int32), scale,
                                   mutation=mutation)
        for b in range(B):
            c = C[b].double()
            ref = F.scaled_dot_product_attention(q[b].double()[None, :, None, :],
                                                 c[None, None].expand(1, H, -1, -1),
                                                 c[None, None, :, :DC].expand(1, H, -1, -1),
                                                 scale=scale)[0, :, 0, :].numpy()
            err = np.abs(got[b] - ref).max()
            assert err < 1e-12, "MLA oracle vs SDPA (case %d): %.3g" % (i, err)


PINS = [pin_absorbed_identity, pin_sdpa_mqa]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_cache_bytes_per_token():
    # "LLM inference systems engineering", 2.4.2: (512 + 64) x 32 x 2 = 36,864 B
    assert kv_formula.mla_bytes_per_token(32, 512, 64, 2) == 36864
    assert round(kv_formula.kv_bytes_per_token(32, 8, 128, 2) / 36864, 2) == 3.56
    # "The math of Transformer inference", MLA: 61 x 576 x 2 = 70,272 B (DeepSeek-V3)
    assert kv_formula.mla_bytes_per_token(61, 512, 64, 2) == 70272
    # same page: MHA with 128 heads of (128 + 64)-d keys and 128-d values
    assert 128 * (128 + 64 + 128) == 40960 and round(40960 / 576) == 71


def test_append_places_the_row():
    q, C = case(2, 4, [20, 9], seed=41)
    pool, tab = page_latent(C, 16, seed=42)
    new = bf16(torch.randn(2, D, generator=torch.Generator().manual_seed(43)))
    pos = np.array([20, 9], np.int32)
    out = oracle.mla_append(pool, new, tab, pos)
    o = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16)
    NB = o.shape[0]
    rows = o.permute(0, 1, 3, 2, 4).reshape(NB, 16, D)  # untile (test-side)
    for b in range(2):
        blk = tab[b, pos[b] // 16]
        assert torch.equal(rows[blk, pos[b] % 16].view(torch.int16), new[b].view(torch.int16))


@pytest.mark.parametrize("mutation", [1, 2, 3])
def test_mutation_is_caught(mutation):
    caught = 0
    for pin in PINS:
        try:
            pin(mutation=mutation)
        except AssertionError:
            caught += 1
    assert caught >= 1, "mutation %d passed every pin" % mutation

"""Pins of the multi-query (speculative verify) oracle, CPU only.

The oracle (oracle/pgd_oracle_verify.c) scores T new query tokens per
sequence over the paged cache with the causal mask of "Module 10: inference
and serving", Lab 2 (position i of the new tokens sees every cached position
up to old + i).  It is pinned to things other than itself:
  * a library routine: torch's scaled_dot_product_attention in float64 with
    that mask (arange(k_len) <= old + arange(T)) over contiguous,
    head-repeated K/V, the paged cache built here by scattering the tokens
    through a random block table;
  * the single-query oracle (pinned on its own): T = 1 is plain decode, and
    query token i equals one decode step over the context cut after it --
    the target's verification reproduces step-by-step decoding ("The math of
    Transformer inference", section 10, greedy version);
  * causality: K/V after a query's position do not change its output;
  * appending T tokens equals T single-token appends;
  * planted mistakes (mask removed, mask off by one, query order reversed)
    each make a pin fail.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from test_oracle_pins import bf16, contiguous_case, page

D = 128


def verify_case(B, T, n_q, n_kv, lens, seed):
    """Contiguous K/V per sequence (lens include the T new tokens) and bf16
    queries [B][T][n_q][d]."""
    _, K, V = contiguous_case(B, n_q, n_kv, lens, seed)
    g = torch.Generator().manual_seed(seed + 1)
    q = bf16(torch.randn(B, T, n_q, D, generator=g))
    return q, K, V


def sdpa_causal(q, K, V, scale):
    """float64 SDPA with Lab 2's mask: new position i sees k <= old + i."""
    B, T, n_q, d = q.shape
    out = np.zeros((B, T, n_q, d))
    for b in range(B):
        n_kv, L, _ = K[b].shape
        G = n_q // n_kv
        old = L - T
        mask = torch.arange(L)[None, :] <= old + torch.arange(T)[:, None]
        qq = q[b].double().permute(1, 0, 2).unsqueeze(0)  # [1][n_q][T][d]
        kk = K[b].double().repeat_interleave(G, dim=0).unsqueeze(0)
        vv = V[b].double().repeat_interleave(G, dim=0).unsqueeze(0)
        o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        out[b] = o[0].permute(1, 0, 2).numpy()
    return out


CASES = [
    # B, T, n_q, n_kv, bs, lens (including the T new tokens)
    (1, 1, 4, 4, 8, [1]),
    (2, 2, 8, 2, 8, [2, 17]),
    (3, 4, 8, 2, 16, [4, 40, 33]),
    (2, 3, 8, 1, 16, [70, 5]),
    (2, 4, 16, 4, 16, [64, 19]),
    (1, 8, 4, 2, 8, [30]),
    (2, 16, 2, 2, 32, [16, 49]),
]


def pin_sdpa_causal(mutation=0):
    for i, (B, T, n_q, n_kv, bs, lens) in enumerate(CASES):
        q, K, V = verify_case(B, T, n_q, n_kv, lens, seed=300 + i)
        kc, vc, tab = page(K, V, bs, seed=400 + i)
        scale = 1.0 / math.sqrt(D)
        got = oracle.paged_verify_attention(q, kc, vc, tab, np.array(lens, np.int32), scale,
                                            mutation=mutation)
        ref = sdpa_causal(q, K, V, scale)
        assert np.all(np.isfinite(got)), "non-finite oracle output"
        err = np.abs(got - ref).max()
        assert err < 1e-12, "verify oracle vs causal SDPA float64: max abs %.3g" % err


def pin_sequential_decode(mutation=0):
    """Row i equals a single decode step over positions 0 .. ctx - T + i."""
    B, T, n_q, n_kv, bs = 3, 5, 8, 2, 16
    lens = [5, 37, 64]
    q, K, V = verify_case(B, T, n_q, n_kv, lens, seed=31)
    kc, vc, tab = page(K, V, bs, seed=32)
    scale = 0.09
    got = oracle.paged_verify_attention(q, kc, vc, tab, np.array(lens, np.int32), scale,
                                        mutation=mutation)
    for i in range(T):
        ctx_i = np.array([c - T + i + 1 for c in lens], np.int32)
        want = oracle.paged_attention(q[:, i].contiguous(), kc, vc, tab, ctx_i, scale)
        err = np.abs(got[:, i] - want).max()
        assert err < 1e-13, "query %d vs one decode step: %.3g" % (i, err)


def pin_causality(mutation=0):
    """Changing K/V of the last new token leaves every earlier query as is."""
    B, T, n_q, n_kv, bs = 2, 4, 8, 2, 8
    lens = [12, 30]
    q, K, V = verify_case(B, T, n_q, n_kv, lens, seed=41)
    kc, vc, tab = page(K, V, bs, seed=42)
    a = oracle.paged_verify_attention(q, kc, vc, tab, np.array(lens, np.int32), 0.1,
                                      mutation=mutation)
    K2 = [k.clone() for k in K]
    V2 = [v.clone() for v in V]
    for b in range(B):
        K2[b][:, -1] = bf16(torch.full((n_kv, D), 3.0))
        V2[b][:, -1] = bf16(torch.full((n_kv, D), -5.0))
    kc2, vc2, tab2 = page(K2, V2, bs, seed=42)
    b_ = oracle.paged_verify_attention(q, kc2, vc2, tab2, np.array(lens, np.int32), 0.1,
                                       mutation=mutation)
    assert np.array_equal(a[:, :T - 1], b_[:, :T - 1]), "earlier queries saw a later token"
    assert not np.array_equal(a[:, T - 1], b_[:, T - 1]), "the last query must see its token"


PINS = [pin_sdpa_causal, pin_sequential_decode, pin_causality]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_t1_is_decode():
    B, n_q, n_kv, bs = 3, 8, 2, 16
    lens = [1, 17, 50]
    q, K, V = verify_case(B, 1, n_q, n_kv, lens, seed=51)
    kc, vc, tab = page(K, V, bs, seed=52)
    a = oracle.paged_verify_attention(q, kc, vc, tab, np.array(lens, np.int32), 0.1)
    b_ = oracle.paged_attention(q[:, 0].contiguous(), kc, vc, tab, np.array(lens, np.int32), 0.1)
    assert np.abs(a[:, 0] - b_).max() < 1e-14


def test_kv_append_tokens_equals_single_appends():
    B, T, n_kv, bs = 3, 5, 2, 8
    lens = [9, 20, 33]
    q, K, V = verify_case(B, T, 4, n_kv, lens, seed=61)
    kc, vc, tab = page(K, V, bs, seed=62)
    g = torch.Generator().manual_seed(63)
    kn = bf16(torch.randn(B, T, n_kv, D, generator=g))
    vn = bf16(torch.randn(B, T, n_kv, D, generator=g))
    pos = np.array([c - T for c in lens], np.int32)
    k1, v1 = oracle.kv_append_tokens(kc, vc, kn, vn, tab, pos)
    k2, v2 = oracle._u16(kc), oracle._u16(vc)
    for j in range(T):
        k2, v2 = oracle.kv_append(k2, v2, kn[:, j].contiguous(), vn[:, j].contiguous(), tab,
                                  pos + j)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)


def test_context_shorter_than_t_is_rejected():
    q, K, V = verify_case(1, 4, 4, 2, [3], seed=71)
    kc, vc, tab = page(K, V, 8, seed=72)
    with pytest.raises(ValueError):
        oracle.paged_verify_attention(q, kc, vc, tab, np.array([3], np.int32), 0.1)


@pytest.mark.parametrize("mutation", [1, 2, 3])
def test_mutation_is_caught(mutation):
    caught = 0
    for pin in PINS:
        try:
            pin(mutation=mutation)
        except AssertionError:
            caught += 1
    assert caught >= 1, "mutation %d passed every pin" % mutation

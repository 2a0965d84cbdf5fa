"""Pins of the oracle to things other than itself (CPU only).

Each pin checks the float64 oracle against something the pages or mathematics
fix independently of the oracle's code:
  * a library routine: torch's scaled_dot_product_attention in float64 over a
    contiguous, explicitly head-repeated K/V (the toy decoder of "Module 10:
    inference and serving", Lab 2, attends with SDPA over repeat_interleave'd
    KV heads), with the paged cache built here by scattering the contiguous
    tokens through a random block table;
  * closed forms: one cached token returns its value; uniform values return
    that value; a zero query returns the mean value; two tokens weigh by the
    logistic function of the score gap; one dominant key returns its value;
  * invariants: softmax weights form a probability vector; permuting physical
    blocks and rewriting the table changes nothing ("Module 10", section
    "Mapping logical positions to physical blocks"); a prefix held in shared
    blocks gives the same result as private copies (section "Share only
    identical state"); splitting the context and merging the parts by
    log-sum-exp gives the unsplit result ("The math of Transformer inference",
    section 8; "LLM inference systems engineering", section 2.8.3).
The last test plants each of the oracle's known mutations and checks that at
least one pin fails for it.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import expit

import oracle

D = 128


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def contiguous_case(B, n_q, n_kv, lens, seed, d=D, kv_std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = bf16(torch.randn(B, n_q, d, generator=g))
    K = [bf16(torch.randn(n_kv, T, d, generator=g) * kv_std) for T in lens]
    V = [bf16(torch.randn(n_kv, T, d, generator=g) * kv_std) for T in lens]
    return q, K, V


def tile(x):
    """Row-major [NB][n_kv][bs][d] -> the pool's tiled layout
    [NB][n_kv][bs/8][d/8][8][8] (8x8 core matrices), by reshape/permute."""
    NB, n_kv, bs, d = x.shape
    return x.reshape(NB, n_kv, bs // 8, 8, d // 8, 8).permute(0, 1, 2, 4, 3, 5).contiguous()


def page(K, V, bs, seed, spare=3, share_prefix_blocks=0):
    """Scatter contiguous per-sequence K/V [n_kv][T][d] into a paged pool
    through a random permutation (built row-major here, then tiled).  Unused blocks, tail slots
    and table entries are poisoned (NaN / -1).  The first
    `share_prefix_blocks` blocks of every sequence are taken from sequence 0
    and stored once."""
    B = len(K)
    n_kv, _, d = K[0].shape
    nblk = [(k.shape[1] + bs - 1) // bs for k in K]
    sp = share_prefix_blocks
    need = sp + sum(n - sp for n in nblk)
    NB = need + spare
    rng = np.random.default_rng(seed)
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(nblk) + 1
    tables = np.full((B, MB), -1, dtype=np.int32)
    kc = torch.full((NB, n_kv, bs, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((NB, n_kv, bs, d), float("nan"), dtype=torch.bfloat16)
    cur = 0
    for b in range(B):
        for j in range(nblk[b]):
            if j < sp and b > 0:
                tables[b, j] = tables[0, j]
                continue
            pid = int(perm[cur]); cur += 1
            tables[b, j] = pid
            t0, t1 = j * bs, min((j + 1) * bs, K[b].shape[1])
            kc[pid, :, : t1 - t0] = K[b][:, t0:t1]
            vc[pid, :, : t1 - t0] = V[b][:, t0:t1]
    return tile(kc), tile(vc), tables


def sdpa_reference(q, K, V, scale):
    """float64 torch SDPA per sequence over contiguous, head-repeated K/V."""
    B, n_q, d = q.shape
    out = np.zeros((B, n_q, d))
    for b in range(B):
        n_kv = K[b].shape[0]
        G = n_q // n_kv
        qq = q[b].double().reshape(1, n_q, 1, d)
        kk = K[b].double().repeat_interleave(G, dim=0).unsqueeze(0)
        vv = V[b].double().repeat_interleave(G, dim=0).unsqueeze(0)
        out[b] = F.scaled_dot_product_attention(qq, kk, vv, scale=scale)[0, :, 0, :].numpy()
    return out


CASES = [
    # B, n_q, n_kv, bs, lens
    (1, 4, 4, 8, [1]),
    (2, 8, 2, 8, [5, 16]),
    (3, 8, 1, 16, [70, 17, 33]),
    (2, 16, 2, 16, [31, 64]),
    (3, 4, 2, 8, [3, 9, 12]),
    (2, 8, 4, 32, [33, 95]),
]


# ----------------------------------------------------------------- pins
def pin_sdpa(mutation=0):
    for i, (B, n_q, n_kv, bs, lens) in enumerate(CASES):
        q, K, V = contiguous_case(B, n_q, n_kv, lens, seed=100 + i)
        kc, vc, tab = page(K, V, bs, seed=200 + i)
        scale = 1.0 / math.sqrt(D)
        got = oracle.paged_attention(q, kc, vc, tab, np.array(lens, np.int32), scale,
                                     mutation=mutation)
        ref = sdpa_reference(q, K, V, scale)
        assert np.all(np.isfinite(got)), "non-finite oracle output"
        err = np.abs(got - ref).max()
        assert err < 1e-12, "oracle vs SDPA float64: max abs %.3g" % err


def pin_ctx1(mutation=0):
    q, K, V = contiguous_case(2, 8, 2, [1, 1], seed=7)
    kc, vc, tab = page(K, V, 16, seed=8)
    got = oracle.paged_attention(q, kc, vc, tab, np.array([1, 1], np.int32), 0.1,
                                 mutation=mutation)
    for b in range(2):
        for h in range(8):
            assert np.array_equal(got[b, h], V[b][h // 4, 0].double().numpy()), "ctx=1 != v_0"


def pin_uniform_v(mutation=0):
    lens = [37, 16]
    q, K, V = contiguous_case(2, 8, 2, lens, seed=9)
    vec = bf16(torch.randn(D, generator=torch.Generator().manual_seed(10)))
    V = [v.clone() for v in V]
    for v in V:
        v[:] = vec
    kc, vc, tab = page(K, V, 8, seed=11)
    got = oracle.paged_attention(q, kc, vc, tab, np.array(lens, np.int32), 1 / math.sqrt(D),
                                 mutation=mutation)
    err = np.abs(got - vec.double().numpy()).max()
    assert err < 1e-13, "uniform V not reproduced: %.3g" % err


def pin_zero_query(mutation=0):
    lens = [23, 40]
    q, K, V = contiguous_case(2, 4, 4, lens, seed=12)
    q = torch.zeros_like(q)
    kc, vc, tab = page(K, V, 8, seed=13)
    got = oracle.paged_attention(q, kc, vc, tab, np.array(lens, np.int32), 1 / math.sqrt(D),
                                 mutation=mutation)
    for b in range(2):
        mean = V[b].double().mean(dim=1).numpy()  # [n_kv][d]
        err = np.abs(got[b] - mean).max()
        assert err < 1e-13, "zero query is not the mean of V: %.3g" % err


def pin_two_tokens(mutation=0):
    q, K, V = contiguous_case(1, 2, 1, [2], seed=14)
    kc, vc, tab = page(K, V, 8, seed=15)
    scale = 1 / math.sqrt(D)
    got = oracle.paged_attention(q, kc, vc, tab, np.array([2], np.int32), scale,
                                 mutation=mutation)
    k = K[0][0].double().numpy()
    v = V[0][0].double().numpy()
    for h in range(2):
        qq = q[0, h].double().numpy()
        gap = scale * (qq @ k[0] - qq @ k[1])
        want = expit(gap) * v[0] + expit(-gap) * v[1]
        assert np.abs(got[0, h] - want).max() < 1e-13, "two-token closed form"


def pin_dominant_key(mutation=0):
    T = 64
    q, K, V = contiguous_case(1, 4, 1, [T], seed=16)
    j = 41
    q = bf16(4.0 * K[0][0, j].float()).reshape(1, 1, D).repeat(1, 4, 1)
    kc, vc, tab = page(K, V, 16, seed=17)
    got = oracle.paged_attention(q, kc, vc, tab, np.array([T], np.int32), 1 / math.sqrt(D),
                                 mutation=mutation)
    want = V[0][0, j].double().numpy()
    assert np.abs(got[0] - want).max() < 1e-9, "dominant key does not win"


def pin_block_permutation(mutation=0):
    lens = [45, 19, 64]
    q, K, V = contiguous_case(3, 8, 2, lens, seed=18)
    kc, vc, tab = page(K, V, 8, seed=19)
    a = oracle.paged_attention(q, kc, vc, tab, np.array(lens, np.int32), 0.09, mutation=mutation)
    NB = kc.shape[0]
    perm = np.random.default_rng(20).permutation(NB)
    inv = np.empty_like(perm); inv[perm] = np.arange(NB)
    kc2 = kc[torch.as_tensor(inv)]
    vc2 = vc[torch.as_tensor(inv)]
    tab2 = np.where(tab >= 0, perm[np.maximum(tab, 0)], -1).astype(np.int32)
    b = oracle.paged_attention(q, kc2, vc2, tab2, np.array(lens, np.int32), 0.09,
                               mutation=mutation)
    assert np.array_equal(a, b), "block permutation changed the output"


def pin_shared_prefix(mutation=0):
    bs, sp = 8, 3  # 3 shared blocks = 24 tokens
    lens = [30, 41, 24]
    q, K, V = contiguous_case(3, 8, 2, lens, seed=21)
    K = [k.clone() for k in K]
    V = [v.clone() for v in V]
    for b in range(1, 3):
        K[b][:, : sp * bs] = K[0][:, : sp * bs]
        V[b][:, : sp * bs] = V[0][:, : sp * bs]
    kc, vc, tab = page(K, V, bs, seed=22, share_prefix_blocks=sp)
    kc2, vc2, tab2 = page(K, V, bs, seed=23)
    assert (tab[1, :sp] == tab[0, :sp]).all() and kc.shape[0] < kc2.shape[0]
    a = oracle.paged_attention(q, kc, vc, tab, np.array(lens, np.int32), 0.09, mutation=mutation)
    b = oracle.paged_attention(q, kc2, vc2, tab2, np.array(lens, np.int32), 0.09,
                               mutation=mutation)
    assert np.array_equal(a, b), "shared prefix differs from private copies"


ATTENTION_PINS = [pin_sdpa, pin_ctx1, pin_uniform_v, pin_zero_query, pin_two_tokens,
                  pin_dominant_key, pin_block_permutation, pin_shared_prefix]


@pytest.mark.parametrize("pin", ATTENTION_PINS, ids=lambda f: f.__name__)
def test_attention_pin(pin):
    pin(0)


@pytest.mark.parametrize("mutation", range(1, 9))
def test_planted_mistake_is_caught(mutation):
    failed = []
    for pin in ATTENTION_PINS:
        try:
            pin(mutation)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, "mutation %d passed every pin" % mutation


def test_weights_are_a_probability_vector():
    lens = [77]
    q, K, V = contiguous_case(1, 8, 2, lens, seed=30)
    kc, vc, tab = page(K, V, 16, seed=31)
    for h in range(8):
        w = oracle.attention_weights(q, kc, tab, np.array(lens, np.int32), 0, h, 1 / math.sqrt(D))
        assert w.shape == (77,) and (w > 0).all()
        assert abs(w.sum() - 1.0) < 1e-14
        # the largest weight sits on the largest dot product (computed here
        # from the contiguous keys, not through the table)
        dots = K[0][h // 4].double().numpy() @ q[0, h].double().numpy()
        assert int(np.argmax(w)) == int(np.argmax(dots))


@pytest.mark.parametrize("n_parts", [1, 2, 3, 7, 64])
def test_split_and_lse_merge_equals_unsplit(n_parts):
    T = 200
    q, K, V = contiguous_case(1, 4, 2, [T], seed=40 + n_parts)
    kc, vc, tab = page(K, V, 16, seed=41)
    scale = 1 / math.sqrt(D)
    full = oracle.paged_attention(q, kc, vc, tab, np.array([T], np.int32), scale)
    rng = np.random.default_rng(n_parts)
    cuts = np.sort(rng.choice(np.arange(0, T + 1), size=n_parts - 1, replace=True)) \
        if n_parts > 1 else np.array([], int)
    bounds = [0] + cuts.tolist() + [T]
    for h in range(4):
        parts = [oracle.attention_part(q, kc, vc, tab, 0, h, bounds[i], bounds[i + 1], scale)
                 for i in range(n_parts)]
        m = [p[0] for p in parts]
        l = [p[1] for p in parts]
        o = np.stack([p[2] for p in parts])
        merged = oracle.lse_merge(m, l, o)
        assert np.abs(merged - full[0, h]).max() < 1e-13
        order = rng.permutation(n_parts)
        merged2 = oracle.lse_merge(np.array(m)[order], np.array(l)[order], o[order])
        assert np.abs(merged2 - full[0, h]).max() < 1e-13


def test_lse_merge_closed_form_two_parts():
    # two single-token parts: merge must give the logistic mix of the values
    m = np.array([0.3, -1.1]); l = np.array([1.0, 1.0])
    o = np.array([[1.0, 0.0], [0.0, 1.0]])
    out = oracle.lse_merge(m, l, o)
    w0 = expit(m[0] - m[1])
    assert np.allclose(out, [w0, 1 - w0], rtol=0, atol=1e-15)


def test_invalid_inputs_are_rejected():
    q, K, V = contiguous_case(1, 4, 2, [5], seed=50)
    kc, vc, tab = page(K, V, 8, seed=51)
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kc, vc, tab, np.array([0], np.int32), 0.1)
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kc, vc, tab, np.array([8 * tab.shape[1] + 1], np.int32), 0.1)
    bad = tab.copy(); bad[0, 0] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kc, vc, bad, np.array([5], np.int32), 0.1)


def test_kv_append_places_bits():
    B, n_kv, bs = 3, 2, 8
    lens = [9, 16, 1]
    q, K, V = contiguous_case(B, 4, n_kv, lens, seed=60)
    kc, vc, tab = page(K, V, bs, seed=61)
    g = torch.Generator().manual_seed(62)
    k_new = bf16(torch.randn(B, n_kv, D, generator=g))
    v_new = bf16(torch.randn(B, n_kv, D, generator=g))
    pos = np.array([9, 15, 0], np.int32)  # 9: slot 1 of block 1; 15: last slot; 0: overwrite
    k2, v2 = oracle.kv_append(kc, vc, k_new, v_new, tab, pos)
    # expected: untile (test-local inverse permute), write rows, tile again
    def untile(x):
        NB, nkv, rg, nc = x.shape[:4]
        return x.permute(0, 1, 2, 4, 3, 5).reshape(NB, nkv, rg * 8, nc * 8)
    ek, ev = untile(kc).clone(), untile(vc).clone()
    for b in range(B):
        blk, slot = int(tab[b, pos[b] // bs]), int(pos[b] % bs)
        ek[blk, :, slot, :] = k_new[b]
        ev[blk, :, slot, :] = v_new[b]
    want_k = tile(ek).view(torch.int16).numpy().view(np.uint16)
    want_v = tile(ev).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(k2, want_k) and np.array_equal(v2, want_v)
    # out-of-range position is refused
    with pytest.raises(ValueError):
        oracle.kv_append(kc, vc, k_new, v_new, tab, np.array([5, 7, bs * tab.shape[1]], np.int32))


def test_tile_layout_of_one_element():
    # element (slot 13, dim 77) of a bs=16 tile sits at ((13//8)*16 + 77//8)*64 + (13%8)*8 + 77%8
    x = torch.zeros(1, 1, 16, 128, dtype=torch.bfloat16)
    x[0, 0, 13, 77] = 1.0
    flat = tile(x).reshape(-1)
    assert int(torch.nonzero(flat).item()) == ((13 // 8) * 16 + 77 // 8) * 64 + (13 % 8) * 8 + 77 % 8

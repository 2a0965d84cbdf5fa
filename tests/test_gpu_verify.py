"""Parity of multi-query (speculative verify) attention and the multi-token
append, through the C ABI, with the float64 oracle on the same seeded inputs.

pgd_kv_append_tokens: the pools bit exact against the oracle's own append of
the same tokens into CPU copies of the caches as generated.  Attention:
max abs error <= 2e-2 and mean abs error <= 2e-3 against the oracle, every
element; T = 1 is bit-identical to the decode entry point.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import inputs
from gpu_common import assert_no_device_errors, cache_bits, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_errors():
    pgd.device_errors(clear=True)
    yield
    assert_no_device_errors()


def _batch(n_q, n_kv, bs, lens, T, seed=1234):
    return inputs.make_verify_batch(len(lens), n_q, n_kv, bs, lens, T, seed=seed,
                                    table_seed=seed + 7, device="cuda")


def _oracle(vb):
    """The oracle's own append into CPU copies of the generated caches, then
    its verify attention over them."""
    pb = vb.paged
    k, v = oracle.kv_append_tokens(pb.k_cache.cpu(), pb.v_cache.cpu(), vb.k_new.cpu(),
                                   vb.v_new.cpu(), pb.block_tables.cpu(), vb.positions.cpu())
    out = oracle.paged_verify_attention(vb.q.cpu(), k, v, pb.block_tables.cpu(),
                                        pb.context_lens.cpu(), pb.scale)
    return out, k, v


def _gpu(vb, num_splits=0):
    pb = vb.paged
    pgd.kv_append_tokens(vb.k_new, vb.v_new, pb.k_cache, pb.v_cache, pb.block_tables,
                         vb.positions)
    return pgd.paged_verify_attention(None, vb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                      pb.context_lens, pb.scale, num_splits=num_splits)


SMALL = [
    # (n_q, n_kv, bs, T, lens)
    (4, 4, 16, 2, [2]),
    (8, 4, 16, 4, [4, 5, 17]),
    (16, 4, 16, 4, [33, 200, 513]),
    (16, 4, 32, 3, [31, 32, 33, 700]),
    (32, 8, 16, 4, [64, 4, 95]),
    (32, 8, 32, 2, [512, 129]),
    (64, 8, 16, 2, [129, 1000, 32]),
    (8, 1, 16, 2, [300, 5]),
    (2, 1, 16, 8, [47, 8]),
    (4, 4, 16, 16, [16, 300]),
    (8, 8, 32, 5, [90, 250]),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "nq%d_nkv%d_bs%d_T%d_%s" % (
    c[0], c[1], c[2], c[3], "-".join(map(str, c[4]))))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_verify_small(case, num_splits):
    n_q, n_kv, bs, T, lens = case
    vb = _batch(n_q, n_kv, bs, lens, T)
    want, k, v = _oracle(vb)
    got = _gpu(vb, num_splits)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(vb.paged.k_cache), k)
    assert np.array_equal(cache_bits(vb.paged.v_cache), v)
    compare(got, want, "verify T=%d splits=%d" % (T, num_splits))


@pytest.mark.parametrize("G,T", [(1, 16), (2, 8), (4, 4), (4, 3), (8, 2)])
@pytest.mark.parametrize("bs", [16, 32])
def test_verify_ragged(G, T, bs):
    g = torch.Generator().manual_seed(G * 100 + T * 10 + bs)
    lens = torch.randint(T, 1500, (19,), generator=g).tolist()
    vb = _batch(4 * G, 4, bs, lens, T, seed=77 + G)
    want, _, _ = _oracle(vb)
    compare(_gpu(vb), want, "verify ragged G=%d T=%d bs=%d" % (G, T, bs))


def test_t1_equals_decode_bit_exactly():
    vb = _batch(32, 8, 16, [1, 17, 300, 2048], 1)
    pb = vb.paged
    pgd.kv_append_tokens(vb.k_new, vb.v_new, pb.k_cache, pb.v_cache, pb.block_tables,
                         vb.positions)
    a = pgd.paged_verify_attention(None, vb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                   pb.context_lens, pb.scale)
    b = pgd.paged_decode_attention(None, vb.q[:, 0].contiguous(), pb.k_cache, pb.v_cache,
                                   pb.block_tables, pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0].view(torch.int16), b.view(torch.int16))


def test_rows_past_16_are_refused():
    vb = _batch(8, 1, 16, [40], 4)
    pb = vb.paged
    with pytest.raises(pgd.PGDError):
        pgd.paged_verify_attention(None, vb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                   pb.context_lens, pb.scale)


def test_verify_full_size_batch16_ctx8192_t4():
    """The benchmark's batch (16 x 8192 tokens, 32/8 heads) verifying 4
    tokens per sequence: 16 query rows per KV head on one pass."""
    vb = _batch(32, 8, 16, [8192] * 16, 4)
    want, _, _ = _oracle(vb)
    compare(_gpu(vb), want, "verify batch16 ctx8192 T=4")


@pytest.mark.parametrize("G,T", [(4, 4), (2, 8)])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_verify_reference_moves_mid_context(G, T, num_splits):
    """16 query rows per KV head; K tiles of later blocks scaled by 8 and then
    by 32 (exact in bf16) before the append: every row with a nonzero query
    moves its reference twice after the first stages, rows of zero-query
    heads keep factor 1."""
    lens = [1500, 1300, 1700]
    vb = _batch(4 * G, 4, 16, lens, T, seed=55 + G)
    pb = vb.paged
    for b, n in enumerate(lens):
        for j in range(-(-n // 16)):
            f = 32.0 if j >= 64 else (8.0 if j >= 32 else 1.0)
            pb.k_cache[int(pb.block_tables[b, j])] *= f
    vb.q[:, :, ::3] = 0
    want, _, _ = _oracle(vb)
    compare(_gpu(vb, num_splits), want, "verify rescale G=%d T=%d splits=%d" % (G, T, num_splits))


# ----------------------------------------- one-call step and host buffers
ONE_CALL = [(8, 4, 16, 4, [4, 5, 17]), (32, 8, 32, 2, [512, 129]), (2, 1, 16, 8, [47, 8]),
            (16, 4, 16, 4, [33, 200, 2100])]


@pytest.mark.parametrize("case", ONE_CALL, ids=lambda c: "nq%d_nkv%d_bs%d_T%d_%s" % (
    c[0], c[1], c[2], c[3], "-".join(map(str, c[4]))))
@pytest.mark.parametrize("num_splits", [0, 3])
def test_append_verify_one_call(case, num_splits):
    """pgd_append_verify_attention appends at context_lens - T + j and then
    attends: the pools bit exact against the oracle's append, the output
    bit-identical to the two calls it replaces and within tolerance of the
    oracle."""
    n_q, n_kv, bs, T, lens = case
    vb = _batch(n_q, n_kv, bs, lens, T)
    pb = vb.paged
    want, k, v = _oracle(vb)
    kc2, vc2 = pb.k_cache.clone(), pb.v_cache.clone()
    got = pgd.append_verify_attention(None, vb.q, vb.k_new, vb.v_new, pb.k_cache, pb.v_cache,
                                      pb.block_tables, pb.context_lens, pb.scale,
                                      num_splits=num_splits)
    pgd.kv_append_tokens(vb.k_new, vb.v_new, kc2, vc2, pb.block_tables, vb.positions)
    two = pgd.paged_verify_attention(None, vb.q, kc2, vc2, pb.block_tables, pb.context_lens,
                                     pb.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(pb.k_cache), k)
    assert np.array_equal(cache_bits(pb.v_cache), v)
    assert torch.equal(got.view(torch.int16), two.view(torch.int16))
    compare(got, want, "append+verify T=%d splits=%d" % (T, num_splits))


def test_append_verify_refusal_enqueues_nothing():
    """More than 16 query rows per KV head: refused before the append runs."""
    vb = _batch(8, 1, 16, [40], 4)
    pb = vb.paged
    before = cache_bits(pb.k_cache)
    with pytest.raises(pgd.PGDError):
        pgd.append_verify_attention(None, vb.q, vb.k_new, vb.v_new, pb.k_cache, pb.v_cache,
                                    pb.block_tables, pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(pb.k_cache), before)


@pytest.mark.parametrize("pinned", ["all", "none", "mixed"])
def test_verify_step_host_buffers(pinned):
    """pgd_verify_step: page-locked host buffers read and written in place,
    pageable ones copied, each on its own; output and pools equal the
    device-buffer one-call step bit for bit."""
    vb = _batch(16, 4, 16, [33, 200, 2100, 4], 4)
    pb = vb.paged
    kc2, vc2 = pb.k_cache.clone(), pb.v_cache.clone()
    want = pgd.append_verify_attention(None, vb.q, vb.k_new, vb.v_new, kc2, vc2,
                                       pb.block_tables, pb.context_lens, pb.scale)
    pin = lambda t: t.cpu().pin_memory()
    page = lambda t: t.cpu().clone()
    hq, hk, hv, ho, hc = {"all": (pin,) * 5, "none": (page,) * 5,
                          "mixed": (pin, page, pin, page, page)}[pinned]
    q_h, kn_h, vn_h = hq(vb.q), hk(vb.k_new), hv(vb.v_new)
    cl_h, out_h = hc(pb.context_lens), ho(torch.zeros_like(vb.q))
    q_d, kn_d, vn_d = torch.empty_like(vb.q), torch.empty_like(vb.k_new), torch.empty_like(vb.v_new)
    cl_d, out_d = torch.empty_like(pb.context_lens), torch.empty_like(vb.q)
    B, T, n_q, _ = vb.q.shape
    ws = torch.zeros(max(1, pgd.verify_workspace_size(B, T, n_q, 4)), dtype=torch.uint8,
                     device="cuda")
    pgd.verify_step(out_h, q_h, kn_h, vn_h, cl_h, out_d, q_d, kn_d, vn_d, cl_d, pb.k_cache,
                    pb.v_cache, pb.block_tables, pb.scale, 0, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), want.cpu().view(torch.int16))
    assert np.array_equal(cache_bits(pb.k_cache), cache_bits(kc2))
    assert np.array_equal(cache_bits(pb.v_cache), cache_bits(vc2))


def test_verify_prepared_calls():
    """prepare("append_verify_attention") and prepare("verify_step") repeat
    the same call: twice over the same inputs gives the same output."""
    vb = _batch(32, 8, 16, [300, 2100], 2)
    pb = vb.paged
    B, T, n_q, _ = vb.q.shape
    ws = torch.zeros(max(1, pgd.verify_workspace_size(B, T, n_q, 8)), dtype=torch.uint8,
                     device="cuda")
    want, _, _ = _oracle(vb)
    call = pgd.prepare("append_verify_attention", None, vb.q, vb.k_new, vb.v_new, pb.k_cache,
                       pb.v_cache, pb.block_tables, pb.context_lens, pb.scale, 0, ws)
    a = call().clone()
    b = call()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    compare(a, want, "prepared append+verify")
    pin = lambda t: t.cpu().pin_memory()
    out_h = pin(torch.zeros_like(vb.q))
    step = pgd.prepare("verify_step", out_h, pin(vb.q), pin(vb.k_new), pin(vb.v_new),
                       pin(pb.context_lens), torch.empty_like(vb.q), torch.empty_like(vb.q),
                       torch.empty_like(vb.k_new), torch.empty_like(vb.v_new),
                       torch.empty_like(pb.context_lens), pb.k_cache, pb.v_cache,
                       pb.block_tables, pb.scale, 0, ws)
    step()
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), a.cpu().view(torch.int16))

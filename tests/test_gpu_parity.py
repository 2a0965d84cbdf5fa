"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Attention output: max abs error <= 2e-2 and mean abs error <= 2e-3 against
the oracle, every element.  kv_append and copy_blocks: bit exact.
Inputs come from the seeded generators; unused blocks, unused tail slots and
unused table entries are poisoned (NaN / -1), so an out-of-range read shows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import inputs
from gpu_common import (assert_no_device_errors, cache_bits, compare, gpu_attention,
                        oracle_append_then_attend, oracle_attention)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_errors():
    pgd.device_errors(clear=True)
    yield
    assert_no_device_errors()


def _batch(B, n_q, n_kv, bs, lens, seed=1234, **kw):
    return inputs.make_batch(B, n_q, n_kv, bs, lens, seed=seed, table_seed=seed + 7,
                             device="cuda", **kw)


SMALL = [
    # (n_q, n_kv, bs, lens)
    (4, 4, 16, [1]),
    (8, 4, 16, [16, 17, 1]),
    (16, 4, 16, [33, 200, 513]),
    (16, 2, 32, [31, 32, 33, 700]),
    (32, 4, 32, [64, 1, 95]),
    (32, 8, 16, [512]),
    (64, 8, 32, [129, 1000, 32]),
    (8, 1, 16, [300, 5]),
    (2, 1, 16, [47]),
    (40, 40, 16, [90, 250]),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "nq%d_nkv%d_bs%d_%s" % (
    c[0], c[1], c[2], "-".join(map(str, c[3]))))
@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 7, 64])
def test_attention_small(case, num_splits):
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens)
    want = oracle_attention(pb)
    got = gpu_attention(pb, num_splits=num_splits)
    compare(got, want, "splits=%d" % num_splits)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_attention_ragged_many(G, bs):
    g = torch.Generator().manual_seed(G * 100 + bs)
    B = 37
    lens = torch.randint(1, 3 * bs * 7, (B,), generator=g).tolist()
    pb = _batch(B, 2 * G, 2, bs, lens, seed=G + bs)
    want = oracle_attention(pb)
    for splits in (0, 1, 5):
        compare(gpu_attention(pb, num_splits=splits), want, "G=%d bs=%d splits=%d" % (G, bs, splits))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_maximum_batch(kv):
    """B = PGD_MAX_BATCH (2048) sequences of 1..100 tokens: the largest cost
    prefix the kernel keeps in shared memory, 4096 units over the SMs, the
    append of every sequence's token; against the oracle."""
    g = torch.Generator().manual_seed(2048)
    B = 2048
    lens = torch.randint(1, 101, (B,), generator=g).tolist()
    pb = _batch(B, 8, 2, 16, lens, seed=2048, append=True, kv_format=kv)
    if kv == "fp8":
        want_k, want_v = oracle.kv_append_fp8(pb.k_cache.cpu(), pb.v_cache.cpu(),
                                              pb.k_new.cpu(), pb.v_new.cpu(),
                                              pb.block_tables.cpu(), pb.positions.cpu(), 16)
        want = oracle.paged_attention_fp8(pb.q.cpu(), want_k, want_v, pb.block_tables.cpu(),
                                          pb.context_lens.cpu(), pb.scale, 16)
        got = pgd.append_decode_attention_fp8(None, pb.q, pb.k_new, pb.v_new, pb.k_cache,
                                              pb.v_cache, pb.block_tables, pb.context_lens,
                                              pb.scale)
    else:
        want, want_k, want_v = oracle_append_then_attend(pb)
        got = pgd.append_decode_attention(None, pb.q, pb.k_new, pb.v_new, pb.k_cache, pb.v_cache,
                                          pb.block_tables, pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    bits = (lambda t: t.cpu().numpy()) if kv == "fp8" else cache_bits
    assert np.array_equal(bits(pb.k_cache), want_k)
    assert np.array_equal(bits(pb.v_cache), want_v)
    compare(got, want, "B = 2048 (%s)" % kv)


def test_workspace_reuse_across_calls():
    # the per-unit arrival counters must return to zero after every call
    pb = _batch(3, 16, 4, 16, [500, 33, 1024])
    want = oracle_attention(pb)
    ws = pgd.make_workspace(3, 16, 4, 0)
    first = gpu_attention(pb, workspace=ws).clone()
    for _ in range(5):
        again = gpu_attention(pb, workspace=ws)
        assert torch.equal(first, again)
    compare(first, want)
    assert int(ws[: 3 * 4 * 4].view(torch.int32).abs().sum()) == 0


def test_ctx1_returns_v0_exactly():
    pb = _batch(4, 16, 4, 16, [1, 1, 1, 1])
    got = gpu_attention(pb)
    G = 4
    for b in range(4):
        blk = int(pb.block_tables[b, 0])
        for h in range(16):
            assert torch.equal(got[b, h], pb.token(pb.v_cache, blk, h // G, 0))


def test_uniform_values():
    pb = _batch(2, 8, 2, 16, [333, 64])
    vec = torch.randn(128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    vr = inputs.untile_pool(pb.v_cache).clone()
    for b in range(2):
        n = (int(pb.context_lens[b]) + 15) // 16
        ids = pb.block_tables[b, :n].long()
        tail = int(pb.context_lens[b]) % 16
        vr[ids] = vec
        if tail:
            vr[ids[-1], :, tail:] = float("nan")
    pb.v_cache = inputs.tile_pool(vr)
    got = gpu_attention(pb)
    diff = (got.float() - vec.float()).abs().max().item()
    assert diff <= abs(vec.float()).max().item() * 2 ** -8


def test_block_permutation_is_bit_identical():
    pb = _batch(5, 16, 4, 16, [700, 5, 129, 256, 1])
    a = gpu_attention(pb).clone()
    NB = pb.num_blocks
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm); inv[perm] = torch.arange(NB)
    k2 = pb.k_cache[inv.cuda()].contiguous()
    v2 = pb.v_cache[inv.cuda()].contiguous()
    t = pb.block_tables.long()
    t2 = torch.where(t >= 0, perm.cuda()[t.clamp(min=0)], t).to(torch.int32).contiguous()
    b = pgd.paged_decode_attention(None, pb.q, k2, v2, t2, pb.context_lens, pb.scale)
    assert torch.equal(a, b)


def test_shared_prefix_equals_private_copies():
    B, bs = 6, 16
    lens = [160 + 7 * i for i in range(B)]
    shared = _batch(B, 32, 8, bs, lens, shared_prefix=160)
    # private copy: every sequence gets its own copies of the prefix blocks
    n_pref = 160 // bs
    NB = shared.num_blocks
    extra = (B - 1) * n_pref
    k2 = torch.cat([shared.k_cache, torch.empty((extra,) + shared.k_cache.shape[1:],
                                                dtype=torch.bfloat16, device="cuda")])
    v2 = torch.cat([shared.v_cache, torch.empty_like(k2[:extra])])
    t2 = shared.block_tables.clone()
    nxt = NB
    for b in range(1, B):
        for j in range(n_pref):
            src = int(shared.block_tables[b, j])
            k2[nxt] = shared.k_cache[src]
            v2[nxt] = shared.v_cache[src]
            t2[b, j] = nxt
            nxt += 1
    a = gpu_attention(shared)
    c = pgd.paged_decode_attention(None, shared.q, k2, v2, t2, shared.context_lens, shared.scale)
    assert torch.equal(a, c)
    compare(a, oracle_attention(shared))


def test_solo_vs_batch():
    lens = [900, 17, 4000, 1, 256]
    pb = _batch(5, 32, 8, 16, lens)
    full = gpu_attention(pb)
    for b in range(5):
        solo = pgd.paged_decode_attention(None, pb.q[b:b + 1].contiguous(), pb.k_cache,
                                          pb.v_cache, pb.block_tables[b:b + 1].contiguous(),
                                          pb.context_lens[b:b + 1].contiguous(), pb.scale)
        d = (solo[0].float() - full[b].float()).abs().max().item()
        assert d <= 2e-2


def test_split_counts_agree():
    pb = _batch(2, 32, 8, 16, [4096, 3000])
    want = oracle_attention(pb)
    outs = [gpu_attention(pb, num_splits=s) for s in (1, 2, 3, 7, 64)]
    for o in outs:
        compare(o, want)
        assert (o.float() - outs[0].float()).abs().max().item() <= 1e-2


# ------------------------------------------------------------- kv_append
@pytest.mark.parametrize("bs", [16, 32])
def test_kv_append_bit_exact(bs):
    B, n_kv = 9, 4
    lens = [1, bs, bs + 1, 2 * bs, 77, 3, 5 * bs - 1, 200, 64]
    pb = _batch(B, 16, n_kv, bs, lens, append=True)
    k_before, v_before = pb.k_cache.cpu(), pb.v_cache.cpu()
    pgd.kv_append(pb.k_new, pb.v_new, pb.k_cache, pb.v_cache, pb.block_tables, pb.positions)
    torch.cuda.synchronize()
    want_k, want_v = oracle.kv_append(k_before, v_before, pb.k_new.cpu(), pb.v_new.cpu(),
                                      pb.block_tables.cpu(), pb.positions.cpu())
    got_k = pb.k_cache.cpu().view(torch.int16).numpy().view(np.uint16)
    got_v = pb.v_cache.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)


def test_append_then_attend_matches_oracle():
    pb = _batch(4, 32, 8, 32, [1, 300, 33, 1024], append=True)
    want, _, _ = oracle_append_then_attend(pb)
    pgd.kv_append(pb.k_new, pb.v_new, pb.k_cache, pb.v_cache, pb.block_tables, pb.positions)
    compare(gpu_attention(pb), want)


APPEND_CASES = [
    # (n_q, n_kv, bs, lens): the new token lands first, mid and last in a block
    (32, 8, 16, [1, 16, 17, 700]),
    (64, 8, 32, [32, 33, 1000, 2, 64]),
    (8, 8, 16, [5, 4096]),
    (16, 2, 32, [31]),
]


@pytest.mark.parametrize("case", APPEND_CASES, ids=lambda c: "nq%d_nkv%d_bs%d_%s" % (
    c[0], c[1], c[2], "-".join(map(str, c[3]))))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_append_decode_attention_one_call(case, num_splits):
    """The one-call append + attention: caches bit exact with the oracle's
    kv_append, output within tolerance of the oracle over those caches."""
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens, append=True)
    want, want_k, want_v = oracle_append_then_attend(pb)
    got = pgd.append_decode_attention(None, pb.q, pb.k_new, pb.v_new, pb.k_cache, pb.v_cache,
                                      pb.block_tables, pb.context_lens, pb.scale,
                                      num_splits=num_splits)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(pb.k_cache), want_k)
    assert np.array_equal(cache_bits(pb.v_cache), want_v)
    compare(got, want, "append+attend splits=%d" % num_splits)


def test_append_decode_attention_back_to_back():
    """Steps issued back to back on one stream (each attention may start its
    prologue while the append before it runs): every step sees its own
    append.  Step i appends token i of a growing context."""
    B, n_q, n_kv, bs = 3, 32, 8, 16
    base = [40, 15, 300]
    steps = 6
    pb = _batch(B, n_q, n_kv, bs, [n + steps for n in base], append=True)
    ws = pgd.make_workspace(B, n_q, n_kv)
    g = torch.Generator().manual_seed(99)
    k_seq = [torch.randn(B, n_kv, 128, generator=g).to(torch.bfloat16) for _ in range(steps)]
    v_seq = [torch.randn(B, n_kv, 128, generator=g).to(torch.bfloat16) for _ in range(steps)]
    k_ref, v_ref = pb.k_cache.cpu(), pb.v_cache.cpu()
    outs, wants = [], []
    for i in range(steps):
        lens = torch.tensor([n + i + 1 for n in base], dtype=torch.int32)
        kn, vn = k_seq[i].cuda(), v_seq[i].cuda()
        outs.append(pgd.append_decode_attention(None, pb.q, kn, vn, pb.k_cache, pb.v_cache,
                                                pb.block_tables, lens.cuda(), pb.scale,
                                                workspace=ws))
        k_ref, v_ref = oracle.kv_append(k_ref, v_ref, k_seq[i], v_seq[i], pb.block_tables.cpu(),
                                        lens - 1)
        wants.append(oracle.paged_attention(pb.q.cpu(), k_ref, v_ref, pb.block_tables.cpu(), lens,
                                            pb.scale))
    torch.cuda.synchronize()
    for i in range(steps):
        compare(outs[i], wants[i], "step %d" % i)
    assert np.array_equal(cache_bits(pb.k_cache), k_ref)
    assert np.array_equal(cache_bits(pb.v_cache), v_ref)


def test_copy_blocks_bit_exact():
    pb = _batch(3, 8, 2, 16, [100, 64, 33])
    src = torch.tensor([0, 3, 5], dtype=torch.int32, device="cuda")
    dst = torch.tensor([7, 1, 2], dtype=torch.int32, device="cuda")
    k0, v0 = pb.k_cache.clone(), pb.v_cache.clone()
    pgd.copy_blocks(pb.k_cache, pb.v_cache, src, dst)
    torch.cuda.synchronize()
    k0v = k0.view(torch.int16); v0v = v0.view(torch.int16)
    for s, d in zip(src.tolist(), dst.tolist()):
        k0v[d] = k0v[s]
        v0v[d] = v0v[s]
    assert torch.equal(pb.k_cache.view(torch.int16), k0v)
    assert torch.equal(pb.v_cache.view(torch.int16), v0v)


@pytest.mark.parametrize("lens", [[700, 16, 17, 1], [2048, 16, 17, 1]], ids=["short", "tc"])
@pytest.mark.parametrize("pinned", ["all", "none", "mixed"])
def test_decode_step_host_buffers_match_device_path(pinned, lens):
    """Page-locked host buffers are read and written in place by the kernels,
    pageable ones go through the device buffers and copies (each buffer on its
    own): every mix equals the device path bit for bit, on the short-context
    kernel and on the tensor-core kernel."""
    B, n_q, n_kv, bs = 4, 32, 8, 16
    pb = _batch(B, n_q, n_kv, bs, lens, append=True)
    ws = pgd.make_workspace(B, n_q, n_kv)
    pin = lambda t: t.cpu().pin_memory()
    page = lambda t: t.cpu().clone()
    hq, hk, hv, ho, hc = {"all": (pin,) * 5, "none": (page,) * 5,
                          "mixed": (pin, page, pin, page, page)}[pinned]
    q_h = hq(pb.q)
    kn_h, vn_h = hk(pb.k_new), hv(pb.v_new)
    cl_h = hc(pb.context_lens)
    out_h = ho(torch.zeros_like(pb.q))
    q_d, kn_d, vn_d = torch.empty_like(pb.q), torch.empty_like(pb.k_new), torch.empty_like(pb.v_new)
    cl_d = torch.empty_like(pb.context_lens)
    out_d = torch.empty_like(pb.q)
    pgd.decode_step(out_h, q_h, kn_h, vn_h, cl_h, out_d, q_d, kn_d, vn_d, cl_d, pb.k_cache,
                    pb.v_cache, pb.block_tables, pb.scale, 0, ws)
    torch.cuda.synchronize()
    ref = gpu_attention(pb)
    assert torch.equal(out_h, ref.cpu())
    compare(out_h, oracle_attention(pb))


# ------------------------------------------------- workloads at full size
@pytest.mark.parametrize("name", ["single_ctx512", "batch16_ctx8192", "mha40_batch4_ctx8192",
                                  "shared_prefix32", "ragged64_g8", "single_ctx131072"])
def test_workload_full_size(name):
    pb = inputs.make_workload(name, device="cuda")
    if pb.k_new is not None:
        want, _, _ = oracle_append_then_attend(pb)
        pgd.kv_append(pb.k_new, pb.v_new, pb.k_cache, pb.v_cache, pb.block_tables, pb.positions)
    else:
        want = oracle_attention(pb)
    compare(gpu_attention(pb), want, name)


def test_bad_block_id_is_flagged_and_contained():
    """A table entry outside [0, NB) inside a sequence's context is caught by
    the kernel's range check: nothing is read through it, the device error
    word gets PGD_DEVERR_BAD_BLOCK_ID, and the other sequences' outputs are
    unaffected."""
    lens = [300, 300, 300]
    pb = inputs.make_batch(3, 32, 8, 16, lens, device="cuda", seed=5, table_seed=6)
    want = oracle_attention(pb)
    tables = pb.block_tables.clone()
    tables[1, 7] = pb.num_blocks + 5
    out = pgd.paged_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, tables,
                                     pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    flags = pgd.device_errors(clear=True)
    assert flags & 1, "device error word %d lacks the bad-block bit" % flags
    got = out.float().cpu().double().numpy()
    for b in (0, 2):
        err = np.abs(got[b] - want[b])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_reference_moves_mid_context(G, num_splits):
    """K tiles of later blocks scaled by 8 and then by 32 (exact in bf16): the
    scores of every head with a nonzero query jump by far more than 2^8 twice
    after the first stages, so the softmax votes, moves the references and
    rescales O mid-unit (and inside split parts); heads with a zero query
    (scores all 0) keep factor 1."""
    lens = [1500, 1300, 1700]
    pb = _batch(len(lens), 2 * G, 2, 16, lens, seed=41 + G)
    for b, n in enumerate(lens):
        for j in range(-(-n // 16)):
            f = 32.0 if j >= 64 else (8.0 if j >= 32 else 1.0)
            pb.k_cache[int(pb.block_tables[b, j])] *= f
    pb.q[:, ::3] = 0
    compare(gpu_attention(pb, num_splits), oracle_attention(pb),
            "G=%d splits=%d" % (G, num_splits))

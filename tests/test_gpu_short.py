"""The short-context kernel (contexts of at most 1024 tokens, at most 64
(sequence, KV head) units and 40960 unit-tokens, automatic split): parity
with the float64 oracle, the fused append bit for bit, masking and error
flags, and agreement with the tensor-core kernel on the same inputs (the
limit set to 0 routes a call there).  Every case asserts which kernel its
sizes select."""
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
def _clean():
    pgd.device_errors(clear=True)
    yield
    pgd.set_short_context_tokens(-1)
    pgd.device_errors(clear=True)


def _batch(B, n_q, n_kv, bs, lens, seed=2024, **kw):
    return inputs.make_batch(B, n_q, n_kv, bs, lens, seed=seed, table_seed=seed + 3,
                             device="cuda", **kw)


def _short(pb) -> bool:
    return pgd.uses_short_path(pb.batch, pb.k_cache.shape[1], pb.block_size,
                               pb.block_tables.shape[1])


CASES = [
    # (n_q, n_kv, bs, lens): every length class of an eighth of the context --
    # empty CTAs (ctx < 8), one partial piece, a full piece, two pieces
    (4, 4, 16, [1]),
    (8, 8, 16, [2, 7, 8, 9]),
    (16, 2, 16, [63, 64, 65, 127, 128, 129]),
    (32, 8, 16, [512, 1, 1000, 1024]),
    (32, 8, 32, [31, 32, 33, 700, 1024]),
    (64, 8, 32, [129, 1000, 32]),
    (8, 1, 16, [300, 5, 513]),
    (40, 40, 16, [250]),
    # 64 units x 640 tokens: the most units and the most work the kernel takes
    (32, 8, 16, [633, 640, 1, 17, 600, 320, 5, 640]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "nq%d_nkv%d_bs%d_%s" % (
    c[0], c[1], c[2], "-".join(map(str, c[3][:6]))))
def test_short_matches_oracle(case):
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens)
    assert _short(pb)
    compare(gpu_attention(pb), oracle_attention(pb), "short")
    assert_no_device_errors()


@pytest.mark.parametrize("case", CASES[2:6], ids=lambda c: "nq%d_nkv%d_bs%d" % c[:3])
def test_short_and_tensor_core_kernels_agree(case):
    """The same call through both kernels: each within tolerance of the
    oracle, and within twice the tolerance of each other."""
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens, seed=77)
    want = oracle_attention(pb)
    a = gpu_attention(pb)
    pgd.set_short_context_tokens(0)
    b = gpu_attention(pb)
    torch.cuda.synchronize()
    compare(a, want, "short")
    compare(b, want, "tensor-core")
    d = (a.float() - b.float()).abs()
    assert float(d.max()) <= 4e-2 and float(d.mean()) <= 4e-3
    assert_no_device_errors()


def test_unit_and_context_limits_select_the_kernel():
    assert pgd.uses_short_path(8, 8, 16, 40)           # 64 units x 640 tokens = 40960
    assert pgd.uses_short_path(4, 8, 16, 64)           # 32 units x 1024 tokens
    assert not pgd.uses_short_path(8, 8, 16, 41)       # 64 x 656 > 40960
    assert not pgd.uses_short_path(9, 8, 16, 8)        # 72 units
    assert not pgd.uses_short_path(1, 8, 16, 65)       # 1040 tokens
    assert not pgd.uses_short_path(1, 8, 16, 8, num_splits=1)
    prev = pgd.set_short_context_tokens(256)
    assert prev == 1024
    assert pgd.uses_short_path(1, 8, 16, 16) and not pgd.uses_short_path(1, 8, 16, 17)
    pgd.set_short_context_tokens(0)
    assert not pgd.uses_short_path(1, 8, 16, 1)
    assert pgd.set_short_context_tokens(-1) == 0


@pytest.mark.parametrize("lens", [[300] * 17, [650] * 8], ids=["136-units", "64x656-tokens"])
def test_just_past_the_limits_uses_the_tensor_core_kernel(lens):
    pb = _batch(len(lens), 32, 8, 16, lens, seed=5)
    assert not _short(pb)
    compare(gpu_attention(pb), oracle_attention(pb), "past the limits")
    assert_no_device_errors()


APPEND_CASES = [
    # the new token first, mid and last in its block, and alone in its context
    (32, 8, 16, [1, 16, 17, 700]),
    (64, 8, 32, [32, 33, 1000, 2, 64]),
    (16, 2, 32, [31, 1024]),
    (4, 1, 16, [8, 9, 65]),
]


@pytest.mark.parametrize("case", APPEND_CASES, ids=lambda c: "nq%d_nkv%d_bs%d_%s" % (
    c[0], c[1], c[2], "-".join(map(str, c[3]))))
def test_short_fused_append(case):
    """One launch appends and attends: caches bit exact with the oracle's
    kv_append, output within tolerance of the oracle over those caches."""
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens, append=True)
    assert _short(pb)
    want, want_k, want_v = oracle_append_then_attend(pb)
    got = pgd.append_decode_attention(None, pb.q, pb.k_new, pb.v_new, pb.k_cache, pb.v_cache,
                                      pb.block_tables, pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(pb.k_cache), want_k)
    assert np.array_equal(cache_bits(pb.v_cache), want_v)
    compare(got, want, "fused append")
    assert_no_device_errors()


def test_short_decode_steps_grow_across_blocks():
    """Twenty fused steps on one stream, contexts crossing block boundaries:
    every step sees its own append, and the caches end bit exact."""
    B, n_q, n_kv, bs = 2, 16, 4, 16
    base, steps = [14, 40], 20
    pb = _batch(B, n_q, n_kv, bs, [n + steps for n in base], append=True, seed=9)
    g = torch.Generator().manual_seed(19)
    k_ref, v_ref = pb.k_cache.cpu(), pb.v_cache.cpu()
    outs, wants = [], []
    for i in range(steps):
        lens = torch.tensor([n + i + 1 for n in base], dtype=torch.int32)
        kn = torch.randn(B, n_kv, 128, generator=g).to(torch.bfloat16)
        vn = torch.randn(B, n_kv, 128, generator=g).to(torch.bfloat16)
        outs.append(pgd.append_decode_attention(None, pb.q, kn.cuda(), vn.cuda(), pb.k_cache,
                                                pb.v_cache, pb.block_tables, lens.cuda(),
                                                pb.scale))
        k_ref, v_ref = oracle.kv_append(k_ref, v_ref, kn, vn, pb.block_tables.cpu(), lens - 1)
        wants.append(oracle.paged_attention(pb.q.cpu(), k_ref, v_ref, pb.block_tables.cpu(), lens,
                                            pb.scale))
    torch.cuda.synchronize()
    for i in range(steps):
        compare(outs[i], wants[i], "step %d" % i)
    assert np.array_equal(cache_bits(pb.k_cache), k_ref)
    assert np.array_equal(cache_bits(pb.v_cache), v_ref)
    assert_no_device_errors()


def test_short_bad_block_id_is_flagged_and_contained():
    lens = [300, 300, 300]
    pb = _batch(3, 32, 8, 16, lens, seed=5)
    assert _short(pb)
    want = oracle_attention(pb)
    tables = pb.block_tables.clone()
    tables[1, 7] = pb.num_blocks + 5
    out = pgd.paged_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, tables,
                                     pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    assert pgd.device_errors(clear=True) & 1
    got = out.float().cpu().double().numpy()
    for b in (0, 2):
        err = np.abs(got[b] - want[b])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_short_bad_context_is_flagged_and_contained():
    lens = [200, 100, 50]
    pb = _batch(3, 16, 4, 16, lens, seed=6)
    want = oracle_attention(pb)
    ctx = pb.context_lens.clone()
    ctx[1] = 0
    out = pgd.paged_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables, ctx,
                                     pb.scale)
    torch.cuda.synchronize()
    assert pgd.device_errors(clear=True) & 2
    got = out.float().cpu().double().numpy()
    for b in (0, 2):
        err = np.abs(got[b] - want[b])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
    assert np.all(got[1] == 0.0)


# The tensor-core kernel on the small shapes that now take the short path
# (the limit set to 0), with the automatic split.
SMALL_TC = [
    (8, 4, 16, [16, 17, 1]),
    (16, 4, 16, [33, 200, 513]),
    (32, 4, 32, [64, 1, 95]),
    (32, 8, 16, [512]),
    (2, 1, 16, [47]),
]


@pytest.mark.parametrize("case", SMALL_TC, ids=lambda c: "nq%d_nkv%d_bs%d" % c[:3])
def test_tensor_core_kernel_on_short_contexts(case):
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens, seed=31)
    pgd.set_short_context_tokens(0)
    compare(gpu_attention(pb), oracle_attention(pb), "tensor-core, automatic split")
    assert_no_device_errors()


@pytest.mark.parametrize("limit", [-1, 0], ids=["short", "tensor-core"])
def test_prepared_calls_match_the_oracle(limit):
    """pgd.prepare: the arguments are checked and marshalled once and every
    call enqueues the same C-ABI call again.  Appending the same token twice
    leaves the same caches, so repeated calls give identical outputs."""
    pgd.set_short_context_tokens(limit)
    pb = _batch(2, 32, 8, 16, [300, 1024], append=True, seed=12)
    want, want_k, want_v = oracle_append_then_attend(pb)
    ws = pgd.make_workspace(2, 32, 8)
    step = pgd.prepare("append_decode_attention", None, pb.q, pb.k_new, pb.v_new, pb.k_cache,
                       pb.v_cache, pb.block_tables, pb.context_lens, pb.scale, workspace=ws)
    first = step().clone()
    again = step()
    attend = pgd.prepare("paged_decode_attention", None, pb.q, pb.k_cache, pb.v_cache,
                         pb.block_tables, pb.context_lens, pb.scale, workspace=ws)
    alone = attend()
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(pb.k_cache), want_k)
    assert np.array_equal(cache_bits(pb.v_cache), want_v)
    compare(first, want, "prepared step")
    assert torch.equal(first, again)
    compare(alone, want, "prepared attention")
    assert_no_device_errors()


# ------------------------------------------------------------ 8-bit cache
def _batch8(B, n_q, n_kv, bs, lens, seed=2024, **kw):
    return _batch(B, n_q, n_kv, bs, lens, seed=seed, kv_format="fp8", **kw)


def _oracle8(pb, k=None, v=None):
    return oracle.paged_attention_fp8(pb.q.cpu(), pb.k_cache.cpu() if k is None else k,
                                      pb.v_cache.cpu() if v is None else v, pb.block_tables.cpu(),
                                      pb.context_lens.cpu(), pb.scale, pb.block_size)


def _gpu8(pb):
    return pgd.paged_decode_attention_fp8(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                          pb.context_lens, pb.scale)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "nq%d_nkv%d_bs%d_%s" % (
    c[0], c[1], c[2], "-".join(map(str, c[3][:6]))))
def test_short_fp8_matches_oracle(case):
    n_q, n_kv, bs, lens = case
    pb = _batch8(len(lens), n_q, n_kv, bs, lens)
    assert _short(pb)
    compare(_gpu8(pb), _oracle8(pb), "short, 8-bit")
    assert_no_device_errors()


@pytest.mark.parametrize("case", CASES[2:6], ids=lambda c: "nq%d_nkv%d_bs%d" % c[:3])
def test_short_fp8_and_tensor_core_kernels_agree(case):
    n_q, n_kv, bs, lens = case
    pb = _batch8(len(lens), n_q, n_kv, bs, lens, seed=78)
    want = _oracle8(pb)
    a = _gpu8(pb)
    pgd.set_short_context_tokens(0)
    b = _gpu8(pb)
    torch.cuda.synchronize()
    compare(a, want, "short, 8-bit")
    compare(b, want, "tensor-core, 8-bit")
    assert_no_device_errors()


@pytest.mark.parametrize("case", APPEND_CASES, ids=lambda c: "nq%d_nkv%d_bs%d_%s" % (
    c[0], c[1], c[2], "-".join(map(str, c[3]))))
def test_short_fp8_fused_append(case):
    """One launch quantises the new token into the 8-bit pools (codes and
    scales bit exact with the oracle's kv_append_fp8) and attends over them."""
    n_q, n_kv, bs, lens = case
    pb = _batch8(len(lens), n_q, n_kv, bs, lens, append=True)
    assert _short(pb)
    want_k, want_v = oracle.kv_append_fp8(pb.k_cache.cpu(), pb.v_cache.cpu(), pb.k_new.cpu(),
                                          pb.v_new.cpu(), pb.block_tables.cpu(),
                                          pb.positions.cpu(), bs)
    want = _oracle8(pb, want_k, want_v)
    got = pgd.append_decode_attention_fp8(None, pb.q, pb.k_new, pb.v_new, pb.k_cache, pb.v_cache,
                                          pb.block_tables, pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    assert np.array_equal(pb.k_cache.cpu().numpy(), want_k)
    assert np.array_equal(pb.v_cache.cpu().numpy(), want_v)
    compare(got, want, "fused 8-bit append")
    assert_no_device_errors()


def test_short_fp8_fused_append_extreme_rows():
    """Rows of zeros, of one huge element, of tiny values and of values
    reaching 448 after scaling, appended by the short kernel: bit exact."""
    B, n_kv, bs = 4, 2, 16
    pb = _batch8(B, 8, n_kv, bs, [5, 16, 17, 40], append=True)
    kn = torch.zeros(B, n_kv, 128)
    kn[1, 0, 7] = 3e38
    kn[1, 1] = torch.linspace(-1e-30, 1e-30, 128)
    kn[2] = torch.linspace(-448, 448, 128)
    kn[3, 0] = torch.tensor([(-1) ** i * 2.0 ** (i % 40 - 20) for i in range(128)])
    kn = kn.to(torch.bfloat16).cuda()
    vn = (-kn).contiguous()
    want_k, want_v = oracle.kv_append_fp8(pb.k_cache.cpu(), pb.v_cache.cpu(), kn.cpu(), vn.cpu(),
                                          pb.block_tables.cpu(), pb.positions.cpu(), bs)
    pgd.append_decode_attention_fp8(None, pb.q, kn, vn, pb.k_cache, pb.v_cache, pb.block_tables,
                                    pb.context_lens, pb.scale)
    torch.cuda.synchronize()
    assert np.array_equal(pb.k_cache.cpu().numpy(), want_k)
    assert np.array_equal(pb.v_cache.cpu().numpy(), want_v)
    pgd.device_errors(clear=True)  # (a 3e38 row may give non-finite scores: not checked here)


def test_short_fp8_reference_moves():
    """K scales of later blocks multiplied by 8 and then 32: the scores jump
    by far more than 2^8 mid-context; every piece's maximum is exact, so the
    online softmax stays within tolerance."""
    lens = [1000, 700, 1024]
    pb = _batch8(len(lens), 8, 2, 16, lens, seed=43)
    codes, scales = inputs.unpack_pool8(pb.k_cache.cpu())
    for b, n in enumerate(lens):
        for jb in range(-(-n // 16)):
            f = 32.0 if jb >= 40 else (8.0 if jb >= 20 else 1.0)
            scales[int(pb.block_tables[b, jb])] *= f
    pb.k_cache.copy_(inputs.pack_pool8(codes, scales).cuda())
    pb.q[:, ::3] = 0
    assert _short(pb)
    compare(_gpu8(pb), _oracle8(pb), "8-bit, moved references")
    assert_no_device_errors()

"""Parity of the 8-bit (FP8 E4M3 + per-(token, head) scale) KV path, through
the C ABI, with the float64 oracle on the same seeded inputs.

kv_append_fp8: the pool bytes (codes and scales) bit exact.  Attention over
the 8-bit cache: max abs error <= 2e-2 and mean abs error <= 2e-3 against
the oracle's attention over the dequantised cache, every element.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import inputs
from gpu_common import assert_no_device_errors, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_errors():
    pgd.device_errors(clear=True)
    yield
    assert_no_device_errors()


def _batch(B, n_q, n_kv, bs, lens, seed=1234, **kw):
    return inputs.make_batch(B, n_q, n_kv, bs, lens, seed=seed, table_seed=seed + 7,
                             device="cuda", kv_format="fp8", **kw)


def oracle_fp8(pb, k=None, v=None):
    return oracle.paged_attention_fp8(pb.q.cpu(), (pb.k_cache if k is None else k),
                                      (pb.v_cache if v is None else v), pb.block_tables.cpu(),
                                      pb.context_lens.cpu(), pb.scale, pb.block_size)


def gpu_fp8(pb, num_splits=0, workspace=None):
    return pgd.paged_decode_attention_fp8(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                          pb.context_lens, pb.scale, num_splits=num_splits,
                                          workspace=workspace)


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
@pytest.mark.parametrize("num_splits", [0, 1, 3, 64])
def test_attention_fp8_small(case, num_splits):
    n_q, n_kv, bs, lens = case
    pb = _batch(len(lens), n_q, n_kv, bs, lens)
    compare(gpu_fp8(pb, num_splits), oracle_fp8(pb), "fp8 splits=%d" % num_splits)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_attention_fp8_ragged(G, bs):
    g = torch.Generator().manual_seed(G * 100 + bs)
    lens = torch.randint(1, 1500, (23,), generator=g).tolist()
    pb = _batch(len(lens), 4 * G, 4, bs, lens, seed=77 + G)
    compare(gpu_fp8(pb), oracle_fp8(pb), "fp8 ragged G=%d bs=%d" % (G, bs))


def test_attention_fp8_ctx1_is_the_scaled_value():
    """One cached token: the output is its dequantised V.  The V scale passes
    through one bf16 rounding inside the probability and the output through
    another, each with relative error at most 2^-8 (bf16 keeps 8 significant
    bits), so the relative error is at most (1 + 2^-8)^2 - 1."""
    pb = _batch(3, 16, 4, 16, [1, 1, 1])
    want = oracle_fp8(pb)
    got = gpu_fp8(pb).float().cpu().double().numpy()
    bound = (1 + 2.0 ** -8) ** 2 - 1
    rel = np.abs(got - want) / np.maximum(np.abs(want), 1e-30)
    assert np.all((rel <= bound * (1 + 1e-9)) | (want == 0)), rel.max()


@pytest.mark.parametrize("bs", [16, 32])
def test_kv_append_fp8_bit_exact(bs):
    lens = [1, bs, bs + 1, 2 * bs, 77, 3, 5 * bs - 1, 200, 64]
    pb = _batch(len(lens), 16, 4, bs, lens, append=True)
    k0, v0 = pb.k_cache.cpu(), pb.v_cache.cpu()
    want_k, want_v = oracle.kv_append_fp8(k0, v0, pb.k_new.cpu(), pb.v_new.cpu(),
                                          pb.block_tables.cpu(), pb.positions.cpu(), bs)
    pgd.kv_append_fp8(pb.k_new, pb.v_new, pb.k_cache, pb.v_cache, pb.block_tables, pb.positions)
    torch.cuda.synchronize()
    assert np.array_equal(pb.k_cache.cpu().numpy(), want_k)
    assert np.array_equal(pb.v_cache.cpu().numpy(), want_v)


def test_kv_append_fp8_extreme_rows():
    """Rows of zeros, of one huge element, of tiny values and of values
    reaching 448 after scaling quantise exactly as the oracle does."""
    B, n_kv, bs = 4, 2, 16
    pb = _batch(B, 8, n_kv, bs, [5, 16, 17, 40], append=True)
    kn = torch.zeros(B, n_kv, 128)
    kn[1, 0, 7] = 3e38
    kn[1, 1] = torch.linspace(-1e-30, 1e-30, 128)
    kn[2] = torch.linspace(-448, 448, 128)
    kn[3, 0] = torch.tensor([(-1) ** i * 2.0 ** (i % 40 - 20) for i in range(128)])
    kn = kn.to(torch.bfloat16).cuda()
    vn = (-kn).contiguous()
    want_k, want_v = oracle.kv_append_fp8(pb.k_cache.cpu(), pb.v_cache.cpu(), kn.cpu(), vn.cpu(),
                                          pb.block_tables.cpu(), pb.positions.cpu(), bs)
    pgd.kv_append_fp8(kn, vn, pb.k_cache, pb.v_cache, pb.block_tables, pb.positions)
    torch.cuda.synchronize()
    assert np.array_equal(pb.k_cache.cpu().numpy(), want_k)
    assert np.array_equal(pb.v_cache.cpu().numpy(), want_v)


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_append_decode_attention_fp8_one_call(num_splits):
    pb = _batch(5, 32, 8, 16, [1, 16, 17, 700, 2048], append=True)
    want_k, want_v = oracle.kv_append_fp8(pb.k_cache.cpu(), pb.v_cache.cpu(), pb.k_new.cpu(),
                                          pb.v_new.cpu(), pb.block_tables.cpu(),
                                          pb.positions.cpu(), 16)
    want = oracle_fp8(pb, want_k, want_v)
    got = pgd.append_decode_attention_fp8(None, pb.q, pb.k_new, pb.v_new, pb.k_cache, pb.v_cache,
                                          pb.block_tables, pb.context_lens, pb.scale,
                                          num_splits=num_splits)
    torch.cuda.synchronize()
    assert np.array_equal(pb.k_cache.cpu().numpy(), want_k)
    assert np.array_equal(pb.v_cache.cpu().numpy(), want_v)
    compare(got, want, "fp8 append+attend splits=%d" % num_splits)


@pytest.mark.parametrize("lens", [[5, 300, 17], [1, 16, 17, 700, 2048]], ids=["short", "tc"])
@pytest.mark.parametrize("pinned", ["all", "none", "mixed"])
def test_decode_step_fp8_host_buffers(pinned, lens):
    """The host-buffer step on an 8-bit pool: page-locked buffers read and
    written in place, pageable ones copied, each on its own.  Output and pool
    equal the device-buffer one-call step bit for bit, and the oracle."""
    pb = _batch(len(lens), 32, 8, 16, lens, append=True)
    kc0, vc0 = pb.k_cache.clone(), pb.v_cache.clone()
    want = pgd.append_decode_attention_fp8(None, pb.q, pb.k_new, pb.v_new, kc0, vc0,
                                           pb.block_tables, pb.context_lens, pb.scale)
    want_k, want_v = oracle.kv_append_fp8(pb.k_cache.cpu(), pb.v_cache.cpu(), pb.k_new.cpu(),
                                          pb.v_new.cpu(), pb.block_tables.cpu(),
                                          pb.positions.cpu(), 16)
    pin = lambda t: t.cpu().pin_memory()
    page = lambda t: t.cpu().clone()
    hq, hk, hv, ho, hc = {"all": (pin,) * 5, "none": (page,) * 5,
                          "mixed": (page, pin, page, pin, pin)}[pinned]
    q_h, kn_h, vn_h = hq(pb.q), hk(pb.k_new), hv(pb.v_new)
    cl_h, out_h = hc(pb.context_lens), ho(torch.zeros_like(pb.q))
    q_d, kn_d, vn_d = torch.empty_like(pb.q), torch.empty_like(pb.k_new), torch.empty_like(pb.v_new)
    cl_d, out_d = torch.empty_like(pb.context_lens), torch.empty_like(pb.q)
    ws = pgd.make_workspace(pb.batch, 32, 8)
    pgd.decode_step(out_h, q_h, kn_h, vn_h, cl_h, out_d, q_d, kn_d, vn_d, cl_d, pb.k_cache,
                    pb.v_cache, pb.block_tables, pb.scale, 0, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, want.cpu())
    assert np.array_equal(pb.k_cache.cpu().numpy(), want_k)
    assert np.array_equal(pb.v_cache.cpu().numpy(), want_v)
    compare(out_h, oracle_fp8(pb, want_k, want_v), "fp8 host-buffer step")


@pytest.mark.parametrize("name", ["single_ctx512", "batch16_ctx8192", "mha40_batch4_ctx8192",
                                  "ragged64_g8", "single_ctx131072"])
def test_workload_full_size_fp8(name):
    pb = inputs.make_workload(name, device="cuda", kv_format="fp8")
    k, v = pb.k_cache.cpu(), pb.v_cache.cpu()
    if pb.k_new is not None:
        k, v = oracle.kv_append_fp8(k, v, pb.k_new.cpu(), pb.v_new.cpu(), pb.block_tables.cpu(),
                                    pb.positions.cpu(), pb.block_size)
        pgd.kv_append_fp8(pb.k_new, pb.v_new, pb.k_cache, pb.v_cache, pb.block_tables,
                          pb.positions)
    compare(gpu_fp8(pb), oracle_fp8(pb, k, v), name + " fp8")


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fp8_reference_moves_mid_context(G, num_splits):
    """The per-token K scales (fp32, beside the codes) of later blocks
    multiplied by 8 and then by 32 -- exact, and read alike by the kernel and
    the oracle, as in the bf16 suite: scores reach about 190 in log2 units,
    every head with a nonzero query moves its reference (when its maximum
    grows past 2^8) after the first stages and rescales O; zero-query heads
    keep factor 1.  The kernel's query split is exact for bf16 elements
    within 2^9 of their head's largest, so the score error does not grow
    with the score beyond fp32 accumulation."""
    lens = [1500, 1300, 1700]
    pb = _batch(len(lens), 2 * G, 2, 16, lens, seed=61 + G)
    for b, n in enumerate(lens):
        for j in range(-(-n // 16)):
            f = 32.0 if j >= 64 else (8.0 if j >= 32 else 1.0)
            if f != 1.0:
                pb.k_cache[int(pb.block_tables[b, j]), :, :, 1024:].view(torch.float32).mul_(f)
    pb.q[:, ::3] = 0
    compare(gpu_fp8(pb, num_splits), oracle_fp8(pb), "fp8 rescale G=%d splits=%d" % (G, num_splits))


@pytest.mark.parametrize("G", [1, 8])
def test_fp8_query_dynamic_range(G):
    """Queries whose elements span many binades (a few of 2^12, most near 1,
    some near 2^-12) and a head of only tiny values (2^-100): the scores stay
    within tolerance of the oracle, which takes the bf16 query exactly."""
    lens = [700, 300]
    pb = _batch(len(lens), 2 * G, 2, 32, lens, seed=90 + G)
    g = torch.Generator().manual_seed(5)
    mag = torch.randint(-12, 13, pb.q.shape, generator=g).float()
    q = (torch.randn(pb.q.shape, generator=g) * torch.exp2(mag) / 64.0)
    q[:, 0] = torch.randn(q[:, 0].shape, generator=g) * 2.0 ** -100
    pb.q.copy_(q.to(torch.bfloat16))
    compare(gpu_fp8(pb), oracle_fp8(pb), "fp8 query range G=%d" % G)

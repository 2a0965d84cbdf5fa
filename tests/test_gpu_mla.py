"""Parity of decode attention over an MLA latent cache, through the C ABI,
with the float64 oracle on the same seeded inputs.

pgd_mla_append: the pool bit exact against the oracle's own append into a
CPU copy of the pool as generated.  Attention: max abs error <= 2e-2 and mean
abs error <= 2e-3 against the oracle, every element.
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


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _run(mb, num_splits=0):
    """Oracle append on a CPU copy, then the oracle's attention; GPU append,
    then attention.  Returns (gpu out, oracle out, oracle pool)."""
    pool = oracle.mla_append(mb.cache.cpu(), mb.c_new.cpu(), mb.block_tables.cpu(),
                             mb.positions.cpu()) if mb.c_new is not None else _bits(mb.cache)
    want = oracle.mla_attention(mb.q.cpu(), pool, mb.block_tables.cpu(), mb.context_lens.cpu(),
                                mb.scale)
    if mb.c_new is not None:
        pgd.mla_append(mb.c_new, mb.cache, mb.block_tables, mb.positions)
    got = pgd.mla_decode_attention(None, mb.q, mb.cache, mb.block_tables, mb.context_lens,
                                   mb.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return got, want, pool


SMALL = [
    # (heads, bs, lens)
    (16, 16, [1]),
    (16, 16, [16, 17, 63, 64, 65]),
    (64, 32, [100, 7, 129]),
    (128, 64, [64, 300, 1000]),
    (128, 16, [513, 2]),
    (32, 64, [1, 640]),
    (100, 32, [77, 200]),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "H%d_bs%d_%s" % (
    c[0], c[1], "-".join(map(str, c[2]))))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_mla_small(case, num_splits):
    H, bs, lens = case
    mb = inputs.make_mla_batch(len(lens), H, bs, lens, append=True, device="cuda",
                               seed=91 + H, table_seed=92)
    got, want, pool = _run(mb, num_splits)
    assert np.array_equal(_bits(mb.cache), pool)
    compare(got, want, "mla H=%d bs=%d splits=%d" % (H, bs, num_splits))


@pytest.mark.parametrize("bs", [16, 64])
def test_mla_ragged(bs):
    g = torch.Generator().manual_seed(bs)
    lens = torch.randint(1, 3000, (13,), generator=g).tolist()
    mb = inputs.make_mla_batch(len(lens), 128, bs, lens, append=True, device="cuda", seed=7)
    got, want, _ = _run(mb)
    compare(got, want, "mla ragged bs=%d" % bs)


def test_mla_ctx1_is_the_latent():
    """One cached token: each head returns its first 512 values (a bf16
    value through a bf16 probability of exactly 1)."""
    mb = inputs.make_mla_batch(3, 64, 16, [1, 1, 1], device="cuda")
    got = pgd.mla_decode_attention(None, mb.q, mb.cache, mb.block_tables, mb.context_lens,
                                   mb.scale)
    rows = inputs.untile_latent(mb.cache)
    for b in range(3):
        want = rows[int(mb.block_tables[b, 0]), 0, :512]
        assert torch.equal(got[b].view(torch.int16), want.expand(64, 512).view(torch.int16))


def test_mla_workload_batch16_ctx8192():
    """16 sequences x 8192 tokens, 128 heads, block 64, at full size."""
    mb = inputs.make_mla_workload("mla128_batch16_ctx8192", device="cuda")
    got, want, _ = _run(mb)
    compare(got, want, "mla128 batch16 ctx8192")


def test_mla_rescale_mid_context():
    """The RoPE part (values 512..575, tile columns 64..71) of later blocks
    scaled by 8 and then by 32 (exact in bf16): scores grow, the latent
    values the output averages do not.  The running maximum of each head with
    a nonzero query jumps by far more than 2^8 twice after the first stage, so
    the O^T columns of those heads are rescaled mid-context while the heads
    with a zero query (scores all 0) keep factor 1 -- with one part per
    context and with several."""
    lens = [640, 600, 700]
    mb = inputs.make_mla_batch(len(lens), 128, 64, lens, device="cuda", seed=13, table_seed=14)
    for b, n in enumerate(lens):
        for j in range(-(-n // 64)):
            f = 32.0 if j >= 7 else (8.0 if j >= 4 else 1.0)
            blk = int(mb.block_tables[b, j])
            mb.cache[blk, :, 64:72] *= f
    mb.q[:, :16] = 0
    for splits in (0, 1, 2):
        got, want, _ = _run(mb, splits)
        compare(got, want, "mla rescale splits=%d" % splits)


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_mla_append_decode_attention_one_call(num_splits):
    """The one-call step (append at context_lens - 1, then attention): the
    pool bit exact with the oracle's own append, the output within tolerance
    of the oracle over it."""
    lens = [1, 64, 65, 700, 2500]
    mb = inputs.make_mla_batch(len(lens), 128, 32, lens, append=True, device="cuda", seed=44,
                               table_seed=45)
    pool = oracle.mla_append(mb.cache.cpu(), mb.c_new.cpu(), mb.block_tables.cpu(),
                             mb.positions.cpu())
    want = oracle.mla_attention(mb.q.cpu(), pool, mb.block_tables.cpu(), mb.context_lens.cpu(),
                                mb.scale)
    got = pgd.mla_append_decode_attention(None, mb.q, mb.c_new, mb.cache, mb.block_tables,
                                          mb.context_lens, mb.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(mb.cache), pool)
    compare(got, want, "mla append+attend splits=%d" % num_splits)


@pytest.mark.parametrize("pinned", ["all", "none", "mixed"])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_mla_step_host_buffers(pinned, num_splits):
    """pgd_mla_step: q copied, page-locked c_new / context lengths / out read
    and written in place, pageable ones copied, each on its own; output and
    pool equal the device-buffer one-call step bit for bit, and the oracle."""
    lens = [1, 64, 65, 700, 2500]
    mb = inputs.make_mla_batch(len(lens), 128, 32, lens, append=True, device="cuda", seed=46,
                               table_seed=47)
    pool = oracle.mla_append(mb.cache.cpu(), mb.c_new.cpu(), mb.block_tables.cpu(),
                             mb.positions.cpu())
    want = oracle.mla_attention(mb.q.cpu(), pool, mb.block_tables.cpu(), mb.context_lens.cpu(),
                                mb.scale)
    cache2 = mb.cache.clone()
    ws = torch.empty(max(256, pgd.mla_workspace_size(len(lens), 128, num_splits)),
                     dtype=torch.uint8, device="cuda")
    dev = pgd.mla_append_decode_attention(None, mb.q, mb.c_new, cache2, mb.block_tables,
                                          mb.context_lens, mb.scale, num_splits=num_splits,
                                          workspace=ws)
    torch.cuda.synchronize()
    pin = lambda t: t.cpu().pin_memory()
    page = lambda t: t.cpu().clone()
    hq, hc, hl, ho = {"all": (pin,) * 4, "none": (page,) * 4,
                      "mixed": (page, pin, page, pin)}[pinned]
    out_d = torch.empty_like(dev)
    out_h = ho(torch.zeros_like(dev))
    pgd.mla_step(out_h, hq(mb.q), hc(mb.c_new), hl(mb.context_lens), out_d,
                 torch.empty_like(mb.q), torch.empty_like(mb.c_new),
                 torch.empty_like(mb.context_lens), mb.cache, mb.block_tables, mb.scale,
                 num_splits, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), dev.cpu().view(torch.int16))
    assert np.array_equal(_bits(mb.cache), _bits(cache2))
    assert np.array_equal(_bits(mb.cache), pool)
    compare(out_h, want, "mla host-buffer step %s splits=%d" % (pinned, num_splits))


def test_mla_steps_back_to_back():
    """Six one-call steps on one stream with a growing context (each
    attention's prologue overlapping the append before it): every step sees
    its own append."""
    base, steps = [300, 63, 1500], 6
    mb = inputs.make_mla_batch(3, 64, 64, [n + steps for n in base], append=True, device="cuda",
                               seed=46, table_seed=47)
    g = torch.Generator().manual_seed(48)
    rows = [torch.randn(3, 576, generator=g).to(torch.bfloat16) for _ in range(steps)]
    pool = _bits(mb.cache)
    ws = torch.empty(pgd.mla_workspace_size(3, 64, 0), dtype=torch.uint8, device="cuda")
    outs, wants = [], []
    for i in range(steps):
        lens = torch.tensor([n + i + 1 for n in base], dtype=torch.int32)
        outs.append(pgd.mla_append_decode_attention(None, mb.q, rows[i].cuda(), mb.cache,
                                                    mb.block_tables, lens.cuda(), mb.scale,
                                                    workspace=ws))
        pool = oracle.mla_append(pool, rows[i], mb.block_tables.cpu(), lens - 1)
        wants.append(oracle.mla_attention(mb.q.cpu(), pool, mb.block_tables.cpu(), lens,
                                          mb.scale))
    torch.cuda.synchronize()
    for i in range(steps):
        compare(outs[i], wants[i], "step %d" % i)
    assert np.array_equal(_bits(mb.cache), pool)


@pytest.mark.parametrize("H", [64, 128])
def test_mla_long_ragged_sequences(H):
    """Few long sequences of different lengths under the automatic split:
    every sequence is cut into the same number of parts, of different
    lengths, merged by the combine kernel."""
    lens = [9000, 5000, 3000, 257]
    mb = inputs.make_mla_batch(len(lens), H, 64, lens, append=True, device="cuda", seed=50,
                               table_seed=51)
    got, want, _ = _run(mb)
    compare(got, want, "mla long ragged H=%d" % H)

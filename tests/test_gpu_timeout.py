"""The kernels' timeout exit, made to happen on purpose.

Every wait of a kernel's role on another role of its CTA is bounded; when the
bound runs out the kernel records PGD_DEVERR_TIMEOUT, stops issuing copies
and MMAs, lets its roles finish their walks with the remaining waits
returning at once, waits for the copies already in flight, frees its tensor
memory and exits.  Here the bound is set to 1 ns (pgd_set_wait_limit_ns), so
that any wait not met within its first polls gives up -- every kernel below
takes that exit.  Each test checks that the call returns, that the error word
reports the timeout, and that the next call with the default bound, on the
same stream and the same workspace (whose split counters the aborted call
must have left at zero), is within tolerance of the oracle.  No wait is left
unbounded and no access leaves its buffers on that path; nothing faults.
"""
import pytest
import torch

import oracle
import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import _native, inputs
from gpu_common import compare, oracle_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _limit_restored():
    pgd.device_errors(clear=True)
    yield
    pgd.set_wait_limit_ns(0)
    pgd.device_errors(clear=True)


def _timed_out(call):
    pgd.set_wait_limit_ns(1)
    call()
    torch.cuda.synchronize()
    flags = pgd.device_errors(clear=True)
    pgd.set_wait_limit_ns(0)
    assert flags & _native.DEVERR_TIMEOUT, "error word %d" % flags


@pytest.mark.parametrize("num_splits", [0, 3])
def test_decode_timeout_then_normal_call(num_splits):
    pb = inputs.make_batch(12, 32, 8, 16, [3000, 17, 900, 2048, 1, 5000, 64, 333, 1200, 4096,
                                           700, 16], device="cuda", seed=31)
    ws = pgd.make_workspace(pb.batch, 32, 8, num_splits)
    out = torch.empty_like(pb.q)

    def call():
        pgd.paged_decode_attention(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                   pb.context_lens, pb.scale, num_splits=num_splits, workspace=ws)
    _timed_out(call)
    call()
    torch.cuda.synchronize()
    assert pgd.device_errors(clear=True) == 0
    compare(out, oracle_attention(pb), "after a timeout, splits=%d" % num_splits)


def test_fp8_timeout_then_normal_call():
    pb = inputs.make_batch(6, 32, 8, 16, [2500, 1, 700, 4000, 130, 64], device="cuda", seed=32,
                           kv_format="fp8")
    ws = pgd.make_workspace(pb.batch, 32, 8)
    out = torch.empty_like(pb.q)

    def call():
        pgd.paged_decode_attention_fp8(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                       pb.context_lens, pb.scale, workspace=ws)
    _timed_out(call)
    call()
    torch.cuda.synchronize()
    assert pgd.device_errors(clear=True) == 0
    want = oracle.paged_attention_fp8(pb.q.cpu(), pb.k_cache, pb.v_cache, pb.block_tables.cpu(),
                                      pb.context_lens.cpu(), pb.scale, pb.block_size)
    compare(out, want, "8-bit after a timeout")


def test_mla_timeout_then_normal_call():
    mb = inputs.make_mla_batch(3, 128, 64, [3000, 64, 1100], device="cuda", seed=33)
    ws = torch.zeros(max(256, pgd.mla_workspace_size(3, 128, 0)), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((3, 128, inputs.MLA_DV), dtype=torch.bfloat16, device="cuda")

    def call():
        pgd.mla_decode_attention(out, mb.q, mb.cache, mb.block_tables, mb.context_lens, mb.scale,
                                 workspace=ws)
    _timed_out(call)
    call()
    torch.cuda.synchronize()
    assert pgd.device_errors(clear=True) == 0
    want = oracle.mla_attention(mb.q.cpu(), mb.cache.cpu(), mb.block_tables.cpu(),
                                mb.context_lens.cpu(), mb.scale)
    compare(out, want, "MLA after a timeout")


def test_cascade_timeout_then_normal_call():
    B, bs, shared = 10, 16, 40
    g = torch.Generator().manual_seed(34)
    lens = [shared * bs + int(s) for s in torch.randint(1, 400, (B,), generator=g)]
    pb = inputs.make_batch(B, 32, 8, bs, lens, shared_prefix=shared * bs, seed=34,
                           table_seed=35, device="cuda")
    seq, gf, gs, gb, mgs, mgb = inputs.prefix_groups(pb, [(0, B, shared)])
    ws = torch.zeros(pgd.cascade_workspace_size(B, 32, 8, bs, mgs, mgb, 0), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(pb.q)

    def call():
        pgd.cascade_decode_attention(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                     pb.context_lens, seq, gf, gs, gb, mgs, mgb, pb.scale,
                                     workspace=ws)
    _timed_out(call)
    call()
    torch.cuda.synchronize()
    assert pgd.device_errors(clear=True) == 0
    compare(out, oracle_attention(pb), "cascade after a timeout")

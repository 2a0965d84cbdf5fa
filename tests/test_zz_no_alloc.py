"""The allocation-free attention entry point, checked against the regular one.

pgd_paged_decode_attention_noalloc is for callers that cannot allocate device
memory -- a plugin or callback running inside another runtime's execution
step gets its inputs and outputs but no scratch, and must not call
cudaMalloc/cudaFree there.  The entry point keeps the split-merge scratch in
a fixed device array owned by the library.  Here it is called through the C
ABI twice in a row and each result is compared with the regular entry point
(caller-provided workspace) and with the float64 oracle, within the attention
tolerances of the parity tests -- including a ragged batch long enough that
the automatic split cuts sequences into parts merged through the scratch; a
size whose scratch would not fit the array must be refused.

This file is named to be collected last, so a run that stops at the first
failure has run every other test first; it also passes alone.
"""
import pytest
import torch

import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import _native, inputs
from gpu_common import MAX_ABS, MEAN_ABS, compare, oracle_attention

pytestmark = pytest.mark.gpu


def _close(a, b):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS


CASES = {
    # a small batch of mixed lengths
    "mixed5": (5, 32, 8, 16, [700, 33, 4096, 1, 129]),
    # one long sequence among short ones: the automatic split cuts it into
    # parts, whose partial states go through the scratch and are merged
    "ragged_long": (6, 16, 2, 32, [20000, 3, 64, 1500, 31, 900]),
}


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_regular_entry_point_and_oracle_twice(case, num_splits):
    B, n_q, n_kv, bs, lens = CASES[case]
    pb = inputs.make_batch(B, n_q, n_kv, bs, lens, device="cuda", seed=77)
    ref = pgd.paged_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                     pb.context_lens, pb.scale, num_splits=num_splits)
    want = oracle_attention(pb)
    compare(ref, want, "regular %s splits=%d" % (case, num_splits))
    for i in range(2):
        out = torch.full_like(pb.q, float("nan"))
        pgd.paged_decode_attention_noalloc(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                           pb.context_lens, pb.scale, num_splits=num_splits)
        torch.cuda.synchronize()
        _close(out, ref)
        compare(out, want, "noalloc %s splits=%d call %d" % (case, num_splits, i))
    assert pgd.device_errors(clear=True) == 0


def test_noalloc_refuses_sizes_beyond_its_array():
    pb = inputs.make_batch(64, 64, 8, 32, [64] * 64, device="cuda", seed=78)
    need = pgd.workspace_size(64, 64, 8, num_splits=64)
    assert need > (16 << 20)
    out = torch.empty_like(pb.q)
    with pytest.raises(pgd.PGDError) as e:
        pgd.paged_decode_attention_noalloc(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                           pb.context_lens, pb.scale, num_splits=64)
    assert e.value.status == _native.ERR_WORKSPACE

"""The allocation-free attention entry point, checked against the regular one.

pgd_paged_decode_attention_noalloc is for callers that cannot allocate device
memory -- a plugin or callback running inside another runtime's execution
step gets its inputs and outputs but no scratch, and must not call
cudaMalloc/cudaFree there.  The entry point keeps the split-merge scratch in
a fixed device array owned by the library.  Here it is called through the C
ABI twice in a row and each result is compared with the regular entry point
(caller-provided workspace) within the attention tolerances of the parity
tests; a size whose scratch would not fit the array must be refused.

This file is named to be collected last, so a run that stops at the first
failure has run every other test first; it also passes alone.
"""
import pytest
import torch

import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import _native, inputs
from gpu_common import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu


def _close(a, b):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS


@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_regular_entry_point_twice(num_splits):
    pb = inputs.make_batch(5, 32, 8, 16, [700, 33, 4096, 1, 129], device="cuda", seed=77)
    ref = pgd.paged_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                     pb.context_lens, pb.scale, num_splits=num_splits)
    for _ in range(2):
        out = torch.full_like(pb.q, float("nan"))
        pgd.paged_decode_attention_noalloc(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                           pb.context_lens, pb.scale, num_splits=num_splits)
        torch.cuda.synchronize()
        _close(out, ref)
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

"""The read-only streaming pass (pgd_read_stream), the third bandwidth
denominator of the benchmark: both access patterns run over sizes that leave
some CTAs without work, end on partial stages, or span many stages, without a
device error, and leave the source unchanged."""
import pytest
import torch

import paged_gqa_decode_kv_gb300 as pgd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("nbytes", [4096, 7 * 4096, 1000 * 4096, 3 * 65536 + 4096, 64 << 20])
def test_read_stream_runs_clean(mode, nbytes):
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 2 ** 31 - 1, (nbytes // 4,), dtype=torch.int32, device="cuda",
                        generator=g)
    before = src.clone()
    pgd.read_stream(src, mode)
    pgd.read_stream(src, mode)
    assert pgd.device_errors(clear=True) == 0
    assert torch.equal(src, before)

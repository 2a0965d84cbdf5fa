"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and
compare it with the oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
import paged_gqa_decode_kv_gb300 as pgd

# Tolerances of the attention output (bf16) against the float64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def oracle_attention(pb, n_threads: int = 0) -> np.ndarray:
    return oracle.paged_attention(pb.q.cpu(), pb.k_cache.cpu(), pb.v_cache.cpu(),
                                  pb.block_tables.cpu(), pb.context_lens.cpu(), pb.scale,
                                  n_threads=n_threads)


def oracle_append_then_attend(pb, n_threads: int = 0):
    """The oracle's own kv_append (on CPU copies of the caches as generated,
    before any GPU append), then its attention over the result.  Returns
    (out, k_cache, v_cache) with the caches as uint16 bit patterns."""
    k, v = oracle.kv_append(pb.k_cache.cpu(), pb.v_cache.cpu(), pb.k_new.cpu(), pb.v_new.cpu(),
                            pb.block_tables.cpu(), pb.positions.cpu())
    out = oracle.paged_attention(pb.q.cpu(), k, v, pb.block_tables.cpu(), pb.context_lens.cpu(),
                                 pb.scale, n_threads=n_threads)
    return out, k, v


def cache_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def gpu_attention(pb, num_splits: int = 0, workspace=None, out=None) -> torch.Tensor:
    return pgd.paged_decode_attention(out, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                      pb.context_lens, pb.scale, num_splits=num_splits,
                                      workspace=workspace)


def compare(got: torch.Tensor, want: np.ndarray, label: str = ""):
    g = got.float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), "%s: non-finite GPU output" % label
    err = np.abs(g - want)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, \
        "%s: max abs %.3g (tol %g), mean abs %.3g (tol %g)" % (label, mx, MAX_ABS, mean, MEAN_ABS)
    return mx, mean


def assert_no_device_errors():
    flags = pgd.device_errors(clear=True)
    assert flags == 0, "device error word = %d" % flags

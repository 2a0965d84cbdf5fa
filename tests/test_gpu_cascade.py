"""Cascade decode attention (shared prefixes read once per group, then each
sequence's suffix) through the C ABI against the oracle's plain attention
over the same paged cache: the cascade is a reordering of the same sum, so
the tolerance is the one of the decode path (max abs 2e-2, mean abs 2e-3)."""
import pytest
import torch

import paged_gqa_decode_kv_gb300 as pgd
from paged_gqa_decode_kv_gb300 import inputs
from gpu_common import assert_no_device_errors, compare, gpu_attention, oracle_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_errors():
    pgd.device_errors(clear=True)
    yield
    assert_no_device_errors()


def _shared_batch(B, n_q, n_kv, bs, shared_blocks, suffix_max, seed=5):
    g = torch.Generator().manual_seed(seed)
    suffix = torch.randint(1, suffix_max + 1, (B,), generator=g).tolist()
    lens = [shared_blocks * bs + s for s in suffix]
    return inputs.make_batch(B, n_q, n_kv, bs, lens, shared_prefix=shared_blocks * bs, seed=seed,
                             table_seed=seed + 1, device="cuda")


def cascade(pb, groups, num_splits=0):
    seq, gf, gs, gb, mgs, mgb = inputs.prefix_groups(pb, groups)
    return pgd.cascade_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                        pb.context_lens, seq, gf, gs, gb, mgs, mgb, pb.scale,
                                        num_splits=num_splits)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_one_group_all_sequences(G, bs):
    pb = _shared_batch(12, 4 * G, 4, bs, shared_blocks=9, suffix_max=300, seed=G + bs)
    compare(cascade(pb, [(0, 12, 9)]), oracle_attention(pb), "G=%d bs=%d" % (G, bs))


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_mixed_groups_and_ungrouped(num_splits):
    """Two groups with different shared lengths (both true prefixes of the
    batch's shared blocks) and ungrouped sequences."""
    pb = _shared_batch(20, 32, 8, 16, shared_blocks=40, suffix_max=500, seed=11)
    groups = [(0, 7, 40), (7, 6, 13)]  # sequences 13..19 take no part
    compare(cascade(pb, groups, num_splits), oracle_attention(pb), "splits=%d" % num_splits)


def test_group_larger_than_one_row_chunk():
    """G = 8: a chunk holds 16 sequences; a group of 40 takes three."""
    pb = _shared_batch(40, 64, 8, 32, shared_blocks=20, suffix_max=200, seed=3)
    compare(cascade(pb, [(0, 40, 20)]), oracle_attention(pb))


def test_long_prefix_split_in_parts():
    pb = _shared_batch(6, 32, 8, 16, shared_blocks=600, suffix_max=100, seed=9)
    compare(cascade(pb, [(0, 6, 600)]), oracle_attention(pb))


def test_one_block_prefix_and_one_token_suffix():
    pb = inputs.make_batch(5, 16, 4, 16, [17, 17, 17, 17, 17], shared_prefix=16, seed=2,
                           table_seed=3, device="cuda")
    compare(cascade(pb, [(0, 5, 1)]), oracle_attention(pb))


def test_no_groups_is_plain_attention():
    pb = _shared_batch(4, 32, 8, 16, shared_blocks=10, suffix_max=50)
    got = cascade(pb, [])
    assert torch.equal(got, gpu_attention(pb))


def test_workspace_reused_across_calls():
    pb = _shared_batch(16, 32, 8, 16, shared_blocks=30, suffix_max=200, seed=21)
    seq, gf, gs, gb, mgs, mgb = inputs.prefix_groups(pb, [(0, 16, 30)])
    n = pgd.cascade_workspace_size(pb.batch, pb.n_q, pb.n_kv, 16, mgs, mgb)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    outs = [pgd.cascade_decode_attention(None, pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                         pb.context_lens, seq, gf, gs, gb, mgs, mgb, pb.scale,
                                         workspace=ws) for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    compare(outs[0], oracle_attention(pb))


def test_shared_prefix32_full_size():
    pb = inputs.make_workload("shared_prefix32", device="cuda")
    want = oracle_attention(pb)
    got = cascade(pb, [(0, pb.batch, pb.shared_blocks)])
    compare(got, want, "shared_prefix32")


@pytest.mark.parametrize("G", [1, 4])
def test_prefix_rescale_mid_prefix(G):
    """The shared prefix's later blocks scaled by 8 and then by 32 (exact in
    bf16): in the prefix pass each row with a nonzero query moves its
    reference twice after the first stage and rescales its O half, while
    rows with a zero query (scores all 0) keep factor 1."""
    pb = _shared_batch(10, 4 * G, 4, 16, shared_blocks=48, suffix_max=100, seed=21 + G)
    for j in range(48):
        f = 32.0 if j >= 32 else (8.0 if j >= 16 else 1.0)
        blk = int(pb.block_tables[0, j])
        pb.k_cache[blk] *= f
    pb.q[:, ::2] = 0
    compare(cascade(pb, [(0, 10, 48)]), oracle_attention(pb), "rescale G=%d" % G)

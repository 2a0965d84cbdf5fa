"""A whole decode lifecycle driven by the host block allocator, on the GPU.

Over 48 steps of one layer, sequences grow one token a step across block
boundaries (pgd_alloc_append_slot opens a block at each boundary), one is
forked mid-block (pgd_alloc_fork shares its partial last block, whose first
write takes the copy-on-write path: a private block and pgd_copy_blocks on
the device), another is forked exactly at a block boundary (full blocks stay
shared, the next write opens a new block), one finishes and releases its
blocks, and a later sequence reuses them.  Every step runs
pgd_append_decode_attention on the active sequences ("Module 10: inference
and serving", sections "Mapping logical positions to physical blocks" and
"Share only identical state"; "Ch. 6 Inference efficiency and serving", 6.4).

After each step:
  * the block tables and every reference count equal those of the plain
    block model (oracle.block_model), which replays the same operations;
  * both pools are bit-identical to the oracle's own copies, to which the
    test applies the oracle's kv_append and the same block copies;
  * the attention output is within tolerance of the float64 oracle over
    those copies.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_kv_gb300 as pgd
from oracle.block_model import BlockModel
from gpu_common import assert_no_device_errors, cache_bits, compare

pytestmark = pytest.mark.gpu

N_Q, N_KV, BS, MB, NB = 8, 2, 16, 8, 40
D = 128
STEPS = 48


class Seq:
    def __init__(self, name, row, n):
        self.name, self.row, self.n = name, row, n   # host table row, tokens cached


def test_allocator_driven_decode_lifecycle():
    dev = torch.device("cuda")
    alloc = pgd.BlockAllocator(NB)
    model = BlockModel(NB)
    nan = float("nan")
    shape = (NB, N_KV, BS // 8, D // 8, 8, 8)
    k = torch.full(shape, nan, dtype=torch.bfloat16, device=dev)
    v = torch.full(shape, nan, dtype=torch.bfloat16, device=dev)
    k_ref, v_ref = cache_bits(k), cache_bits(v)
    scale = D ** -0.5
    g = torch.Generator().manual_seed(2024)
    ws = pgd.make_workspace(8, N_Q, N_KV)

    active = [Seq("A", [-1] * MB, 0), Seq("C", [-1] * MB, 0)]
    mrows = {"A": [-1] * MB, "C": [-1] * MB}
    events = {"cow": 0, "opened": 0, "released": 0}

    def check_model():
        for s in active:
            assert s.row == mrows[s.name], s.name
        for i in range(NB):
            assert alloc.refcount(i) == model.refcount(i), i
        assert alloc.num_free == model.num_free()

    def fork(src, name, n_tokens):
        row, mrow = [-1] * MB, [-1] * MB
        alloc.fork(src.row, n_tokens, BS, row)
        model.fork(mrows[src.name], n_tokens, BS, mrow)
        mrows[name] = mrow
        active.append(Seq(name, row, n_tokens))

    for step in range(STEPS):
        if step == 5:
            active.append(Seq("B", [-1] * MB, 0))
            mrows["B"] = [-1] * MB
        if step == 20:
            fork(active[0], "D", active[0].n)          # A holds 20 tokens: mid-block
        if step == 34:
            d = next(s for s in active if s.name == "D")
            fork(d, "E", 32)                            # a block boundary of D
            assert next(s for s in active if s.name == "E").row[:2] == d.row[:2]
        if step == 30:
            c = next(s for s in active if s.name == "C")
            held = [i for i in c.row if i >= 0]
            alloc.release(held)
            model.release(held)
            active.remove(c)
            events["released"] += len(held)
        if step == 32:
            active.append(Seq("F", [-1] * MB, 0))      # takes C's freed blocks
            mrows["F"] = [-1] * MB
        check_model()

        # make each sequence's next slot writable: open a block or copy on write
        cow_src, cow_dst = [], []
        for s in active:
            j = s.n // BS
            before = s.row[j]
            src, dst = alloc.append_slot(s.row, s.n, BS)
            chosen = s.row[j] if s.row[j] != before else None
            msrc, mdst = model.append_slot(mrows[s.name], s.n, BS, chosen=chosen)
            assert (src, dst) == (msrc, mdst)
            if src >= 0:
                cow_src.append(src)
                cow_dst.append(dst)
                events["cow"] += 1
            elif before < 0:
                events["opened"] += 1
        check_model()
        if cow_src:
            pgd.copy_blocks(k, v, torch.tensor(cow_src, dtype=torch.int32, device=dev),
                            torch.tensor(cow_dst, dtype=torch.int32, device=dev))
            for a, b in zip(cow_src, cow_dst):
                k_ref[b] = k_ref[a]
                v_ref[b] = v_ref[a]

        B = len(active)
        tables = torch.tensor([s.row for s in active], dtype=torch.int32)
        lens = torch.tensor([s.n + 1 for s in active], dtype=torch.int32)
        pgd.validate_tables(tables, lens, NB, BS)
        q = torch.randn(B, N_Q, D, generator=g).to(torch.bfloat16)
        kn = torch.randn(B, N_KV, D, generator=g).to(torch.bfloat16)
        vn = torch.randn(B, N_KV, D, generator=g).to(torch.bfloat16)
        out = pgd.append_decode_attention(None, q.to(dev), kn.to(dev), vn.to(dev), k, v,
                                          tables.to(dev), lens.to(dev), scale, workspace=ws)
        k_ref, v_ref = oracle.kv_append(k_ref, v_ref, kn, vn, tables, lens - 1)
        want = oracle.paged_attention(q, k_ref, v_ref, tables, lens, scale)
        torch.cuda.synchronize()
        compare(out, want, "step %d" % step)
        assert np.array_equal(cache_bits(k), k_ref), "K pool, step %d" % step
        assert np.array_equal(cache_bits(v), v_ref), "V pool, step %d" % step
        for s in active:
            s.n += 1

    assert_no_device_errors()
    # the scenario really took each path
    assert events["cow"] >= 1 and events["opened"] >= 8 and events["released"] >= 2
    alloc.close()

"""The host block allocator (C++, through the C ABI) against the plain-Python
block model of the pages' semantics (oracle.block_model), and the model
itself against scenarios the pages describe.  Integer work: bit exact."""
import random

import pytest
import torch

import paged_gqa_decode_kv_gb300 as pgd
from oracle import block_model
from oracle.block_model import BlockModel, OutOfBlocks, BlockError


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_gqa_decode_kv_gb300 import build
    build.build()


# ----------------------------------------------------- the model on its own
def test_model_growth_wastes_less_than_a_block():
    # "Module 10", mapping logical positions to physical blocks: a request
    # takes one more block as it grows; with bs = 16 at most 15 slots idle
    bs = 16
    m = BlockModel(100)
    row = [-1] * 20
    for pos in range(0, 16 * 5 + 3):
        m.append_slot(row, pos, bs)
        held = sum(1 for r in row if r >= 0)
        assert held == block_model.blocks_for(pos + 1, bs)
        assert held * bs - (pos + 1) <= bs - 1


def test_model_cow_keeps_the_other_sequence_intact():
    # "Share only identical state": forks share full prefix blocks; a write
    # into a shared partial block makes a private copy
    bs = 4
    m = BlockModel(20)
    a = [-1] * 8
    for pos in range(10):          # blocks 0, 1 full; block 2 holds 2 tokens
        m.append_slot(a, pos, bs)
    b = [-1] * 8
    m.fork(a, 10, bs, b)
    assert b[:3] == a[:3] and all(m.refcount(i) == 2 for i in a[:3])
    src, dst = m.append_slot(b, 10, bs)   # write into the shared partial block
    assert src == a[2] and dst not in a[:3] and b[2] == dst
    assert m.refcount(a[2]) == 1 and m.refcount(dst) == 1
    assert b[:2] == a[:2]                 # full prefix blocks stay shared
    assert m.append_slot(a, 10, bs) == (-1, -1)   # a's block is private again


def test_model_rejects_invalid():
    m = BlockModel(2)
    m.allocate(2)
    with pytest.raises(OutOfBlocks):
        m.allocate(1)
    with pytest.raises(BlockError):
        m.release([0, 0])
    with pytest.raises(BlockError):
        BlockModel(3).share([1])


# ------------------------------------------- the C++ allocator vs the model
def test_allocate_release_share_counts():
    a = pgd.BlockAllocator(8)
    ids = a.allocate(5)
    assert len(set(ids)) == 5 and a.num_free == 3
    a.share(ids[:2])
    assert [a.refcount(i) for i in ids] == [2, 2, 1, 1, 1]
    a.release(ids)
    assert a.num_free == 6
    a.release(ids[:2])
    assert a.num_free == 8 and a.refcount(ids[0]) == 0
    assert a.refcount(-1) == -1 and a.refcount(8) == -1


def test_all_or_nothing_failures():
    a = pgd.BlockAllocator(4)
    ids = a.allocate(3)
    with pytest.raises(pgd.PGDError) as e:
        a.allocate(2)
    assert e.value.status == 3 and a.num_free == 1
    with pytest.raises(pgd.PGDError) as e:
        a.release([ids[0], ids[0]])          # held once, released twice
    assert e.value.status == 6 and a.refcount(ids[0]) == 1
    with pytest.raises(pgd.PGDError):
        a.share([ids[0], 3])                 # 3 is free
    assert a.refcount(ids[0]) == 1
    with pytest.raises(pgd.PGDError):
        pgd.BlockAllocator(0)


def test_append_slot_gap_and_range():
    a = pgd.BlockAllocator(4)
    row = [-1] * 2
    with pytest.raises(pgd.PGDError):
        a.append_slot(row, 5, 4)       # middle of an unopened block
    with pytest.raises(pgd.PGDError):
        a.append_slot(row, 8, 4)       # past the row
    a.append_slot(row, 0, 4)
    with pytest.raises(pgd.PGDError):
        a.append_slot([-1, -1], 4, 4)  # block 1 before block 0


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_model(seed):
    rng = random.Random(seed)
    NB, bs, MB = 40, 4, 12
    a = pgd.BlockAllocator(NB)
    m = BlockModel(NB)
    rows_a, rows_m, lens = [], [], []
    for step in range(400):
        op = rng.random()
        if op < 0.5 and rows_a:                      # append one token
            i = rng.randrange(len(rows_a))
            pos = lens[i]
            if pos >= MB * bs:
                continue
            try:
                src, dst = a.append_slot(rows_a[i], pos, bs)
            except pgd.PGDError as e:
                assert e.status == 3
                with pytest.raises(OutOfBlocks):
                    m.append_slot(list(rows_m[i]), pos, bs)
                continue
            chosen = rows_a[i][pos // bs] if (src >= 0 or rows_m[i][pos // bs] < 0) else None
            msrc, mdst = m.append_slot(rows_m[i], pos, bs, chosen=chosen)
            assert (src, dst) == (msrc, mdst)
            assert rows_a[i] == rows_m[i]
            lens[i] += 1
        elif op < 0.65 and rows_a:                   # fork
            i = rng.randrange(len(rows_a))
            n = rng.randint(0, lens[i])
            ra, rm = [-1] * MB, [-1] * MB
            a.fork(rows_a[i], n, bs, ra)
            m.fork(rows_m[i], n, bs, rm)
            assert ra == rm
            rows_a.append(ra); rows_m.append(rm); lens.append(n)
        elif op < 0.8 and rows_a:                    # finish a sequence
            i = rng.randrange(len(rows_a))
            held = [x for x in rows_a[i] if x >= 0]
            a.release(held)
            m.release(held)
            del rows_a[i], rows_m[i], lens[i]
        else:                                        # new sequence
            rows_a.append([-1] * MB); rows_m.append([-1] * MB); lens.append(0)
        assert a.num_free == m.num_free()
        assert all(a.refcount(k) == m.refcount(k) for k in range(NB))


def test_validate_tables():
    t = torch.tensor([[3, 1, -1], [0, -1, -1]], dtype=torch.int32)
    pgd.validate_tables(t, torch.tensor([20, 16], dtype=torch.int32), 4, 16)
    with pytest.raises(pgd.PGDError):
        pgd.validate_tables(t, torch.tensor([33, 16], dtype=torch.int32), 4, 16)  # needs 3 blocks
    with pytest.raises(pgd.PGDError):
        pgd.validate_tables(t, torch.tensor([20, 0], dtype=torch.int32), 4, 16)
    with pytest.raises(pgd.PGDError):
        pgd.validate_tables(t, torch.tensor([20, 16], dtype=torch.int32), 3, 16)  # id 3 >= NB
    with pytest.raises(pgd.PGDError):
        pgd.validate_tables(t, torch.tensor([20, 16 * 3 + 1], dtype=torch.int32), 4, 16)

"""The seeded generator's pool layouts against the element formulas that
include/pgd.h documents for the kernels (CPU only).  Both sides read these
layouts -- the kernels through bulk copies, the oracle through its own index
arithmetic -- so the generator that writes them is checked against the
header's formulas, element by element, with distinct values.

  * bf16 pool [NB][n_kv][bs/8][d/8][8][8]: element (slot s, dim i) of a
    (block, head) tile at ((s / 8) * (d / 8) + i / 8) * 64 + (s % 8) * 8 + i % 8;
  * 8-bit pool [NB][n_kv][bs/8][8 d + 32]: code of group slot r, dim i at
    (i / 16) * 128 + r * 16 + i % 16, then the 8 slots' fp32 scales;
  * MLA latent pool [NB][bs/8][72][8][8]: element (slot s, value i) of a block
    at ((s / 8) * 72 + i / 8) * 64 + (s % 8) * 8 + i % 8.
"""
import itertools

import torch

from paged_gqa_decode_kv_gb300 import inputs


def test_bf16_pool_layout():
    NB, n_kv, bs, d = 3, 2, 16, 128
    x = torch.arange(NB * n_kv * bs * d, dtype=torch.int64).reshape(NB, n_kv, bs, d)
    t = inputs.tile_pool(x)
    assert tuple(t.shape) == inputs.pool_shape(NB, n_kv, bs, d)
    flat = t.reshape(NB, n_kv, bs * d)
    for blk, h, s, i in itertools.product(range(NB), range(n_kv), range(bs), range(0, d, 7)):
        assert flat[blk, h, ((s // 8) * (d // 8) + i // 8) * 64 + (s % 8) * 8 + i % 8] == \
            x[blk, h, s, i]
    assert torch.equal(inputs.untile_pool(t), x)


def test_pool8_layout():
    NB, n_kv, bs, d = 2, 2, 16, 128
    codes = torch.arange(NB * n_kv * bs * d, dtype=torch.int64).remainder(251).to(torch.uint8)
    codes = codes.reshape(NB, n_kv, bs, d)
    scales = (torch.arange(NB * n_kv * bs, dtype=torch.float32) + 0.5).reshape(NB, n_kv, bs)
    pool = inputs.pack_pool8(codes, scales)
    assert tuple(pool.shape) == inputs.pool_shape8(NB, n_kv, bs, d)
    for blk, h, s in itertools.product(range(NB), range(n_kv), range(bs)):
        grp, r = pool[blk, h, s // 8], s % 8
        for i in range(0, d, 5):
            assert grp[(i // 16) * 128 + r * 16 + i % 16] == codes[blk, h, s, i]
        sc = grp[8 * d + 4 * r: 8 * d + 4 * r + 4].view(torch.float32)
        assert sc.item() == scales[blk, h, s].item()
    c2, s2 = inputs.unpack_pool8(pool)
    assert torch.equal(c2, codes) and torch.equal(s2, scales)


def test_latent_pool_layout():
    NB, bs, D = 2, 16, 576
    x = torch.arange(NB * bs * D, dtype=torch.int64).reshape(NB, bs, D)
    t = inputs.tile_latent(x)
    assert tuple(t.shape) == (NB, bs // 8, D // 8, 8, 8)
    flat = t.reshape(NB, bs * D)
    for blk, s, i in itertools.product(range(NB), range(bs), range(0, D, 11)):
        assert flat[blk, ((s // 8) * 72 + i // 8) * 64 + (s % 8) * 8 + i % 8] == x[blk, s, i]
    assert torch.equal(inputs.untile_latent(t), x)

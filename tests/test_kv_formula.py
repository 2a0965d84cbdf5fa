"""The KV byte closed form against every count the pages print
(tests/golden/kv_bytes.txt), and the paged pool the input generator builds
against the same closed form."""
import os

import pytest

from oracle import kv_formula
from paged_gqa_decode_kv_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes.txt")


def _rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            data, cite = line.split("|", 1)
            L, B, T, H, d, b, want, kind = data.split()
            rows.append((int(L), int(B), int(T), int(H), int(d), int(b), int(want), kind,
                         cite.strip()))
    return rows


@pytest.mark.parametrize("row", _rows(), ids=lambda r: r[8][:40])
def test_closed_form_matches_printed_value(row):
    L, B, T, H, d, b, want, kind, cite = row
    got = kv_formula.kv_bytes(L, B, T, H, d, b)
    if kind == "exact":
        assert got == want, cite
    else:
        # the page prints a rounded decimal: agree to its last printed digit
        digits = len(str(want).rstrip("0"))
        unit = 10 ** (len(str(want)) - digits)
        assert abs(got - want) <= unit // 2, (got, want, cite)


def test_golden_file_is_not_empty():
    assert len(_rows()) >= 10


@pytest.mark.parametrize("name", ["single_ctx512", "shared_prefix32"])
def test_generator_pool_matches_closed_form(name):
    pb = inputs.make_workload(name)
    nbytes = pb.k_cache.numel() * pb.k_cache.element_size() + \
        pb.v_cache.numel() * pb.v_cache.element_size()
    assert nbytes == kv_formula.paged_pool_bytes(pb.num_blocks, pb.block_size, pb.n_kv,
                                                 pb.head_dim, 2)


def test_workload_logical_bytes():
    # batch 16 x 8192 tokens x 8 KV heads x 128 x bf16 x (K, V) = 512 MiB
    w = inputs.WORKLOADS["batch16_ctx8192"]
    assert kv_formula.kv_bytes(1, w.batch, w.ctx, w.n_kv, w.head_dim, 2) == 512 * 2**20
    w = inputs.WORKLOADS["mha40_batch4_ctx8192"]
    assert kv_formula.kv_bytes(1, w.batch, w.ctx, w.n_kv, w.head_dim, 2) == 640 * 2**20

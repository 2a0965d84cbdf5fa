"""Pins of the 8-bit KV oracle (CPU): the E4M3 codec against torch's
float8_e4m3fn, the per-(token, head) quantiser against its defining
properties, kv_append_fp8's placement against an independent untiling, and
attention over the 8-bit cache against float64 SDPA on the dequantised
values.  Each planted mistake in the oracle must trip at least one pin."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_kv_gb300 import inputs

E4M3 = torch.float8_e4m3fn


def torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(E4M3) \
        .to(torch.float64).numpy()


def torch_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(E4M3) \
        .view(torch.uint8).numpy()


# ----------------------------------------------------------------- codec
def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_decode(codes), torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_landmarks():
    # OCP E4M3: largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9
    v = oracle.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x38, 0x00, 0x80, 0xFE], dtype=np.uint8))
    assert list(v[:5]) == [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, 0.0]
    assert math.copysign(1.0, v[5]) == -1.0 and v[6] == -448.0


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_matches_torch_including_ties():
    finite = np.sort(np.unique(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))
    mids = (finite[:-1] + finite[1:]) / 2          # exact ties: round to even
    rng = np.random.default_rng(5)
    rand = rng.uniform(-448, 448, 20000)
    small = rng.uniform(-2.0 ** -5, 2.0 ** -5, 5000)  # subnormal range
    x = np.concatenate([mids, -mids, rand, small]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x))


def test_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 460.0, 464.0, 1e4, 3e38, -500.0, np.inf, -np.inf, np.nan],
                 dtype=np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F]


def test_truncating_encoder_is_caught():
    x = np.linspace(-400, 400, 1001).astype(np.float32)
    assert not np.array_equal(oracle.e4m3_encode(x, truncate=True), torch_encode(x))


# ------------------------------------------------------------- quantiser
def _bf16_rows(n, d=128, std=1.0, seed=3):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, d, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("std", [1e-3, 1.0, 300.0])
def test_quantizer_against_its_definition(std):
    x = _bf16_rows(64, std=std)
    codes, scales = oracle.quantize_rows(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))
    # the largest element maps to +-448 exactly
    top = np.abs(xf).argmax(axis=1)
    assert np.all(np.isin(codes[np.arange(64), top], [0x7E, 0xFE]))
    # codes = torch's E4M3 cast of the binary32 quotient
    q = (xf / scales[:, None]).astype(np.float32)
    assert np.array_equal(codes, torch_encode(q))
    # dequantisation error within half a code step
    deq = oracle.e4m3_decode(codes) * scales[:, None].astype(np.float64)
    step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6))) - 3), 2.0 ** -9)
    assert np.all(np.abs(deq - xf) <= 0.5 * step * scales[:, None] * (1 + 1e-6))


def test_quantizer_zero_row():
    codes, scales = oracle.quantize_rows(torch.zeros(2, 128, dtype=torch.bfloat16))
    assert np.all(codes == 0) and np.all(scales == 1.0)


def test_quantizer_truncation_mutation_is_caught():
    x = _bf16_rows(16)
    good, _ = oracle.quantize_rows(x)
    bad, _ = oracle.quantize_rows(x, mutation=12)
    assert not np.array_equal(good, bad)


# ------------------------------------------------------------- kv_append
@pytest.mark.parametrize("bs", [16, 32])
def test_kv_append_fp8_places_quantised_rows(bs):
    lens = [1, bs, bs + 1, 3 * bs - 2, 77]
    pb = inputs.make_batch(len(lens), 16, 4, bs, lens, append=True, kv_format="fp8")
    k, v = oracle.kv_append_fp8(pb.k_cache, pb.v_cache, pb.k_new, pb.v_new, pb.block_tables,
                                pb.positions, bs)
    kc, ksc = oracle.quantize_rows(pb.k_new)
    vc, vsc = oracle.quantize_rows(pb.v_new)
    k_rows, ks = (t.numpy() for t in inputs.unpack_pool8(torch.from_numpy(k)))
    v_rows, vs = (t.numpy() for t in inputs.unpack_pool8(torch.from_numpy(v)))
    before_k = inputs.unpack_pool8(pb.k_cache)[0].numpy()
    touched = np.zeros(k_rows.shape[:3], dtype=bool)
    for b, pos in enumerate(pb.positions.tolist()):
        blk = int(pb.block_tables[b, pos // bs])
        slot = pos % bs
        touched[blk, :, slot] = True
        assert np.array_equal(k_rows[blk, :, slot], kc[b])
        assert np.array_equal(v_rows[blk, :, slot], vc[b])
        assert np.array_equal(ks[blk, :, slot], ksc[b]) and np.array_equal(vs[blk, :, slot], vsc[b])
    # nothing else changed
    assert np.array_equal(k_rows[~touched], before_k[~touched])


# ------------------------------------------------------------- attention
def _dequantised_rows(pool):
    codes, scales = inputs.unpack_pool8(torch.as_tensor(pool).cpu())
    return torch_decode(codes.numpy()) * scales.double().numpy()[..., None]


def sdpa_fp8(pb, k, v):
    """float64 SDPA over contiguous dequantised K/V gathered through the tables."""
    K = _dequantised_rows(k)
    V = _dequantised_rows(v)
    B, n_q, d = pb.q.shape
    G = n_q // pb.n_kv
    out = np.zeros((B, n_q, d))
    for b in range(B):
        n = int(pb.context_lens[b])
        ids = [int(pb.block_tables[b, t // pb.block_size]) for t in range(n)]
        slots = [t % pb.block_size for t in range(n)]
        kk = torch.from_numpy(np.stack([K[i, :, s] for i, s in zip(ids, slots)], 1))  # [n_kv][n][d]
        vv = torch.from_numpy(np.stack([V[i, :, s] for i, s in zip(ids, slots)], 1))
        qq = pb.q[b].double()[:, None, :]                                            # [n_q][1][d]
        kk = kk.repeat_interleave(G, 0)
        vv = vv.repeat_interleave(G, 0)
        out[b] = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv)[:, 0].numpy()
    return out


CASES = [(8, 2, 16, [1, 16, 17, 70]), (32, 8, 32, [33, 100]), (4, 4, 16, [5]), (16, 2, 16, [200])]


@pytest.mark.parametrize("case", CASES)
def test_attention_fp8_matches_sdpa_on_dequantised_values(case):
    n_q, n_kv, bs, lens = case
    pb = inputs.make_batch(len(lens), n_q, n_kv, bs, lens, kv_format="fp8")
    got = oracle.paged_attention_fp8(pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                     pb.context_lens, pb.scale, bs)
    want = sdpa_fp8(pb, pb.k_cache, pb.v_cache)
    assert np.abs(got - want).max() <= 1e-12


def test_attention_fp8_after_append():
    pb = inputs.make_batch(3, 16, 4, 16, [20, 1, 48], append=True, kv_format="fp8")
    k, v = oracle.kv_append_fp8(pb.k_cache, pb.v_cache, pb.k_new, pb.v_new, pb.block_tables,
                                pb.positions, 16)
    got = oracle.paged_attention_fp8(pb.q, k, v, pb.block_tables, pb.context_lens, pb.scale, 16)
    assert np.all(np.isfinite(got))
    assert np.abs(got - sdpa_fp8(pb, k, v)).max() <= 1e-12


@pytest.mark.parametrize("mutation", [9, 10, 11])
def test_fp8_attention_mutations_are_caught(mutation):
    pb = inputs.make_batch(2, 8, 2, 16, [40, 70], kv_format="fp8")
    want = sdpa_fp8(pb, pb.k_cache, pb.v_cache)
    bad = oracle.paged_attention_fp8(pb.q, pb.k_cache, pb.v_cache, pb.block_tables,
                                     pb.context_lens, pb.scale, 16, mutation=mutation)
    assert not np.all(np.abs(bad - want) <= 1e-6)  # NaN counts as caught

"""Pins of the oracle's FP8 (E4M3) KV path (no GPU).

The format is the OCP 8-bit float E4M3 (1 sign, 4 exponent bits with bias 7,
3 mantissa bits, no infinities, S.1111.111 = NaN). The row reading mirrors
the INT8 one (one fp32 scale per (token, KV head) row, amax mapped to 448,
fp32 IEEE steps, nearest code with ties to even, saturating at 448); it is
stated in the oracle's header. These tests pin the codes to the format's
published constants and to PyTorch's own float8_e4m3fn conversion (an
independent implementation), and the row path to the rounding bound, exact
power-of-two scaling, sign symmetry and equality with the bf16 attention
oracle on pools whose dequantised values are exact in bf16.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_decode_18_gb300 import workloads as W
from tests.pools import oracle_attention, oracle_attention_f8, oracle_pools_f8


def test_published_constants():
    v = oracle.e4m3_values(np.array([0x7E, 0x08, 0x01, 0x38, 0x00, 0x80, 0xFE, 0x07, 0x78],
                                    np.uint8))
    assert v[0] == 448.0          # largest finite
    assert v[1] == 2.0 ** -6      # smallest normal
    assert v[2] == 2.0 ** -9      # smallest subnormal
    assert v[3] == 1.0
    assert v[4] == 0.0 and not np.signbit(v[4])
    assert v[5] == 0.0 and np.signbit(v[5])
    assert v[6] == -448.0
    assert v[7] == 7.0 * 2.0 ** -9   # largest subnormal
    assert v[8] == 256.0
    assert np.all(np.isnan(oracle.e4m3_values(np.array([0x7F, 0xFF], np.uint8))))


def test_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_values(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_encoding_matches_torch_in_range():
    g = torch.Generator().manual_seed(11)
    parts = [torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)]
    # every midpoint between neighbouring codes, and the codes themselves
    vals = torch.from_numpy(np.arange(0, 0x7F, dtype=np.uint8)).view(torch.float8_e4m3fn).float()
    mids = (vals[1:] + vals[:-1]) / 2
    y = torch.cat(parts + [vals, mids, -vals, -mids, torch.tensor([448.0, 460.0, 464.0, -464.0])])
    y = y[y.abs() <= 464.0]  # beyond, torch's conversion gives NaN where the rule saturates
    ours = oracle.e4m3_codes(y.numpy())
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_saturation_and_round_trip():
    assert oracle.e4m3_codes(np.array([500.0, -1e6, 465.0], np.float32)).tolist() == [0x7E, 0xFE, 0x7E]
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    back = oracle.e4m3_codes(oracle.e4m3_values(finite).astype(np.float32))
    assert np.array_equal(back, finite)


def test_representable_row_is_exact():
    # amax 448 -> inv 1 and scale 1: every finite E4M3 value comes back as its own code
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_values(finite)
    row = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    codes, scales = oracle.quantize_rows_f8(row.unsqueeze(0))
    assert scales[0] == 1.0
    assert np.array_equal(oracle.e4m3_values(codes[0]), vals)


def _random_rows(seed, n=64, d=128):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g)
    x[:, 7] *= 20.0
    x *= torch.logspace(-3, 3, n).unsqueeze(1)
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("seed", [0, 1])
def test_row_round_trip_within_half_a_step(seed):
    x = _random_rows(seed)
    codes, scales = oracle.quantize_rows_f8(x)
    xf = x.float().numpy().astype(np.float64)
    s = scales.astype(np.float64)[:, None]
    deq = oracle.e4m3_values(codes) * s
    # nearest E4M3 value of x/scale: within 2^-4 relative (normal) or 2^-10
    # absolute (subnormal) of it, up to the fp32 rounding of inv and scale
    y = xf / s
    assert np.all(np.abs(xf - deq) <= (np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-5)) * s)
    amax_idx = np.abs(xf).argmax(axis=1)
    top = oracle.e4m3_values(codes[np.arange(len(xf)), amax_idx])
    assert np.all(top ** 2 == 448.0 ** 2)
    # and the largest element dequantises back to itself (the scale is the
    # row's amax over 448, rounded once to fp32)
    xtop = xf[np.arange(len(xf)), amax_idx]
    assert np.all(np.abs(top * s[:, 0] - xtop) <= 2.0 ** -23 * np.abs(xtop))


def test_zero_row_and_sign_symmetry():
    codes, scales = oracle.quantize_rows_f8(torch.zeros(2, 128, dtype=torch.bfloat16))
    assert not codes.any() and not scales.any()
    x = _random_rows(4)
    c0, s0 = oracle.quantize_rows_f8(x)
    c1, s1 = oracle.quantize_rows_f8(-x)
    assert np.array_equal(c1, c0 ^ 0x80) and np.array_equal(s1, s0)


@pytest.mark.parametrize("k", [-9, -1, 4])
def test_power_of_two_scaling_is_exact(k):
    x = _random_rows(3)
    c0, s0 = oracle.quantize_rows_f8(x)
    c1, s1 = oracle.quantize_rows_f8((x.float() * 2.0 ** k).to(torch.bfloat16))
    assert np.array_equal(c0, c1)
    assert np.array_equal(s1, (s0.astype(np.float64) * 2.0 ** k).astype(np.float32))


def test_fp8_attention_equals_bf16_on_representable_pools():
    # random E4M3 codes (no NaN) with power-of-two row scales: every
    # dequantised value has at most 4 significant bits, exact in bf16
    w = W.make("tiny", seed=5)
    g = np.random.default_rng(6)
    shape = w.pool_shape()
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    kc, vc = g.choice(finite, size=shape), g.choice(finite, size=shape)
    ks = (2.0 ** g.integers(-6, 3, size=shape[:3])).astype(np.float32)
    vs = (2.0 ** g.integers(-6, 3, size=shape[:3])).astype(np.float32)

    def to_bf16(c, s):
        x = torch.from_numpy((oracle.e4m3_values(c) * s[..., None]).astype(np.float32))
        b = x.to(torch.bfloat16)
        assert torch.equal(b.float(), x)
        return b.view(torch.int16).numpy().view(np.uint16)
    out8, lse8 = oracle_attention_f8(w, pools=(kc, vc, ks, vs))
    outb, lseb = oracle_attention(w, to_bf16(kc, ks), to_bf16(vc, vs))
    assert np.array_equal(out8, outb) and np.array_equal(lse8, lseb)


def test_fp8_cache_write_places_quantised_rows():
    w = W.make("tiny", seed=7)
    kc, vc, ks, vs = oracle_pools_f8(w)
    rows_k = torch.cat([w.k_hist, w.k_new])
    slots = torch.cat([w.slot_hist, w.slot_new]).numpy()
    codes, scales = oracle.quantize_rows_f8(rows_k)
    BS = w.block_size
    for t in range(0, len(slots), 37):
        b, o = divmod(int(slots[t]), BS)
        for h in range(w.num_kv_heads):
            assert np.array_equal(kc[b, h, o], codes[t, h]) and ks[b, h, o] == scales[t, h]
    written = np.zeros(w.pool_shape()[:3], bool)
    for t in range(len(slots)):
        b, o = divmod(int(slots[t]), BS)
        written[b, :, o] = True
    assert np.all(kc[~written] == W.POOL_SENTINEL_F8) and np.all(np.isnan(ks[~written]))


def test_fp8_attention_close_to_bf16_attention():
    w = W.make("tiny", seed=8)
    out8, lse8 = oracle_attention_f8(w)
    outb, lseb = oracle_attention(w)
    assert np.max(np.abs(out8 - outb)) < 0.1
    assert np.max(np.abs(lse8 - lseb)) < 0.1

"""Pins of the oracle's INT8 KV path (no GPU).

The pages name an INT8 KV cache and group-wise scales but fix no formula; the
reading used (symmetric, one fp32 scale per (token, KV head) row, fp32 IEEE
steps, ties to even) is stated in the oracle's header. These tests pin that
reading to facts that hold independently of the code: exact cases, the
rounding bound, exact power-of-two scaling and sign symmetry, and equality
with the bf16 attention oracle on pools whose dequantised values are exactly
representable in bf16.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_decode_18_gb300 import workloads as W
from tests.pools import oracle_attention, oracle_attention_i8, oracle_pools, oracle_pools_i8


def _q(rows):
    return oracle.quantize_rows_i8(torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16))


def test_integer_row_is_exact():
    # amax 127 -> inv 1: every integer code comes back unchanged, scale 1
    row = [float(i) for i in range(-127, 128)] + [0.0]
    codes, scales = _q([row])
    assert np.array_equal(codes[0].astype(np.int64), np.array(row, dtype=np.int64))
    assert scales[0] == 1.0


def test_ties_round_to_even():
    # inv = 1 (amax 127): x.5 values land on the even neighbour
    codes, _ = _q([[0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 127.0]])
    assert codes[0].tolist() == [0, 2, 2, 0, -2, -2, 4, 127]


def test_zero_row_has_zero_scale():
    codes, scales = _q([[0.0] * 128, [0.0] * 127 + [-3.0]])
    assert not codes[0].any() and scales[0] == 0.0
    assert codes[1, -1] == -127 and scales[1] == np.float32(3.0) / np.float32(127.0)


def _random_rows(seed, n=64, d=128, outliers=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g)
    if outliers:
        x[:, 7] *= 20.0  # a channel of outliers, as in real K caches
    x *= torch.logspace(-3, 3, n).unsqueeze(1)  # rows of very different magnitude
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("seed", [0, 1])
def test_round_trip_within_half_a_step(seed):
    x = _random_rows(seed)
    codes, scales = oracle.quantize_rows_i8(x)
    xf = x.float().numpy().astype(np.float64)
    deq = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
    step = scales.astype(np.float64)[:, None]
    assert np.all(np.abs(codes.astype(np.int64)) <= 127)
    # |x - code*scale| <= scale/2, up to the fp32 rounding of inv and scale
    assert np.all(np.abs(xf - deq) <= 0.5 * step * (1 + 1e-5) + 1e-30)
    # the largest magnitude of each row maps to +-127
    amax_idx = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(len(xf)), amax_idx]) == 127)


@pytest.mark.parametrize("k", [-9, -1, 4])
def test_power_of_two_scaling_is_exact(k):
    x = _random_rows(3)
    c0, s0 = oracle.quantize_rows_i8(x)
    c1, s1 = oracle.quantize_rows_i8((x.float() * 2.0 ** k).to(torch.bfloat16))
    assert np.array_equal(c0, c1)
    assert np.array_equal(s1, (s0.astype(np.float64) * 2.0 ** k).astype(np.float32))


def test_sign_symmetry():
    x = _random_rows(4)
    c0, s0 = oracle.quantize_rows_i8(x)
    c1, s1 = oracle.quantize_rows_i8(-x)
    assert np.array_equal(c1, -c0) and np.array_equal(s1, s0)


def _integer_pools(w, seed):
    """Random int8 codes with per-row power-of-two scales, and the bf16 pool
    holding exactly code * scale (|code| <= 127 fits bf16's 8-bit significand)."""
    g = np.random.default_rng(seed)
    shape = w.pool_shape()
    kc = g.integers(-127, 128, size=shape, dtype=np.int8)
    vc = g.integers(-127, 128, size=shape, dtype=np.int8)
    ks = (2.0 ** g.integers(-6, 3, size=shape[:3])).astype(np.float32)
    vs = (2.0 ** g.integers(-6, 3, size=shape[:3])).astype(np.float32)

    def to_bf16(c, s):
        x = torch.from_numpy(c.astype(np.float32) * s[..., None])
        b = x.to(torch.bfloat16)
        assert torch.equal(b.float(), x)  # exactly representable
        return b.view(torch.int16).numpy().view(np.uint16)
    return (kc, vc, ks, vs), to_bf16(kc, ks), to_bf16(vc, vs)


@pytest.mark.parametrize("name,sizes", [("tiny", {}), ("mixed", dict(num_verify=3, lo=40, hi=300,
                                                                       prefill_chunk=40,
                                                                       prefill_offsets=(0, 30)))])
def test_int8_attention_equals_bf16_on_representable_pools(name, sizes):
    w = W.make(name, seed=5, **sizes)
    i8, kb, vb = _integer_pools(w, 6)
    out8, lse8 = oracle_attention_i8(w, pools=i8)
    outb, lseb = oracle_attention(w, kb, vb)
    assert np.array_equal(out8, outb) and np.array_equal(lse8, lseb)


def test_int8_cache_write_places_quantised_rows():
    w = W.make("tiny", seed=7)
    kc, vc, ks, vs = oracle_pools_i8(w)
    # every written row is the row quantiser's output, at its slot
    rows_k = torch.cat([w.k_hist, w.k_new])
    slots = torch.cat([w.slot_hist, w.slot_new]).numpy()
    codes, scales = oracle.quantize_rows_i8(rows_k)
    Hkv, BS = w.num_kv_heads, w.block_size
    for t in range(0, len(slots), 37):
        b, o = divmod(int(slots[t]), BS)
        for h in range(Hkv):
            assert np.array_equal(kc[b, h, o], codes[t, h]) and ks[b, h, o] == scales[t, h]
    # untouched rows keep the sentinels
    written = np.zeros(w.pool_shape()[:3], bool)
    for t in range(len(slots)):
        b, o = divmod(int(slots[t]), BS)
        written[b, :, o] = True
    assert np.all(kc[~written] == W.POOL_SENTINEL_CODE) and np.all(np.isnan(ks[~written]))


def test_int8_attention_close_to_bf16_attention():
    # quantisation error of the whole path on generator data (a sanity bound,
    # not parity): outputs move by a small fraction of their scale
    w = W.make("tiny", seed=8)
    out8, lse8 = oracle_attention_i8(w)
    outb, lseb = oracle_attention(w)
    assert np.max(np.abs(out8 - outb)) < 0.05
    assert np.max(np.abs(lse8 - lseb)) < 0.05

"""CUDA FP8 (E4M3) KV path vs the oracle: the quantising cache write
bit-exact (codes and scale bits; untouched rows keep their NaN sentinels,
which the decode must never let into a result), and decode over the FP8
pool within |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3 of the fp64
oracle over the same dequantised rows, for every split mode, at small sizes
with ragged tails and at the full sizes of the workloads."""
import numpy as np
import pytest
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import Int8Batch, assert_attention_close, device, int8_pools_numpy
from tests.pools import oracle_attention_f8, oracle_pools_f8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


def _same_pools(got, ref):
    kc, vc, ks, vs = got
    rkc, rvc, rks, rvs = ref
    assert np.array_equal(kc.view(np.uint8), rkc) and np.array_equal(vc.view(np.uint8), rvc), \
        "fp8 codes differ"
    assert np.array_equal(ks.view(np.uint32), rks.view(np.uint32)), "k scales differ"
    assert np.array_equal(vs.view(np.uint32), rvs.view(np.uint32)), "v scales differ"


@pytest.mark.parametrize("name,sizes", [("tiny", {}), ("engine", {}),
                                        ("ragged", dict(num_seqs=40, max_context=700))])
def test_fp8_cache_write_bit_exact(name, sizes):
    w = W.make(name, seed=31, **sizes)
    db = Int8Batch(w, fp8=True)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    _same_pools(db.pools(), oracle_pools_f8(w))


def test_fp8_cache_write_ties_zero_rows_and_padding():
    from oracle import oracle
    w = W.make("tiny", seed=32)
    dev = device()
    kc, vc = w.empty_pool_f8(dev)
    k = w.k_new.clone()
    v = w.v_new.clone()
    k[0] = 0  # whole rows of zeros -> codes 0, scale 0
    v[1, 0] = 0
    k[2, 1, 5] = 3e4  # an outlier in one row
    # a row with amax 448 (inv = 1 exactly) whose other values sit on the
    # midpoints between E4M3 neighbours: each must go to the even code
    mids = torch.tensor([1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, 0.53125,
                         -5 * 2.0 ** -10, 13.0, 15.0, 232.0, 240.0, -416.0])
    row = torch.zeros(w.head_dim)
    row[0] = 448.0
    row[1:1 + len(mids)] = mids
    v[2, 0] = row.to(torch.bfloat16)
    slots = w.slot_new.clone()
    slots[3] = -1  # padding: skipped
    B.pa_reshape_and_cache_fp8(k.to(dev), v.to(dev), slots.to(dev), kc, vc)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    rk = np.full(w.pool_shape(), W.POOL_SENTINEL_F8, np.uint8)
    rv = rk.copy()
    rks = np.full(w.pool_shape()[:3], np.nan, np.float32)
    rvs = rks.copy()
    oracle.reshape_and_cache_f8(k, v, slots, rk, rv, rks, rvs)
    _same_pools(int8_pools_numpy(kc, vc), (rk, rv, rks, rvs))
    # the tie row's codes, against PyTorch's own E4M3 rounding
    b, o = divmod(int(slots[2]), w.block_size)
    ref = row.to(torch.bfloat16).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(rv[b, 0, o], ref)


CASES = {
    "tiny": ("tiny", {}),
    "engine": ("engine", {}),
    "ragged_small": ("ragged", dict(num_seqs=40, max_context=700)),
    "long_small": ("long", dict(num_seqs=2, context=3000)),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fp8_decode_matches_oracle(case, num_splits):
    name, sizes = CASES[case]
    w = W.make(name, seed=33, **sizes)
    db = Int8Batch(w, fp8=True)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_f8(w)  # the oracle quantises its own pool
    assert_attention_close(out, lse, ref, ref_lse, what=f"fp8 {case} P={num_splits}")


@pytest.mark.parametrize("name", ["ragged", "long"])
def test_fp8_decode_full_size(name):
    w = W.make(name, seed=34)
    db = Int8Batch(w, fp8=True)
    out, lse = db.decode(0)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_f8(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"fp8 full {name}")
    out_nl, _ = db.decode(0, with_lse=False)
    assert torch.equal(out, out_nl)


def test_fp8_decode_close_to_bf16_decode():
    from tests.gpu_util import DeviceBatch
    w = W.make("engine", seed=35)
    out8, lse8 = Int8Batch(w, fp8=True).decode(0)
    outb, lseb = DeviceBatch(w).decode(0)
    torch.cuda.synchronize()
    assert (out8.float() - outb.float()).abs().max().item() < 0.1
    assert (lse8 - lseb).abs().max().item() < 0.1

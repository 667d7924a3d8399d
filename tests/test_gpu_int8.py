"""CUDA INT8 KV path vs the oracle: the quantising cache write bit-exact
(codes and scale bits, untouched rows keep their sentinels), and decode over
the int8 pool within |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3 of
the fp64 oracle over the same dequantised rows, for every split mode, at small
sizes with ragged tails and at the full sizes of the workloads."""
import numpy as np
import pytest
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import Int8Batch, assert_attention_close, device, int8_pools_numpy
from tests.pools import oracle_attention_i8, oracle_pools_i8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


def _same_pools(got, ref):
    kc, vc, ks, vs = got
    rkc, rvc, rks, rvs = ref
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc), "int8 codes differ"
    # scales compared as bit patterns (NaN sentinels included)
    assert np.array_equal(ks.view(np.uint32), rks.view(np.uint32)), "k scales differ"
    assert np.array_equal(vs.view(np.uint32), rvs.view(np.uint32)), "v scales differ"


@pytest.mark.parametrize("name,sizes", [("tiny", {}), ("engine", {}),
                                        ("ragged", dict(num_seqs=40, max_context=700))])
def test_int8_cache_write_bit_exact(name, sizes):
    w = W.make(name, seed=21, **sizes)
    db = Int8Batch(w)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    _same_pools(db.pools(), oracle_pools_i8(w))


def test_int8_cache_write_zero_rows_and_padding():
    w = W.make("tiny", seed=22)
    dev = device()
    kc, vc = w.empty_pool_i8(dev)
    k = w.k_new.clone()
    v = w.v_new.clone()
    k[0] = 0  # whole rows of zeros -> codes 0, scale 0
    v[1, 0] = 0
    k[2, 1, 5] = 3e4  # an outlier in one row
    slots = w.slot_new.clone()
    slots[3] = -1  # padding: skipped
    B.pa_reshape_and_cache_int8(k.to(dev), v.to(dev), slots.to(dev), kc, vc)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    from oracle import oracle
    rk, rv = np.full(w.pool_shape(), W.POOL_SENTINEL_CODE, np.int8), None
    rv = rk.copy()
    rks = np.full(w.pool_shape()[:3], np.nan, np.float32)
    rvs = rks.copy()
    oracle.reshape_and_cache_i8(k, v, slots, rk, rv, rks, rvs)
    _same_pools(int8_pools_numpy(kc, vc), (rk, rv, rks, rvs))


CASES = {
    "tiny": ("tiny", {}),
    "engine": ("engine", {}),
    "ragged_small": ("ragged", dict(num_seqs=40, max_context=700)),
    "long_small": ("long", dict(num_seqs=2, context=3000)),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_int8_decode_matches_oracle(case, num_splits):
    name, sizes = CASES[case]
    w = W.make(name, seed=23, **sizes)
    db = Int8Batch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_i8(w)  # the oracle quantises its own pool
    assert_attention_close(out, lse, ref, ref_lse, what=f"int8 {case} P={num_splits}")


@pytest.mark.parametrize("name", ["ragged", "long"])
def test_int8_decode_full_size(name):
    # the full ragged (256 sequences up to 4096) and long (8 x 32k) batches:
    # every row of the ragged batch, sampled rows of the long one
    w = W.make(name, seed=24)
    db = Int8Batch(w)
    out, lse = db.decode(0)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_i8(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"int8 full {name}")
    out_nl, _ = db.decode(0, with_lse=False)
    assert torch.equal(out, out_nl)


def test_int8_decode_close_to_bf16_decode():
    # the same batch through both pool formats: the int8 answer stays near
    # the bf16 one (quantisation error, not parity)
    from tests.gpu_util import DeviceBatch
    w = W.make("engine", seed=25)
    out8, lse8 = Int8Batch(w).decode(0)
    outb, lseb = DeviceBatch(w).decode(0)
    torch.cuda.synchronize()
    assert (out8.float() - outb.float()).abs().max().item() < 0.05
    assert (lse8 - lseb).abs().max().item() < 0.05


@pytest.mark.parametrize("num_splits", [0, 3])
def test_int8_decode_queries_with_outlier_dims(num_splits):
    """Queries whose dims 7 and 77 are 64x the others (a power of two: exact
    in bf16). The K dot products over the codes hold fp32-level precision
    across the whole range of q, so lse stays within 1e-3 of the oracle even
    where the largest component sets the fixed-point step."""
    name, sizes = CASES["ragged_small"]
    w = W.make(name, seed=26, **sizes)
    q = w.q.clone()
    q[:, :, 7] *= 64
    q[:, :, 77] *= 64
    w.q = q
    db = Int8Batch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_i8(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"int8 outlier q P={num_splits}")

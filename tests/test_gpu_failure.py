"""Failure detection on the GPU without a GPU fault: bad device-resident
values are injected on the host (block ids past the pool, slots past the
pool, query windows longer than their context) and a copy is left out through
the library's test hook, so that a bounded wait runs out. Each case must set
its bit of the device error word, end without a trap or a hang, and leave the
context usable: a normal call right after matches the oracle."""
import time

import pytest
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, assert_attention_close
from tests.pools import oracle_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


def _still_usable(db):
    out, lse = db.decode(0)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(db.w)
    assert_attention_close(out, lse, ref, ref_lse, what="call after the injected failure")


def test_missing_copy_runs_into_the_bounded_wait():
    w = W.tiny(seed=40)
    db = DeviceBatch(w)
    B.pa_debug_read_error()
    B.pa_debug_inject_missing_copy(0)
    t0 = time.time()
    db.decode(0)
    torch.cuda.synchronize()
    dt = time.time() - t0
    err = B.pa_debug_read_error()
    assert err & B.PA_DEVERR_PIPE_TIMEOUT, err
    assert dt < 30, dt  # bounded: the wait gives up after its limit
    _still_usable(db)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_missing_copy_in_the_8bit_loop_runs_into_the_bounded_wait(fmt):
    from tests.gpu_util import Int8Batch
    from tests.pools import oracle_attention_f8, oracle_attention_i8
    w = W.tiny(seed=42)
    db = Int8Batch(w, fp8=fmt == "fp8")
    B.pa_debug_read_error()
    B.pa_debug_inject_missing_copy(0)
    t0 = time.time()
    db.decode(0)
    torch.cuda.synchronize()
    dt = time.time() - t0
    err = B.pa_debug_read_error()
    assert err & B.PA_DEVERR_PIPE_TIMEOUT, err
    assert dt < 30, dt
    out, lse = db.decode(0)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_f8(w) if fmt == "fp8" else oracle_attention_i8(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"{fmt} call after the injected failure")


def test_injection_is_consumed_by_one_launch():
    w = W.tiny(seed=41)
    db = DeviceBatch(w)
    B.pa_debug_inject_missing_copy(3)
    B.pa_debug_inject_missing_copy(-1)  # cleared before any launch
    _still_usable(db)


def _varlen_batch(seed, q_lens):
    ctx = [300, 900, 700, 64]
    return W.build("inject", seed, ctx, q_lens, pool_factor=1.2)


@pytest.mark.parametrize("q_lens", [[5, 5, 5, 5], [5, 64, 40, 5]])
def test_bad_block_id_in_varlen_is_flagged(q_lens):
    # verify-only, and verify + long chunks (tcgen05 path)
    w = _varlen_batch(42, q_lens)
    db = DeviceBatch(w)
    bt = db.block_tables.clone()
    bt[1, 2] = w.num_blocks + 7   # past the pool
    bt[2, 0] = -3                 # negative
    db.block_tables = bt
    db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() & B.PA_DEVERR_BLOCK_RANGE
    db.block_tables = w.block_tables.to(db.dev)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="varlen after bad ids")


def test_window_longer_than_context_is_flagged():
    w = _varlen_batch(43, [5, 5, 5, 5])
    db = DeviceBatch(w)
    cl = db.context_lens.clone()
    cl[0] = 3  # a causal window of 5 queries over 3 keys
    db.context_lens = cl
    db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() & B.PA_DEVERR_QLEN_RANGE


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_8bit_bad_slot_and_block_are_flagged(fmt):
    w = W.tiny(seed=44)
    dev = torch.device("cuda:0")
    fp8 = fmt == "fp8"
    kc, vc = w.empty_pool_f8(dev) if fp8 else w.empty_pool_i8(dev)
    slots = w.slot_new.clone()
    slots[1] = w.num_blocks * w.block_size + 5
    write = B.pa_reshape_and_cache_fp8 if fp8 else B.pa_reshape_and_cache_int8
    write(w.k_new.to(dev), w.v_new.to(dev), slots.to(dev), kc, vc)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() & B.PA_DEVERR_SLOT_RANGE
    q = w.q.to(dev)
    bt = w.block_tables.clone()
    bt[0, 0] = w.num_blocks + 1
    bt = bt.to(dev)
    out = torch.empty_like(q)
    sh = B.shape_of(q, kc, bt)
    if fp8:
        ws = B.workspace(B.pa_decode_fp8_workspace_size(sh, 0), dev)
        B.pa_decode_fp8(q, kc, vc, bt, w.context_lens.to(dev), w.scale, out, None, workspace=ws)
    else:
        ws = B.workspace(B.pa_decode_int8_workspace_size(sh, 0), dev)
        B.pa_decode_int8(q, kc, vc, bt, w.context_lens.to(dev), w.scale, out, None,
                         workspace=ws)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() & B.PA_DEVERR_BLOCK_RANGE
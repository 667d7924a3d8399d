"""CUDA paged decode (q_len 1) vs the fp64 oracle on the same seeded inputs:
|out - ref| <= 1e-2 + 1e-2 |ref| and |lse - ref| <= 1e-3, over every split
mode, at reduced sizes that span several tiles with ragged tails and at the
full sizes of the workloads (the benchmark's launch configuration is
num_splits = 0)."""
import numpy as np
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


CASES = {
    "tiny": ("tiny", {}),
    "engine": ("engine", {}),
    "ragged_small": ("ragged", dict(num_seqs=40, max_context=700)),
    "ragged_full": ("ragged", {}),
    "long_small": ("long", dict(num_seqs=2, context=3000)),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_matches_oracle(case, num_splits):
    name, sizes = CASES[case]
    w = W.make(name, seed=11, **sizes)
    db = DeviceBatch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"{case}/splits={num_splits}")


@pytest.mark.parametrize("num_splits", [0, 16, 32, 64])
def test_long_context_full_size(num_splits):
    # batch 8 x 32768 tokens, 1% outlier keys x8, split-K 16..64 or balanced
    w = W.long(seed=12)
    db = DeviceBatch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"long/splits={num_splits}")


def test_split_modes_agree():
    w = W.ragged(seed=13, num_seqs=64, max_context=2000)
    db = DeviceBatch(w)
    outs = [db.decode(p) for p in (0, 1, 2, 7)]
    base = outs[1][0].float()
    for o, l in outs:
        assert (o.float() - base).abs().max().item() <= 2e-2
        assert (l - outs[1][1]).abs().max().item() <= 1e-4


def test_deterministic_and_workspace_reuse():
    w = W.engine(seed=14)
    db = DeviceBatch(w)
    o1, l1 = db.decode(0)
    o2, l2 = db.decode(0)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_lse_optional():
    w = W.tiny(seed=15)
    db = DeviceBatch(w)
    o1, _ = db.decode(0, with_lse=False)
    o2, _ = db.decode(0, with_lse=True)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("num_splits", [0, 1, 4])
def test_empty_context_rows(num_splits):
    w = W.tiny(seed=16)
    db = DeviceBatch(w)
    db.context_lens[1] = 0
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    ref, ref_lse = oracle_attention(w)
    rows = [0, 2, 3]
    assert_attention_close(out, lse, ref, ref_lse, rows=rows, what="non-empty rows")


def test_bad_block_id_is_flagged_not_read():
    w = W.tiny(seed=17)
    db = DeviceBatch(w)
    B.pa_debug_read_error()
    db.block_tables[0, 0] = w.num_blocks + 5
    db.block_tables[2, 3] = -7
    out, lse = db.decode(0)
    err = B.pa_debug_read_error()
    assert err & B.PA_DEVERR_BLOCK_RANGE
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, rows=[1, 3], what="untouched rows")


def test_context_past_table_is_flagged():
    w = W.tiny(seed=18)
    db = DeviceBatch(w)
    B.pa_debug_read_error()
    db.context_lens[0] = w.max_blocks_per_seq * w.block_size + 1
    db.decode(0)
    assert B.pa_debug_read_error() & B.PA_DEVERR_CONTEXT_RANGE


def test_workspace_too_small_is_rejected():
    w = W.tiny(seed=19)
    db = DeviceBatch(w)
    sh = B.shape_of(db.q, db.kc, db.block_tables)
    need = B.pa_decode_workspace_size(sh, 0)
    small = torch.empty(need // 2, dtype=torch.uint8, device=db.dev)
    out = torch.empty_like(db.q)
    with pytest.raises(B.PAError) as e:
        B.pa_decode(db.q, db.kc, db.vc, db.block_tables, db.context_lens, w.scale, out,
                    num_splits=0, workspace=small)
    assert e.value.status == B.PA_ERR_WORKSPACE


APPEND_CASES = dict(CASES, ragged_600=("ragged", dict(num_seqs=600, max_context=300)))


@pytest.mark.parametrize("case", ["tiny", "engine", "ragged_small", "ragged_600"])
def test_append_decode_equals_two_calls(case):
    """pa_append_decode (write + decode in one call, the decode's preparation
    overlapping the write) gives the same pool bytes as pa_reshape_and_cache
    and the same results as pa_decode, from a handful of new rows to 600."""
    name, sizes = APPEND_CASES[case]
    w = W.make(name, seed=20, **sizes)
    ref = DeviceBatch(w)                  # history + new tokens written
    ref_out, ref_lse = ref.decode(0)
    fused = DeviceBatch(w, write_new=False)  # history only
    out = torch.empty_like(fused.q)
    lse = torch.empty(fused.q.shape[:2], dtype=torch.float32, device=fused.dev)
    sh = B.shape_of(fused.q, fused.kc, fused.block_tables)
    ws = B.workspace(B.pa_decode_workspace_size(sh, 0), fused.dev)
    for _ in range(2):
        B.pa_append_decode(fused.k_new, fused.v_new, fused.slot_new, fused.q, fused.kc, fused.vc,
                           fused.block_tables, fused.context_lens, w.scale, out, lse,
                           workspace=ws)
        torch.cuda.synchronize()
        assert B.pa_debug_read_error() == 0
        assert torch.equal(fused.kc.view(torch.int16), ref.kc.view(torch.int16))
        assert torch.equal(fused.vc.view(torch.int16), ref.vc.view(torch.int16))
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)
    ro, rl = oracle_attention(w)
    assert_attention_close(out, lse, ro, rl, what=f"append/{case}")


def test_append_decode_any_token_order_skips_and_bad_slots():
    """New rows in any token order, with a skipped token (slot < 0) and an
    out-of-range slot mixed in: the same pool bytes and results as the two
    calls, and the bad slot flagged as pa_reshape_and_cache flags it."""
    name, sizes = CASES["ragged_small"]
    w = W.make(name, seed=22, **sizes)
    ref = DeviceBatch(w)
    ref_out, ref_lse = ref.decode(0)
    fused = DeviceBatch(w, write_new=False)
    n = fused.k_new.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5)).to(fused.dev)
    g = torch.Generator().manual_seed(6)
    extra = torch.randn((2,) + tuple(fused.k_new.shape[1:]), generator=g).to(torch.bfloat16)
    extra = extra.to(fused.dev)
    bad = torch.tensor([-1, fused.kc.shape[0] * fused.kc.shape[2] + 5], dtype=torch.int64,
                       device=fused.dev)
    k_new = torch.cat([fused.k_new[perm], extra])
    v_new = torch.cat([fused.v_new[perm], -extra])
    slots = torch.cat([fused.slot_new[perm], bad])
    out = torch.empty_like(fused.q)
    lse = torch.empty(fused.q.shape[:2], dtype=torch.float32, device=fused.dev)
    sh = B.shape_of(fused.q, fused.kc, fused.block_tables)
    ws = B.workspace(B.pa_decode_workspace_size(sh, 0), fused.dev)
    B.pa_append_decode(k_new, v_new, slots, fused.q, fused.kc, fused.vc, fused.block_tables,
                       fused.context_lens, w.scale, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == B.PA_DEVERR_SLOT_RANGE
    assert torch.equal(fused.kc.view(torch.int16), ref.kc.view(torch.int16))
    assert torch.equal(fused.vc.view(torch.int16), ref.vc.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("variant", ["permuted", "skipped", "bad_slot"])
def test_append_decode_one_row_per_sequence_mappings(variant):
    """One new token per sequence, as a decode step has, under mappings other
    than token t -> its own sequence's last position: tokens permuted, a
    skipped token (slot < 0), an out-of-range slot. Pool bytes, results and
    error bits equal those of pa_reshape_and_cache followed by pa_decode."""
    name, sizes = CASES["ragged_small"]
    w = W.make(name, seed=23, **sizes)
    dev_batch = DeviceBatch(w, write_new=False)
    k_new, v_new, slots = dev_batch.k_new, dev_batch.v_new, dev_batch.slot_new.clone()
    if variant == "permuted":
        perm = torch.randperm(k_new.shape[0], generator=torch.Generator().manual_seed(7))
        perm = perm.to(dev_batch.dev)
        k_new, v_new, slots = k_new[perm], v_new[perm], slots[perm]
    elif variant == "skipped":
        slots[3] = -1
    else:
        slots[5] = dev_batch.kc.shape[0] * dev_batch.kc.shape[2] + 7
    expect_err = B.PA_DEVERR_SLOT_RANGE if variant == "bad_slot" else 0

    ref = DeviceBatch(w, write_new=False)
    B.pa_reshape_and_cache(k_new, v_new, slots, ref.kc, ref.vc)
    ref_out, ref_lse = ref.decode(0)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == expect_err

    fused = dev_batch
    out = torch.empty_like(fused.q)
    lse = torch.empty(fused.q.shape[:2], dtype=torch.float32, device=fused.dev)
    sh = B.shape_of(fused.q, fused.kc, fused.block_tables)
    ws = B.workspace(B.pa_decode_workspace_size(sh, 0), fused.dev)
    B.pa_append_decode(k_new, v_new, slots, fused.q, fused.kc, fused.vc, fused.block_tables,
                       fused.context_lens, w.scale, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == expect_err
    assert torch.equal(fused.kc.view(torch.int16), ref.kc.view(torch.int16))
    assert torch.equal(fused.vc.view(torch.int16), ref.vc.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    # bit patterns: a skipped token leaves the pool's sentinel (NaN) row in
    # place, read the same way by both paths
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))

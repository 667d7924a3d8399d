"""Closed forms of attention run through the CUDA kernels.

* A query that sees exactly one key gives that key's softmax weight exactly
  1, so its output is that key's V row with no rounding at all: a length-1
  context (one valid token in an otherwise unwritten, NaN-filled block) must
  return V bit for bit through pa_decode in every split mode, through
  pa_decode_varlen (the first query of a causal window that starts at
  position 0 sees key 0 only, on both tensor-core tiles), and through
  pa_decode_int8 at the dequantised row's precision (fp32 code * scale,
  rounded once to bf16).
* A context whose keys are all equal gives every key the same weight, so the
  output is the mean of V and lse = scale * q.k + ln c.

Both facts come from the definition of softmax attention; the GPU results are
also compared with the fp64 oracle at the usual tolerance.
"""
import math

import numpy as np
import pytest
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, Int8Batch, assert_attention_close
from tests.pools import logical_kv, oracle_attention, oracle_attention_i8, oracle_pools_i8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16)


def _length_one_batch(seed, num_seqs=48):
    """Length-1 contexts interleaved with longer ones (so the balanced cut
    runs through real work around them)."""
    g = torch.Generator().manual_seed(seed)
    longer = torch.randint(2, 3000, (num_seqs,), generator=g).tolist()
    ctx = [1 if s % 3 != 1 else longer[s] for s in range(num_seqs)]
    return W.build("len1", seed, ctx, [1] * num_seqs, pool_factor=1.2)


def _first_key_v_rows(w, rows_of):
    """V row of each sequence's key 0, per query head: [len(rows), Hq, D] bf16."""
    G = w.num_q_heads // w.num_kv_heads
    out = []
    for s in rows_of:
        _, v = logical_kv(w, s)
        out.append(v[0].repeat_interleave(G, 0))
    return torch.stack(out)


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_length_one_context_returns_v_bit_exactly(num_splits):
    w = _length_one_batch(31)
    db = DeviceBatch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"len1/splits={num_splits}")
    ones = [s for s in range(w.num_seqs) if int(w.context_lens[s]) == 1]
    got = out.cpu()[ones]
    want = _first_key_v_rows(w, ones)
    assert torch.equal(_bits(got), _bits(want)), "a length-1 context did not return V exactly"
    # the oracle agrees exactly too (its weight is 1.0 in fp64)
    assert np.array_equal(got.double().numpy(), ref[ones])


def test_length_one_context_through_append_decode():
    # the engine's one-call step: the token is written, then attended alone
    w = _length_one_batch(32, num_seqs=64)
    db = DeviceBatch(w, write_new=False)
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.dev)
    sh = B.shape_of(db.q, db.kc, db.block_tables)
    ws = B.workspace(B.pa_decode_workspace_size(sh, 0), db.dev)
    B.pa_append_decode(db.k_new, db.v_new, db.slot_new, db.q, db.kc, db.vc, db.block_tables,
                       db.context_lens, w.scale, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ones = [s for s in range(w.num_seqs) if int(w.context_lens[s]) == 1]
    assert torch.equal(_bits(out.cpu()[ones]), _bits(_first_key_v_rows(w, ones)))


def test_first_causal_query_returns_v0_on_both_tensor_core_tiles():
    # sequences whose query window starts at position 0 (c == q_len): query 0
    # sees key 0 only. Windows of 1, 5 and 8 queries go through the 16-row
    # mma.sync tile, windows of 64 and 130 through the 128-row tcgen05 tile.
    ctx = [1, 5, 64, 300, 8, 130, 1, 700]
    ql = [1, 5, 64, 5, 8, 130, 1, 40]
    w = W.build("v0", 33, ctx, ql, pool_factor=1.2)
    db = DeviceBatch(w)
    out, lse = db.varlen(causal=True)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="varlen first query")
    seqs = [s for s in range(w.num_seqs) if int(w.context_lens[s]) == int(w.q_lens[s])]
    rows = [int(w.cu_seqlens_q[s]) for s in seqs]
    got = out.cpu()[rows]
    assert torch.equal(_bits(got), _bits(_first_key_v_rows(w, seqs)))
    assert np.array_equal(got.double().numpy(), ref[rows])


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_int8_length_one_context_returns_dequantised_v(num_splits):
    w = _length_one_batch(34)
    db = Int8Batch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    pools = oracle_pools_i8(w)
    ref, ref_lse = oracle_attention_i8(w, pools)
    assert_attention_close(out, lse, ref, ref_lse, what=f"int8 len1/splits={num_splits}")
    ones = [s for s in range(w.num_seqs) if int(w.context_lens[s]) == 1]
    # the oracle's output there is the dequantised row code * scale, exact in
    # fp64; the kernel forms it as one fp32 product and rounds it to bf16
    want = torch.from_numpy(ref[ones]).float().to(torch.bfloat16)
    assert torch.equal(_bits(out.cpu()[ones]), _bits(want))
    # and that row is the pool's own codes times its scale
    _, vc, _, vs = pools
    G = w.num_q_heads // w.num_kv_heads
    for s in ones:
        phys = int(w.block_tables[s, 0])
        row = torch.from_numpy(vc[phys, :, 0, :].astype(np.float32)) * \
            torch.from_numpy(vs[phys, :, 0]).unsqueeze(1)
        assert torch.equal(_bits(row.to(torch.bfloat16).repeat_interleave(G, 0)),
                           _bits(out.cpu()[s]))


def _equal_keys(w):
    """Make every key row of each (sequence, KV head) equal to that sequence's
    new token's key, in place (history and new rows alike)."""
    for s in range(w.num_seqs):
        q0, q1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
        h0, h1 = int(w.cu_hist[s]), int(w.cu_hist[s + 1])
        key = w.k_new[q0].clone()
        w.k_new[q0:q1] = key
        w.k_hist[h0:h1] = key
    return w


@pytest.mark.parametrize("num_splits", [0, 1, 16])
def test_equal_keys_give_mean_of_v(num_splits):
    g = torch.Generator().manual_seed(35)
    ctx = torch.randint(1, 4000, (40,), generator=g).tolist() + [1, 16, 17, 8192]
    w = _equal_keys(W.build("eqk", 35, ctx, [1] * len(ctx), pool_factor=1.2))
    db = DeviceBatch(w)
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"equal keys/splits={num_splits}")
    # the closed form, from the logical K/V with no pool and no oracle
    G = w.num_q_heads // w.num_kv_heads
    mean = np.zeros(ref.shape)
    lse_cf = np.zeros(ref_lse.shape)
    for s in range(w.num_seqs):
        k, v = logical_kv(w, s)
        c = k.shape[0]
        r = int(w.cu_seqlens_q[s])
        vm = v.double().mean(0).repeat_interleave(G, 0).numpy()
        mean[r] = vm
        z = (w.q[r].double() * k[0].double().repeat_interleave(G, 0)).sum(-1) * w.scale
        lse_cf[r] = (z + math.log(c)).numpy()
    np.testing.assert_allclose(ref, mean, rtol=0, atol=1e-12)  # the oracle meets it
    assert_attention_close(out, lse, mean, lse_cf, what="equal keys vs closed form")

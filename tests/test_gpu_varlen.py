"""CUDA verify / chunked-prefill attention (several query tokens per
sequence, tensor cores) vs the fp64 oracle."""
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


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed", [21, 22])
def test_mixed_small(seed, causal):
    w = W.mixed(seed=seed, num_verify=6, lo=40, hi=700, prefill_chunk=70,
                prefill_offsets=(0, 100))
    w.causal = causal
    db = DeviceBatch(w)
    out, lse = db.varlen(causal=causal)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"mixed small causal={causal}")


def test_mixed_full_size():
    # 48 verify sequences (q_len 5, contexts 256..8192) + prefill chunks of
    # 512 at offsets 0 and 1536
    w = W.mixed(seed=23)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="mixed full")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (16, 2), (32, 2)])
def test_other_group_sizes(hq, hkv):
    w = W.build("groups", 24, [33, 90, 17, 260], [3, 9, 1, 20], pool_factor=1.3,
                num_q_heads=hq, num_kv_heads=hkv)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"G={hq // hkv}")


def test_q_len_one_matches_decode():
    w = W.ragged(seed=25, num_seqs=30, max_context=500)
    db = DeviceBatch(w)
    o1, l1 = db.varlen()
    o2, l2 = db.decode(0)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_zero_q_len_sequences_produce_no_rows():
    w = W.build("zq", 26, [40, 64, 1, 100], [0, 7, 0, 12], pool_factor=1.2)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="zero q_len")


# Sequences with q_len >= 32 run on the tcgen05 prefill tile (128 query rows
# per KV head); shorter ones on the mma.sync tile. These cases cover the long
# path with every group size, ragged context tails, and both paths at once.

@pytest.mark.parametrize("hq,hkv", [(16, 8), (8, 8), (16, 4), (32, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_tiles_group_sizes(hq, hkv, causal):
    # q_len 32..300 at offsets that leave ragged 16- and 128-key tails
    w = W.build("tc", 31, [45, 300, 777, 130, 1029], [32, 300, 129, 65, 40], pool_factor=1.2,
                num_q_heads=hq, num_kv_heads=hkv, causal=causal)
    db = DeviceBatch(w)
    out, lse = db.varlen(causal=causal)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"tc G={hq // hkv} causal={causal}")


def test_prefill_and_verify_in_one_call():
    w = W.build("both", 32, [300, 17, 2000, 64, 600, 5], [200, 5, 512, 33, 31, 5],
                pool_factor=1.15)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="tc + mma paths")


def test_prefill_segment_cut_into_many_pieces():
    # one query tile per KV head over 8192 keys: 8 segments of 64 key tiles
    # spread over every CTA, so each segment is merged from ~20 pieces
    w = W.build("cut", 33, [8192, 40], [64, 40], pool_factor=1.1)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    out_nl, _ = db.varlen(with_lse=False)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="many pieces")
    assert torch.equal(out, out_nl)


def _varlen_max_q(db, max_q_len):
    # pa_decode_varlen with a max_q_len above the batch's longest window (an
    # upper bound is allowed)
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.dev)
    sh = B.shape_of(db.q, db.kc, db.block_tables)
    ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, db.q.shape[0], max_q_len), db.dev)
    B.pa_decode_varlen(db.q, db.kc, db.vc, db.block_tables, db.context_lens, db.cu_seqlens_q,
                       max_q_len, db.w.scale, out, lse, causal=True, workspace=ws)
    return out, lse


def test_side_by_side_split_one_prefill_cta():
    # 59 verify windows over long contexts beside one 32-token chunk: the
    # prefill grid keeps a single CTA, the verify grid the other SMs
    ctx = [2000 + 37 * i for i in range(59)] + [32]
    ql = [5] * 59 + [32]
    w = W.build("split1", 41, ctx, ql, pool_factor=1.1)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="split K=1")


def test_side_by_side_split_one_verify_cta():
    # one 1024-token chunk and one short verify window beside 98 sequences
    # with no queries (the batch still averages under 32 query tokens): the
    # prefill grid keeps all but one CTA, the verify grid works on one
    ctx = [4096, 16] + [16] * 98
    ql = [1024, 5] + [0] * 98
    w = W.build("splitN", 42, ctx, ql, pool_factor=1.1)
    db = DeviceBatch(w)
    out, lse = db.varlen()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="split K=N-1")


def test_side_by_side_split_no_prefill_work():
    # only verify windows, with max_q_len declared above the tensor-core
    # threshold: both grids launch, the prefill grid finds no work and leaves
    # every SM to the verify grid
    w = W.build("split0", 43, [300, 900, 40, 1500], [5, 7, 3, 9], pool_factor=1.2)
    db = DeviceBatch(w)
    out, lse = _varlen_max_q(db, 64)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="split K=0")
    out2, lse2 = db.varlen()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)

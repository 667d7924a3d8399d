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

"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test checks the oracle against a fact the pages or the mathematics fix:
closed forms, a library routine (torch's scaled_dot_product_attention and
logsumexp in float64), and the invariants the course README claims for its
own NumPy code ("paged attention == contiguous attention", "online softmax is
exact; paged and split-K variants agree", "chunked prefill produces a
bit-identical KV cache"). The cases are chosen so that a dropped scale, a
wrong GQA mapping, an off-by-one in the causal window, a transposed block
index or a wrong merge weight fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle
from paged_kv_decode_18_gb300 import workloads as W
from tests.pools import bf16_bits, logical_kv, oracle_attention, oracle_pools


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_two_keys_closed_form():
    # q=(1,0), k0=(0,0), k1=(2,0), scale 1/2: logits 0 and 1, so the weights
    # are 1/(1+e) and e/(1+e); V = identity rows gives out = the weights.
    q = _bf16([1.0, 0.0])
    K = _bf16([[0.0, 0.0], [2.0, 0.0]])
    V = _bf16([[1.0, 0.0], [0.0, 1.0]])
    out, lse = oracle.attention_dense(q, K, V, 0.5)
    e = math.e
    assert out == pytest.approx([1 / (1 + e), e / (1 + e)], abs=1e-15)
    assert lse == pytest.approx(math.log(1 + e), abs=1e-15)


def test_length_one_context_returns_v():
    g = torch.Generator().manual_seed(1)
    q = torch.randn(128, generator=g).to(torch.bfloat16)
    K = torch.randn(1, 128, generator=g).to(torch.bfloat16)
    V = torch.randn(1, 128, generator=g).to(torch.bfloat16)
    out, lse = oracle.attention_dense(q, K, V, 0.125)
    assert np.array_equal(out, V[0].double().numpy())  # weight is exactly 1
    assert lse == pytest.approx(0.125 * float(q.double() @ K[0].double()), abs=1e-12)


def test_equal_keys_give_mean_of_v():
    g = torch.Generator().manual_seed(2)
    n = 37
    q = torch.randn(64, generator=g).to(torch.bfloat16)
    k = torch.randn(64, generator=g).to(torch.bfloat16)
    K = k.repeat(n, 1)
    V = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    out, lse = oracle.attention_dense(q, K, V, 0.3)
    np.testing.assert_allclose(out, V.double().mean(0).numpy(), rtol=0, atol=1e-14)
    z = 0.3 * float(q.double() @ k.double())
    assert lse == pytest.approx(z + math.log(n), abs=1e-12)


def test_zero_scale_gives_mean_and_log_n():
    g = torch.Generator().manual_seed(3)
    n = 50
    q = torch.randn(32, generator=g).to(torch.bfloat16)
    K = torch.randn(n, 32, generator=g).to(torch.bfloat16)
    V = torch.randn(n, 32, generator=g).to(torch.bfloat16)
    out, lse = oracle.attention_dense(q, K, V, 0.0)
    np.testing.assert_allclose(out, V.double().mean(0).numpy(), rtol=0, atol=1e-14)
    assert lse == pytest.approx(math.log(n), abs=1e-14)


def test_extreme_logit_spread_stays_exact():
    # logits 0 and 1024 (both exact in bf16): the softmax must subtract the
    # true maximum, or exp() overflows. Weight of the first key is e^-1024 = 0
    # in fp64, so out = V[1] and lse = 1024 exactly.
    q = _bf16([1.0, 0.0])
    K = _bf16([[0.0, 0.0], [1024.0, 0.0]])
    V = _bf16([[3.0, -1.0], [0.5, 2.0]])
    for tile in (0, 1):
        out, lse = oracle.attention_dense(q, K, V, 1.0, online_tile=tile)
        assert out.tolist() == [0.5, 2.0]
        assert lse == 1024.0


def test_empty_context_convention():
    q = _bf16([1.0, 2.0])
    K = torch.zeros(0, 2, dtype=torch.bfloat16)
    out, lse = oracle.attention_dense(q, K, K, 1.0)
    assert np.all(out == 0.0) and lse == -math.inf


# --------------------------------------------------------------------------
# brute force against torch (float64, CPU) on tiny paged inputs
# --------------------------------------------------------------------------

def _sdpa_reference(w):
    """Per sequence: expand KV heads to query heads (head h reads h // G),
    build the causal window explicitly, and call torch's SDPA in float64."""
    G = w.num_q_heads // w.num_kv_heads
    outs, lses = [], []
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        q0, q1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
        lq = q1 - q0
        if lq == 0:
            continue
        k, v = logical_kv(w, s)                              # [c, Hkv, D]
        K = k.double().permute(1, 0, 2).repeat_interleave(G, 0)[None]  # [1,Hq,c,D]
        V = v.double().permute(1, 0, 2).repeat_interleave(G, 0)[None]
        Q = w.q[q0:q1].double().permute(1, 0, 2)[None]       # [1,Hq,lq,D]
        pos = torch.arange(c - lq, c)[:, None]
        keys = torch.arange(c)[None, :]
        allowed = keys <= pos if w.causal else torch.ones(lq, c, dtype=torch.bool)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=allowed, scale=w.scale)
        logits = (Q @ K.transpose(-1, -2)) * w.scale
        logits = logits.masked_fill(~allowed, -math.inf)
        outs.append(o[0].permute(1, 0, 2))                   # [lq, Hq, D]
        lses.append(torch.logsumexp(logits, -1)[0].permute(1, 0))  # [lq, Hq]
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_torch_sdpa_small_heads(seed, causal):
    # Hq=6 over Hkv=2 (group 3), D=8, block_size 4, a few ragged sequences with
    # 1, 3 and 5 query tokens, tables shuffled over a pool with spare blocks.
    w = W.build("bf", seed, [9, 23, 40, 5], [1, 3, 5, 2], pool_factor=1.5, causal=causal,
                num_q_heads=6, num_kv_heads=2, head_dim=8, block_size=4, scale=0.37)
    out, lse = oracle_attention(w)
    ref_out, ref_lse = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_matches_torch_sdpa_model_shape():
    # the built shape: 16 query heads over 8 KV heads, head_dim 128, block 16
    w = W.build("bf", 5, [1, 17, 64, 130], [1, 1, 5, 12], pool_factor=1.3)
    out, lse = oracle_attention(w)
    ref_out, ref_lse = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# invariants claimed on the pages
# --------------------------------------------------------------------------

def test_paged_equals_contiguous():
    # course README: "paged attention == contiguous attention"
    w = W.tiny(seed=4)
    out, lse = oracle_attention(w)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        k, v = logical_kv(w, s)
        row = int(w.cu_seqlens_q[s])
        for h in range(w.num_q_heads):
            o_ref, l_ref = oracle.attention_dense(w.q[row, h], k[:, h // G], v[:, h // G],
                                                  w.scale)
            np.testing.assert_allclose(out[row, h], o_ref, rtol=0, atol=1e-14)
            assert abs(lse[row, h] - l_ref) <= 1e-14


@pytest.mark.parametrize("tile", [1, 7, 16, 1000])
def test_online_equals_two_pass(tile):
    # course README: "online softmax is exact"
    w = W.build("online", 6, [1, 31, 200, 77], [1, 1, 3, 6], pool_factor=1.2,
                outlier_frac=0.05)
    kp, vp = oracle_pools(w)
    o2, l2 = oracle_attention(w, kp, vp)
    o1, l1 = oracle_attention(w, kp, vp, online_tile=tile)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("P", [2, 7, 64])
def test_split_equals_unsplit(P):
    # course README: "paged and split-K variants agree"
    g = torch.Generator().manual_seed(7)
    n, D = 300, 128
    q = torch.randn(D, generator=g).to(torch.bfloat16)
    K = (torch.randn(n, D, generator=g) * 1.5).to(torch.bfloat16)
    V = torch.randn(n, D, generator=g).to(torch.bfloat16)
    full_o, full_l = oracle.attention_dense(q, K, V, 1 / math.sqrt(D))
    bounds = [(i * n) // P for i in range(P + 1)]
    po = np.zeros((1, P, D))
    pl = np.zeros((1, P))
    for i in range(P):
        po[0, i], pl[0, i] = oracle.attention_dense(q, K[bounds[i]:bounds[i + 1]],
                                                    V[bounds[i]:bounds[i + 1]],
                                                    1 / math.sqrt(D))
    mo, ml = oracle.splitk_merge(po, pl)
    np.testing.assert_allclose(mo[0], full_o, rtol=0, atol=1e-13)
    assert abs(ml[0] - full_l) <= 1e-13


def test_merge_ignores_empty_partials_and_empty_rows():
    g = np.random.default_rng(8)
    po = g.standard_normal((3, 4, 16))
    pl = g.standard_normal((3, 4))
    mo, ml = oracle.splitk_merge(po, pl)
    po2 = np.concatenate([po, g.standard_normal((3, 2, 16))], axis=1)
    pl2 = np.concatenate([pl, np.full((3, 2), -np.inf)], axis=1)
    mo2, ml2 = oracle.splitk_merge(po2, pl2)
    np.testing.assert_array_equal(mo, mo2)
    np.testing.assert_array_equal(ml, ml2)
    eo, el = oracle.splitk_merge(po, np.full((3, 4), -np.inf))
    assert np.all(eo == 0) and np.all(el == -np.inf)


def test_merge_weights_by_lse():
    # two partials with lse ln1 and ln3 carry weights 1/4 and 3/4, LSE ln4
    po = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    pl = np.array([[math.log(1.0), math.log(3.0)]])
    mo, ml = oracle.splitk_merge(po, pl)
    np.testing.assert_allclose(mo[0], [0.25, 0.75], rtol=0, atol=1e-15)
    assert ml[0] == pytest.approx(math.log(4.0), abs=1e-15)


# --------------------------------------------------------------------------
# cache write
# --------------------------------------------------------------------------

def test_cache_write_places_rows_by_table():
    w = W.tiny(seed=9)
    kp, vp = oracle_pools(w)
    # read every token back through the block table with numpy indexing
    for s in range(w.num_seqs):
        k, v = logical_kv(w, s)
        c = int(w.context_lens[s])
        p = np.arange(c)
        blocks = w.block_tables[s].numpy()[p // w.block_size]
        np.testing.assert_array_equal(kp[blocks, :, p % w.block_size, :], bf16_bits(k))
        np.testing.assert_array_equal(vp[blocks, :, p % w.block_size, :], bf16_bits(v))
    # every slot outside the contexts still holds the sentinel
    used = np.zeros((w.num_blocks, w.block_size), bool)
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        p = np.arange(c)
        used[w.block_tables[s].numpy()[p // w.block_size], p % w.block_size] = True
    assert np.all(kp.transpose(0, 2, 1, 3)[~used] == W.POOL_SENTINEL_BITS)


def test_chunked_write_is_bit_identical():
    # course README: "chunked prefill produces a bit-identical KV cache"
    w = W.mixed(seed=10, num_verify=3, lo=40, hi=90, prefill_chunk=48,
                prefill_offsets=(0, 32))
    one_k, one_v = oracle_pools(w)
    kp = np.full(w.pool_shape(), W.POOL_SENTINEL_BITS, np.uint16)
    vp = kp.copy()
    T = w.k_hist.shape[0]
    for a in range(0, T, 37):
        b = min(T, a + 37)
        oracle.reshape_and_cache(w.k_hist[a:b], w.v_hist[a:b], w.slot_hist[a:b], kp, vp,
                                 w.block_size)
    for a in range(0, w.num_q_tokens, 11):
        b = min(w.num_q_tokens, a + 11)
        oracle.reshape_and_cache(w.k_new[a:b], w.v_new[a:b], w.slot_new[a:b], kp, vp,
                                 w.block_size)
    assert np.array_equal(kp, one_k) and np.array_equal(vp, one_v)


def test_cache_write_rejects_slot_past_pool():
    kp = np.zeros((2, 1, 4, 8), np.uint16)
    vp = kp.copy()
    k = torch.zeros(1, 1, 8, dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(k, k, torch.tensor([8]), kp, vp, 4)


def test_paged_attention_rejects_bad_block_id():
    w = W.tiny(seed=11, num_seqs=2, lo=20, hi=30, num_blocks=8)
    kp, vp = oracle_pools(w)
    bt = w.block_tables.clone()
    bt[0, 0] = w.num_blocks
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(w.q, kp, vp, bt, w.context_lens, w.cu_seqlens_q, w.scale)


# --------------------------------------------------------------------------
# non-causal windows longer than their context
# --------------------------------------------------------------------------

def _queries_over_pool(w, q_lens, seed):
    """A fresh set of query rows (q_lens[s] per sequence) over w's pool:
    (q [Tq, Hq, D] bf16, cu_seqlens_q [S + 1] int32)."""
    g = torch.Generator().manual_seed(seed)
    tq = int(sum(q_lens))
    q = torch.randn(tq, w.num_q_heads, w.head_dim, generator=g).to(torch.bfloat16)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    return q, cu


def test_non_causal_window_longer_than_context_matches_sdpa():
    # S20 "The conflicts" / prefix caching: several sequences' queries attend
    # one shared context at once, so a non-causal window may hold more query
    # rows than the context has keys. Every row then sees the whole context:
    # torch SDPA in float64 with no mask, GQA expanded, is the reference.
    w = W.build("nc", 21, [3, 9, 20, 16], [1, 1, 1, 1], pool_factor=1.5, causal=False,
                num_q_heads=4, num_kv_heads=2, head_dim=8, block_size=4, scale=0.41)
    kp, vp = oracle_pools(w)
    q_lens = [7, 12, 25, 16]  # longer than contexts 3, 9, 20, equal to 16
    q, cu = _queries_over_pool(w, q_lens, 22)
    out, lse = oracle.paged_attention(q, kp, vp, w.block_tables, w.context_lens, cu, w.scale,
                                      causal=False)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        k, v = logical_kv(w, s)
        K = k.double().permute(1, 0, 2).repeat_interleave(G, 0)[None]
        V = v.double().permute(1, 0, 2).repeat_interleave(G, 0)[None]
        r0, r1 = int(cu[s]), int(cu[s + 1])
        Q = q[r0:r1].double().permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(Q, K, V, scale=w.scale)[0].permute(1, 0, 2)
        ref_lse = torch.logsumexp((Q @ K.transpose(-1, -2)) * w.scale, -1)[0].permute(1, 0)
        np.testing.assert_allclose(out[r0:r1], ref.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[r0:r1], ref_lse.numpy(), rtol=1e-12, atol=1e-12)
    # rows of one sequence share one context: with equal queries they agree
    q2 = q.clone()
    q2[int(cu[2]):int(cu[3])] = q[int(cu[2])]
    out2, _ = oracle.paged_attention(q2, kp, vp, w.block_tables, w.context_lens, cu, w.scale,
                                     causal=False)
    assert np.all(out2[int(cu[2]):int(cu[3])] == out2[int(cu[2])])


def test_causal_window_longer_than_context_is_rejected():
    # a causal query j sits at position c - Lq + j, which is negative for
    # Lq > c: no such window exists, and the oracle refuses it (as it refuses
    # any non-empty window over an empty context)
    w = W.build("nc", 23, [3, 9], [1, 1], pool_factor=1.5, num_q_heads=4, num_kv_heads=2,
                head_dim=8, block_size=4)
    kp, vp = oracle_pools(w)
    q, cu = _queries_over_pool(w, [4, 2], 24)
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(q, kp, vp, w.block_tables, w.context_lens, cu, w.scale,
                               causal=True)
    cl0 = w.context_lens.clone()
    cl0[1] = 0
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(q, kp, vp, w.block_tables, cl0, cu, w.scale, causal=False)

"""Test helpers that build the oracle's own view of a workload.

Everything here runs on the CPU through the oracle only (never through the
CUDA path): the pool is filled with the sentinel and written by the oracle's
slot-mapped cache write, exactly as the GPU side fills its pool with the CUDA
cache-write kernel.
"""
import numpy as np
import torch

from oracle import oracle
from paged_kv_decode_18_gb300.workloads import POOL_SENTINEL_BITS


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_pools(w):
    """(k_pool, v_pool) as uint16 arrays after the history and the new tokens
    have been written by the oracle."""
    kp = np.full(w.pool_shape(), POOL_SENTINEL_BITS, dtype=np.uint16)
    vp = kp.copy()
    oracle.reshape_and_cache(w.k_hist, w.v_hist, w.slot_hist, kp, vp, w.block_size)
    oracle.reshape_and_cache(w.k_new, w.v_new, w.slot_new, kp, vp, w.block_size)
    return kp, vp


def logical_kv(w, s: int):
    """Sequence s's K and V in position order ([c, Hkv, D] bf16), straight
    from the generator (history then new tokens), without any pool."""
    h0, h1 = int(w.cu_hist[s]), int(w.cu_hist[s + 1])
    q0, q1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
    k = torch.cat([w.k_hist[h0:h1], w.k_new[q0:q1]])
    v = torch.cat([w.v_hist[h0:h1], w.v_new[q0:q1]])
    return k, v


def oracle_attention(w, kp=None, vp=None, num_threads=0, online_tile=0):
    if kp is None:
        kp, vp = oracle_pools(w)
    return oracle.paged_attention(w.q, kp, vp, w.block_tables, w.context_lens,
                                  w.cu_seqlens_q, w.scale, causal=w.causal,
                                  online_tile=online_tile, num_threads=num_threads)


def oracle_pools_i8(w):
    """(k codes, v codes, k scales, v scales) after the oracle's quantising
    cache write of the history and the new tokens; unwritten rows keep the
    sentinels (-128, NaN)."""
    from paged_kv_decode_18_gb300.workloads import POOL_SENTINEL_CODE
    kc = np.full(w.pool_shape(), POOL_SENTINEL_CODE, dtype=np.int8)
    vc = kc.copy()
    ks = np.full(w.pool_shape()[:3], np.nan, dtype=np.float32)
    vs = ks.copy()
    if w.k_hist.shape[0]:
        oracle.reshape_and_cache_i8(w.k_hist, w.v_hist, w.slot_hist, kc, vc, ks, vs)
    oracle.reshape_and_cache_i8(w.k_new, w.v_new, w.slot_new, kc, vc, ks, vs)
    return kc, vc, ks, vs


def oracle_attention_i8(w, pools=None, num_threads=0):
    kc, vc, ks, vs = oracle_pools_i8(w) if pools is None else pools
    return oracle.paged_attention_i8(w.q, kc, vc, ks, vs, w.block_tables, w.context_lens,
                                     w.cu_seqlens_q, w.scale, causal=w.causal,
                                     num_threads=num_threads)


def oracle_pools_f8(w):
    """(k codes, v codes, k scales, v scales) of the fp8 (E4M3) pool after the
    oracle's quantising cache write of the history and the new tokens;
    unwritten rows keep the sentinels (0x7F, NaN)."""
    from paged_kv_decode_18_gb300.workloads import POOL_SENTINEL_F8
    kc = np.full(w.pool_shape(), POOL_SENTINEL_F8, dtype=np.uint8)
    vc = kc.copy()
    ks = np.full(w.pool_shape()[:3], np.nan, dtype=np.float32)
    vs = ks.copy()
    if w.k_hist.shape[0]:
        oracle.reshape_and_cache_f8(w.k_hist, w.v_hist, w.slot_hist, kc, vc, ks, vs)
    oracle.reshape_and_cache_f8(w.k_new, w.v_new, w.slot_new, kc, vc, ks, vs)
    return kc, vc, ks, vs


def oracle_attention_f8(w, pools=None, num_threads=0):
    kc, vc, ks, vs = oracle_pools_f8(w) if pools is None else pools
    return oracle.paged_attention_f8(w.q, kc, vc, ks, vs, w.block_tables, w.context_lens,
                                     w.cu_seqlens_q, w.scale, causal=w.causal,
                                     num_threads=num_threads)

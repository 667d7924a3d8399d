"""CUDA slot-mapped cache write vs the oracle's: bit-exact over the whole pool
(untouched slots keep the sentinel)."""
import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, device
from tests.pools import oracle_pools

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


@pytest.mark.parametrize("name,sizes", [
    ("tiny", {}),
    ("engine", {}),
    ("ragged", dict(num_seqs=48, max_context=900)),
    ("mixed", dict(num_verify=5, lo=40, hi=300, prefill_chunk=40, prefill_offsets=(0, 24))),
])
def test_pool_matches_oracle(name, sizes):
    w = W.make(name, seed=1, **sizes)
    db = DeviceBatch(w)
    torch.cuda.synchronize()
    kp, vp = oracle_pools(w)
    gk, gv = db.pools_u16()
    assert np.array_equal(gk, kp) and np.array_equal(gv, vp)
    assert B.pa_debug_read_error() == 0


def test_random_unique_slots_and_skips():
    dev = device()
    NB, Hkv, D, BS, T = 40, 8, 128, 16, 300
    g = torch.Generator().manual_seed(3)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    slots = W.random_unique_slots(T, NB, BS, seed=4)
    slots[::7] = -1  # padding tokens are skipped
    kc = torch.full((NB, Hkv, BS, D), W.POOL_SENTINEL_BITS, dtype=torch.int16,
                    device=dev).view(torch.bfloat16)
    vc = kc.clone()
    B.pa_reshape_and_cache(k.to(dev), v.to(dev), slots.to(dev), kc, vc)
    kp = np.full((NB, Hkv, BS, D), W.POOL_SENTINEL_BITS, np.uint16)
    vp = kp.copy()
    oracle.reshape_and_cache(k, v, slots, kp, vp, BS)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), kp)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy().view(np.uint16), vp)


def test_chunked_write_bit_identical_on_gpu():
    w = W.mixed(seed=5, num_verify=4, lo=30, hi=200, prefill_chunk=64, prefill_offsets=(0, 48))
    dev = device()
    one = DeviceBatch(w)
    kc, vc = w.empty_pool(dev)
    kh, vh, sh = w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev)
    for a in range(0, kh.shape[0], 29):
        B.pa_reshape_and_cache(kh[a:a + 29], vh[a:a + 29], sh[a:a + 29], kc, vc)
    for a in range(0, w.num_q_tokens, 13):
        B.pa_reshape_and_cache(one.k_new[a:a + 13], one.v_new[a:a + 13],
                               one.slot_new[a:a + 13], kc, vc)
    assert torch.equal(kc.view(torch.int16), one.kc.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), one.vc.view(torch.int16))


def test_slot_past_pool_is_flagged_and_skipped():
    dev = device()
    NB, Hkv, D, BS = 4, 8, 128, 16
    k = torch.ones(3, Hkv, D, dtype=torch.bfloat16, device=dev)
    slots = torch.tensor([0, NB * BS, 5], dtype=torch.int64, device=dev)  # middle one is past
    kc = torch.zeros(NB, Hkv, BS, D, dtype=torch.bfloat16, device=dev)
    vc = kc.clone()
    B.pa_debug_read_error()
    B.pa_reshape_and_cache(k, k, slots, kc, vc)
    err = B.pa_debug_read_error()
    assert err & B.PA_DEVERR_SLOT_RANGE
    assert float(kc.float().sum()) == 2 * Hkv * D  # only the two valid rows landed
    assert B.pa_debug_read_error() == 0  # reading clears the word

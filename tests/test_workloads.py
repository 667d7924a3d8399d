"""The seeded generator: determinism, the structure each workload promises,
and the page's own KV-cache size figures."""
import json
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_decode_18_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_same_seed_same_bits():
    a, b = W.tiny(seed=3), W.tiny(seed=3)
    for f in ("q", "k_hist", "v_hist", "k_new", "block_tables", "slot_hist", "slot_new"):
        x, y = getattr(a, f), getattr(b, f)
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y), f
    c = W.tiny(seed=4)
    assert not torch.equal(a.q.view(torch.int16), c.q.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "engine", "ragged", "mixed"])
def test_slots_are_unique_and_inside_the_pool(name):
    w = W.make(name, seed=0)
    slots = torch.cat([w.slot_hist, w.slot_new])
    live = slots[slots >= 0]
    assert live.unique().numel() == live.numel()
    assert int(live.max()) < w.num_blocks * w.block_size
    # every table entry a sequence uses is a valid physical block
    for s in range(w.num_seqs):
        nb = (int(w.context_lens[s]) + w.block_size - 1) // w.block_size
        row = w.block_tables[s, :nb]
        assert int(row.min()) >= 0 and int(row.max()) < w.num_blocks
        assert torch.all(w.block_tables[s, nb:] == -1)


def test_named_shapes():
    t = W.tiny()
    assert t.num_seqs == 4 and t.num_blocks == 128
    assert int(t.context_lens.min()) >= 128 and int(t.context_lens.max()) <= 384
    e = W.engine()
    assert e.num_seqs == 64 and torch.all(e.context_lens == 384)
    assert e.num_blocks == 64 * 24 and e.num_q_tokens == 64
    r = W.ragged()
    assert r.num_seqs == 256 and int(r.context_lens.max()) <= 4096
    assert int(r.context_lens.min()) >= 1
    assert r.num_blocks == math.ceil(1.2 * r.meta["needed_blocks"])
    m = W.mixed()
    assert m.num_seqs == 50 and m.num_q_tokens == 48 * 5 + 2 * 512
    assert m.context_lens[-2:].tolist() == [512, 2048]
    assert m.q_lens[-2:].tolist() == [512, 512]


def test_ragged_prefix_is_shared_by_thirty_percent():
    r = W.ragged()
    nb = r.meta["prefix_tokens"] // r.block_size
    assert nb == 32
    first = r.block_tables[:, :nb]
    rows, counts = torch.unique(first, dim=0, return_counts=True)
    assert int(counts.max()) == round(0.3 * 256)
    sharers = (first == rows[counts.argmax()]).all(1)
    assert torch.all(r.context_lens[sharers] > 512)


def test_long_has_one_percent_outlier_keys():
    w = W.long(num_seqs=1, context=4096)
    norms = w.k_hist.float().norm(dim=-1).flatten()
    frac = float((norms > 4 * math.sqrt(128)).float().mean())
    assert 0.008 < frac < 0.012


def test_page_kv_cache_size_figures():
    """KV bytes per token of the built layout against the work-log's VRAM
    table (bf16, 28 layers, 8 KV heads of 128): the growth of VRAM between
    batch 128 and 256 is almost all KV cache, and the page quotes ~50 MB of
    cache at batch 1 and nearly 12 GB at batch 256."""
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_vram_qwen3_l4.json")))
    tokens = g["prompt_len"] + g["max_tokens"]
    per_token_layer = 2 * W.NUM_KV_HEADS * W.HEAD_DIM * 2   # K and V, bf16
    assert per_token_layer == 4096
    per_token = per_token_layer * g["model"]["layers"]
    vram = dict(g["vram_gb_by_batch"])
    slope = (vram[256] - vram[128]) * 1e9 / ((256 - 128) * tokens)
    assert abs(slope / per_token - 1) < 0.10
    assert abs(per_token * tokens / 1e6 / g["text_claims"]["cache_at_batch_1_mb_about"] - 1) < 0.15
    b256 = per_token * tokens * 256 / 1e9
    assert 0.9 * g["text_claims"]["cache_at_batch_256_gb_nearly"] < b256 <= 12.0


def test_random_unique_slots():
    s = W.random_unique_slots(100, 20, 16, seed=1)
    assert s.unique().numel() == 100 and int(s.max()) < 320 and s.dtype == torch.int64


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_8bit_empty_pool_tiles(fmt):
    # 2112-byte tiles: 16 x 128 sentinel codes, then 16 NaN scales; packing
    # and splitting the tile layout are inverse
    w = W.tiny(seed=3)
    kc, vc = w.empty_pool_f8() if fmt == "fp8" else w.empty_pool_i8()
    NB, H = w.num_blocks, w.num_kv_heads
    assert kc.shape == (NB, H, W.INT8_TILE_BYTES) == vc.shape and kc.dtype == torch.uint8
    codes, scales = W.int8_pool_split(kc)
    sentinel = W.POOL_SENTINEL_F8 if fmt == "fp8" else W.POOL_SENTINEL_CODE & 0xFF
    assert torch.all(codes.view(torch.uint8) == sentinel)
    assert torch.all(torch.isnan(scales))
    g = torch.Generator().manual_seed(4)
    c2 = torch.randint(-128, 128, codes.shape, generator=g, dtype=torch.int8)
    s2 = torch.rand(scales.shape, generator=g)
    back = W.int8_pool_split(W.int8_pool_pack(c2, s2))
    assert torch.equal(back[0], c2) and torch.equal(back[1], s2)

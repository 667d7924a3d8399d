"""Host-side logic of the benchmark, on CPU: how K steps map onto graph
replays, the algorithmic byte counts (logical and with a shared prefix
counted once), the sequence sampling of the oracle's CPU baseline, and one
short timed oracle run."""
import pytest
import torch

import bench
from paged_kv_decode_18_gb300 import workloads as W


@pytest.mark.parametrize("K", [1, 5, 20, 27, 28, 29, 56, 4000])
def test_graph_plan_covers_exactly_k_steps(K):
    chunk, full, rem = bench.graph_plan(K)
    assert chunk * full + rem == K
    assert 1 <= chunk <= bench.GRAPH_STEPS and 0 <= rem < chunk
    # 20 steps (fewer than one model's layers) are one graph of 20, not 20 graphs
    if K <= bench.GRAPH_STEPS:
        assert (chunk, full, rem) == (K, 1, 0)


def test_algorithmic_bytes_engine():
    w = W.engine(seed=1)
    # 64 x 384 tokens x 4096 B + q/out (64 x 16 x 128 x 2 x 2) + lse (64 x 16 x 4)
    # + 64 x 24 table entries x 4 + 64 context lengths x 4
    want = 64 * 384 * 4096 + 64 * 16 * 128 * 4 + 64 * 16 * 4 + 64 * 24 * 4 + 64 * 4
    assert bench.decode_algorithmic_bytes(w) == want == 101198080
    assert bench.decode_algorithmic_bytes(w, unique=True) == want


def test_unique_bytes_count_a_shared_prefix_once():
    w = W.ragged(seed=1, num_seqs=40, max_context=1000)
    seqs, t = w.meta["prefix_groups"][0]
    diff = bench.decode_algorithmic_bytes(w) - bench.decode_algorithmic_bytes(w, unique=True)
    assert diff == (len(seqs) - 1) * t * 4096
    # the same count as the physical blocks the tables reference
    ctx = w.context_lens.tolist()
    ids = set()
    for s, c in enumerate(ctx):
        ids.update(w.block_tables[s, :(c + 15) // 16].tolist())
    full_blocks = sum((c + 15) // 16 for c in ctx)
    assert full_blocks - len(ids) == (len(seqs) - 1) * (t // 16)


def test_subset_workload_keeps_rows_and_lengths():
    w = W.mixed(seed=2, num_verify=5, lo=40, hi=90, prefill_chunk=48, prefill_offsets=(0, 32))
    sub = bench.subset_workload(w, [1, 3, 6])
    assert sub.num_seqs == 3
    assert sub.context_lens.tolist() == [int(w.context_lens[i]) for i in (1, 3, 6)]
    assert sub.cu_seqlens_q.tolist() == [0, 5, 10, 58]
    assert torch.equal(sub.q[10:], w.q[int(w.cu_seqlens_q[6]):int(w.cu_seqlens_q[7])])
    assert torch.equal(sub.slot_new[:5], w.slot_new[5:10])


def test_oracle_rate_samples_when_a_step_is_too_long():
    w = W.tiny(seed=3)
    rate, threads, desc, steps, tokens = bench.oracle_rate(w, 0.2, num_threads=1)
    assert rate > 0 and threads == 1 and steps >= 3 and tokens == w.num_q_tokens
    # a budget far below one step's time makes it sample fewer sequences
    w2 = W.engine(seed=3)
    _, _, desc2, _, tokens2 = bench.oracle_rate(w2, 1e-6, num_threads=1, max_steps=1)
    assert tokens2 < w2.num_q_tokens and "sample" in desc2

"""Seeded synthetic workloads for paged KV-cache attention.

This module only draws random numbers and hands out physical blocks the way a
block manager would (a shuffled pool, per-sequence block tables, slot numbers
``phys_block * block_size + offset``). It holds none of the attention
arithmetic. Both the CUDA path (through its tests and the benchmark) and the
CPU oracle consume what it produces; it imports neither of them.

Shapes follow the attention of Qwen3-0.6B as described on the LLM inference
engine work-log (shehab-ashraf.github.io/posts/llm-inference, "The Baseline"
benchmark header: 28 layers, 16 query heads, head_dim 128) with 8 KV heads
(GQA group 2). Every draw comes from one ``torch.Generator`` seeded by the
caller, in a fixed order, so a (name, seed, sizes) triple always gives the
same bits.

A workload describes one attention call of one layer:

* history tokens (positions ``0 .. c - Lq - 1`` of each sequence) whose K/V
  are already in the pool before the step; their slots are in ``slot_hist``;
* the step's new tokens (the last ``Lq`` positions of each sequence), one per
  query row: their K/V (``k_new``/``v_new``) are written by the cache-write
  call at ``slot_new`` and then attended over together with the history;
* ``context_lens`` counts both, so query ``j`` of a sequence sits at position
  ``c - Lq + j``.

Unused pool slots hold ``POOL_SENTINEL_BITS`` (a bf16 NaN) so that a read of a
slot outside any context shows up in the results.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

POOL_SENTINEL_BITS = 0x7FC0  # bf16 quiet NaN
POOL_SENTINEL_CODE = -128    # int8 pools
POOL_SENTINEL_F8 = 0x7F      # fp8 (E4M3) pools: a NaN code
INT8_CODE_BYTES = 16 * 128   # codes of one (block, KV head) tile of the int8 pool
INT8_TILE_BYTES = INT8_CODE_BYTES + 16 * 4  # then the 16 rows' fp32 scales

NUM_Q_HEADS = 16
NUM_KV_HEADS = 8
HEAD_DIM = 128
BLOCK_SIZE = 16
NUM_LAYERS = 28  # only used to quote per-model-step context figures


@dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    causal: bool
    context_lens: torch.Tensor   # int32 [S]
    q_lens: torch.Tensor         # int32 [S]
    cu_seqlens_q: torch.Tensor   # int32 [S + 1]
    block_tables: torch.Tensor   # int32 [S, max_blocks_per_seq], -1 padded
    q: torch.Tensor              # bf16 [Tq, Hq, D]
    k_new: torch.Tensor          # bf16 [Tq, Hkv, D]
    v_new: torch.Tensor          # bf16 [Tq, Hkv, D]
    slot_new: torch.Tensor       # int64 [Tq]
    k_hist: torch.Tensor         # bf16 [Th, Hkv, D]
    v_hist: torch.Tensor         # bf16 [Th, Hkv, D]
    slot_hist: torch.Tensor      # int64 [Th], -1 where another sequence owns the slot
    cu_hist: torch.Tensor        # int32 [S + 1]
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_q_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max().item()) if self.num_seqs else 0

    def pool_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def empty_pool(self, device="cpu"):
        """A pool pair filled with the sentinel bit pattern."""
        pool = torch.full(self.pool_shape(), POOL_SENTINEL_BITS, dtype=torch.int16,
                          device=device)
        pool = pool.view(torch.bfloat16)
        return pool, pool.clone()

    def empty_pool_f8(self, device="cpu"):
        """An fp8 (E4M3) pool pair (k, v) in the same tile layout as the int8
        pool, uint8 [NB, Hkv, 2112]. Unwritten codes hold 0x7F (a NaN code,
        never produced by the quantiser) and unwritten scales NaN."""
        NB, H, BS, D = self.pool_shape()
        codes = torch.full((NB, H, BS, D), POOL_SENTINEL_F8, dtype=torch.uint8)
        scales = torch.full((NB, H, BS), float("nan"), dtype=torch.float32)
        t = int8_pool_pack(codes.view(torch.int8), scales).to(device)
        return t, t.clone()

    def empty_pool_i8(self, device="cpu"):
        """An int8 pool pair (k, v) in the library's tile layout, uint8
        [NB, Hkv, 2112]: each (block, KV head) tile holds its 16 x 128 codes,
        then its 16 fp32 row scales. Unwritten codes hold -128 (never produced
        by the quantiser) and unwritten scales NaN."""
        NB, H, BS, D = self.pool_shape()
        codes = torch.full((NB, H, BS, D), POOL_SENTINEL_CODE, dtype=torch.int8)
        scales = torch.full((NB, H, BS), float("nan"), dtype=torch.float32)
        t = int8_pool_pack(codes, scales).to(device)
        return t, t.clone()


def _randn_bf16(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def build(name: str, seed: int, context_lens, q_lens, *, num_blocks: int | None = None,
          pool_factor: float = 1.0, share_prefix_seqs=(), prefix_tokens: int = 0,
          outlier_frac: float = 0.0, outlier_gain: float = 8.0, causal: bool = True,
          num_q_heads: int = NUM_Q_HEADS, num_kv_heads: int = NUM_KV_HEADS,
          head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE,
          max_blocks_per_seq: int | None = None, scale: float | None = None,
          meta: dict | None = None, prefix_groups=()) -> Workload:
    """Build a workload from explicit per-sequence lengths.

    context_lens[s] counts all tokens of sequence s including its q_lens[s]
    new ones. Sequences listed in ``share_prefix_seqs`` use the same physical
    blocks for their first ``prefix_tokens`` positions (a refcounted prefix);
    their K/V there is one shared draw, written once (by the first sharer).
    ``prefix_groups`` generalises this to several disjoint groups, a list of
    (sequences, prefix_tokens); the single-group arguments are its first entry.
    ``outlier_frac`` of all key rows (token, KV head) are multiplied by
    ``outlier_gain`` before rounding to bf16.
    """
    g = torch.Generator().manual_seed(int(seed))
    ctx = [int(c) for c in context_lens]
    ql = [int(x) for x in q_lens]
    S = len(ctx)
    assert len(ql) == S
    for c, l in zip(ctx, ql):
        assert 0 <= l <= c, (l, c)
    BS = block_size
    groups = []  # (sorted sequences, prefix tokens)
    legacy = sorted(set(int(s) for s in share_prefix_seqs))
    if legacy:
        groups.append((legacy, int(prefix_tokens)))
    for seqs, tokens in prefix_groups:
        groups.append((sorted(set(int(s) for s in seqs)), int(tokens)))
    group_of = {}
    for gi, (seqs, tokens) in enumerate(groups):
        assert tokens % BS == 0 and tokens > 0 and seqs
        for s in seqs:
            assert s not in group_of, "prefix groups must be disjoint"
            group_of[s] = gi
            # a sharer's own new tokens must land past the shared prefix
            assert ctx[s] - ql[s] >= tokens, (s, ctx[s], ql[s])
    sharers = sorted(group_of)
    nblk = [(c + BS - 1) // BS for c in ctx]
    needed = sum(nblk) - sum((t // BS) * (len(ss) - 1) for ss, t in groups)
    if num_blocks is None:
        num_blocks = max(int(math.ceil(needed * pool_factor)), needed, 1)
    assert num_blocks >= needed, (num_blocks, needed)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(nblk + [1])

    # --- block manager: shuffled pool, per-sequence tables -----------------
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    tables = torch.full((S, max_blocks_per_seq), -1, dtype=torch.int32)
    cursor = 0
    prefix_ids = []
    for seqs, tokens in groups:
        prefix_ids.append(perm[cursor:cursor + tokens // BS])
        cursor += tokens // BS
    for s in range(S):
        row = []
        if s in group_of:
            row.extend(prefix_ids[group_of[s]].tolist())
        k = nblk[s] - len(row)
        row.extend(perm[cursor:cursor + k].tolist())
        cursor += k
        if row:
            tables[s, :len(row)] = torch.tensor(row, dtype=torch.int32)

    def slots_of(s: int, p0: int, p1: int) -> torch.Tensor:
        """Slots the block manager gave positions p0 .. p1-1 of sequence s."""
        p = torch.arange(p0, p1, dtype=torch.int64)
        return tables[s].to(torch.int64)[p // BS] * BS + p % BS

    # --- data --------------------------------------------------------------
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    hist_lens = [c - l for c, l in zip(ctx, ql)]
    Th, Tq = sum(hist_lens), sum(ql)
    prefix_kv = []
    for seqs, tokens in groups:
        pk = _randn_bf16(g, (tokens, Hkv, D))
        pv = _randn_bf16(g, (tokens, Hkv, D))
        prefix_kv.append((pk, pv))
    k_hist = _randn_bf16(g, (Th, Hkv, D))
    v_hist = _randn_bf16(g, (Th, Hkv, D))
    k_new = _randn_bf16(g, (Tq, Hkv, D))
    v_new = _randn_bf16(g, (Tq, Hkv, D))
    q = _randn_bf16(g, (Tq, Hq, D))
    slot_hist = torch.empty(Th, dtype=torch.int64)
    slot_new = torch.empty(Tq, dtype=torch.int64)
    cu_hist = torch.zeros(S + 1, dtype=torch.int32)
    cu_q = torch.zeros(S + 1, dtype=torch.int32)
    th = 0
    tq = 0
    for s in range(S):
        h = hist_lens[s]
        slot_hist[th:th + h] = slots_of(s, 0, h)
        if s in group_of:
            seqs, tokens = groups[group_of[s]]
            pk, pv = prefix_kv[group_of[s]]
            k_hist[th:th + tokens] = pk
            v_hist[th:th + tokens] = pv
            if s != seqs[0]:
                slot_hist[th:th + tokens] = -1  # the group's first sequence writes these
        slot_new[tq:tq + ql[s]] = slots_of(s, h, h + ql[s])
        th += h
        tq += ql[s]
        cu_hist[s + 1] = th
        cu_q[s + 1] = tq

    if outlier_frac > 0.0:
        # scale a seeded 1%-style subset of key rows (token, kv head)
        for kt in (k_hist, k_new):
            n_rows = kt.shape[0] * Hkv
            if n_rows == 0:
                continue
            n_out = max(1, int(round(outlier_frac * n_rows)))
            rows = torch.randperm(n_rows, generator=g)[:n_out]
            flat = kt.view(n_rows, D)
            flat[rows] = (flat[rows].float() * outlier_gain).to(torch.bfloat16)

    return Workload(
        name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=BS,
        num_blocks=int(num_blocks), max_blocks_per_seq=int(max_blocks_per_seq),
        scale=float(scale if scale is not None else 1.0 / math.sqrt(D)), causal=causal,
        context_lens=torch.tensor(ctx, dtype=torch.int32),
        q_lens=torch.tensor(ql, dtype=torch.int32), cu_seqlens_q=cu_q,
        block_tables=tables, q=q, k_new=k_new, v_new=v_new, slot_new=slot_new,
        k_hist=k_hist, v_hist=v_hist, slot_hist=slot_hist, cu_hist=cu_hist,
        meta=dict(meta or {}, seed=int(seed), needed_blocks=int(needed),
                  shared_prefix_seqs=len(sharers),
                  prefix_tokens=int(groups[0][1]) if groups else 0,
                  prefix_groups=[(list(ss), int(t)) for ss, t in groups]))


# --------------------------------------------------------------------------
# The five named workloads. Sizes can be reduced for parity tests; the
# defaults are the full sizes.
# --------------------------------------------------------------------------

def tiny(seed: int = 0, num_seqs: int = 4, lo: int = 128, hi: int = 384,
         num_blocks: int = 128) -> Workload:
    """Batch 4 decode, contexts uniform in [128, 384], a 128-block pool whose
    tables are a seeded random permutation."""
    g = torch.Generator().manual_seed(int(seed) * 7919 + 1)
    ctx = torch.randint(lo, hi + 1, (num_seqs,), generator=g).tolist()
    return build("tiny", seed, ctx, [1] * num_seqs, num_blocks=num_blocks,
                 meta={"config": "tiny paged decode"})


def engine(seed: int = 0, num_seqs: int = 64, context: int = 384) -> Workload:
    """Engine-shaped decode: batch 64, every context 384 (128-token prompt +
    256 generated), a shuffled pool of exactly the blocks needed, and one new
    token per sequence written through a random slot mapping."""
    return build("engine", seed, [context] * num_seqs, [1] * num_seqs, pool_factor=1.0,
                 meta={"config": "engine-shaped decode"})


def ragged(seed: int = 0, num_seqs: int = 256, max_context: int = 4096,
           share_frac: float = 0.30, prefix_tokens: int = 512,
           pool_factor: float = 1.2) -> Workload:
    """Ragged continuous batch: contexts log-uniform in [1, max_context];
    ``share_frac`` of the sequences (seeded choice) share a refcounted
    ``prefix_tokens`` prefix, their contexts raised to prefix_tokens + 1 so
    that their own new token lands past it. Pool = 1.2x the blocks needed."""
    g = torch.Generator().manual_seed(int(seed) * 7919 + 3)
    u = torch.rand(num_seqs, generator=g, dtype=torch.float64)
    ctx = torch.floor(torch.exp(u * math.log(max_context + 1))).clamp(1, max_context)
    ctx = ctx.to(torch.int64).tolist()
    n_share = int(round(share_frac * num_seqs))
    sharers = torch.randperm(num_seqs, generator=g)[:n_share].tolist()
    if n_share:
        prefix_tokens = min(prefix_tokens, max_context - 1 - (max_context - 1) % BLOCK_SIZE)
    for s in sharers:
        ctx[s] = max(ctx[s], prefix_tokens + 1)
    return build("ragged", seed, ctx, [1] * num_seqs, pool_factor=pool_factor,
                 share_prefix_seqs=sharers, prefix_tokens=prefix_tokens if n_share else 0,
                 meta={"config": "ragged continuous batch"})


def long(seed: int = 0, num_seqs: int = 8, context: int = 32768,
         outlier_frac: float = 0.01) -> Workload:
    """Long-context decode: batch 8 at 32768 tokens each, 1% of key rows
    scaled x8 (outlier logits)."""
    return build("long", seed, [context] * num_seqs, [1] * num_seqs, pool_factor=1.0,
                 outlier_frac=outlier_frac, meta={"config": "long-context split-K"})


def shared_prompt(seed: int = 0, num_seqs: int = 128, prefix_tokens: int = 4096,
                  lo: int = 1, hi: int = 512, pool_factor: float = 1.1) -> Workload:
    """Decode batch behind one long shared prompt: every sequence holds the
    same ``prefix_tokens`` (same physical blocks) plus a private suffix of
    uniform length in [lo, hi] whose last token is the step's new one."""
    g = torch.Generator().manual_seed(int(seed) * 7919 + 5)
    suf = torch.randint(lo, hi + 1, (num_seqs,), generator=g).tolist()
    ctx = [prefix_tokens + x for x in suf]
    return build("shared_prompt", seed, ctx, [1] * num_seqs, pool_factor=pool_factor,
                 prefix_groups=[(list(range(num_seqs)), prefix_tokens)],
                 meta={"config": "shared-prompt decode (cascade)"})


def mixed(seed: int = 0, num_verify: int = 48, verify_q: int = 5, lo: int = 256,
          hi: int = 8192, prefill_chunk: int = 512, prefill_offsets=(0, 1536),
          pool_factor: float = 1.1) -> Workload:
    """Mixed verify + chunked prefill: ``num_verify`` sequences scoring
    1 + 4 draft tokens each at contexts uniform in [lo, hi], plus one
    sequence per prefill offset whose 512-token chunk starts at that offset
    (earlier tokens already cached). All causal over one shuffled pool."""
    g = torch.Generator().manual_seed(int(seed) * 7919 + 5)
    ctx = torch.randint(lo, hi + 1, (num_verify,), generator=g).tolist()
    ql = [verify_q] * num_verify
    for off in prefill_offsets:
        ctx.append(int(off) + prefill_chunk)
        ql.append(prefill_chunk)
    return build("mixed", seed, ctx, ql, pool_factor=pool_factor,
                 meta={"config": "mixed verify + chunked prefill"})


def int8_pool_pack(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """(codes int8 [NB, H, 16, 128], scales fp32 [NB, H, 16]) -> the tile
    layout, uint8 [NB, H, 2112] (codes, then scales, per tile). Layout only."""
    NB, H = codes.shape[:2]
    t = torch.empty((NB, H, INT8_TILE_BYTES), dtype=torch.uint8, device=codes.device)
    t[..., :INT8_CODE_BYTES] = codes.contiguous().view(torch.uint8).reshape(NB, H, -1)
    t[..., INT8_CODE_BYTES:] = scales.contiguous().view(torch.uint8).reshape(NB, H, -1)
    return t


def int8_pool_split(t: torch.Tensor):
    """The tile layout uint8 [NB, H, 2112] -> (codes int8 [NB, H, 16, 128],
    scales fp32 [NB, H, 16]), copies. Layout only."""
    NB, H = t.shape[:2]
    codes = t[..., :INT8_CODE_BYTES].contiguous().view(torch.int8).reshape(NB, H, 16, 128)
    scales = t[..., INT8_CODE_BYTES:].contiguous().view(torch.float32)
    return codes, scales


CONFIGS = {
    "tiny": tiny,
    "engine": engine,
    "ragged": ragged,
    "long": long,
    "mixed": mixed,
}


def make(name: str, seed: int = 0, **sizes) -> Workload:
    return CONFIGS[name](seed=seed, **sizes)


def random_unique_slots(num_tokens: int, num_blocks: int, block_size: int,
                        seed: int) -> torch.Tensor:
    """A fully random set of distinct slots (int64), for a scatter test."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randperm(num_blocks * block_size, generator=g)[:num_tokens].to(torch.int64)


def cascade_groups(w: Workload):
    """The prefix-sharing structure of a workload, as the cascade decode call
    takes it: (seq_group [S], cu_group [G+1], group_members [M], prefix_lens [G])
    int32 tensors (members in increasing order) plus the host bounds
    (max_group_size, max_prefix_len)."""
    groups = w.meta.get("prefix_groups", [])
    S = w.num_seqs
    seq_group = torch.full((S,), -1, dtype=torch.int32)
    cu, members, plens = [0], [], []
    for gi, (seqs, tokens) in enumerate(groups):
        seqs = sorted(seqs)
        for s in seqs:
            seq_group[s] = gi
        members.extend(seqs)
        cu.append(len(members))
        plens.append(tokens)
    return (seq_group, torch.tensor(cu, dtype=torch.int32),
            torch.tensor(members, dtype=torch.int32), torch.tensor(plens, dtype=torch.int32),
            max((len(ss) for ss, _ in groups), default=0),
            max((t for _, t in groups), default=0))

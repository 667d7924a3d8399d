"""The calls are stream-ordered, allocate nothing and never synchronise, so an
engine can capture a whole decode step in a CUDA graph (S20, "The conflicts":
CUDA graphs need fixed shapes) and replay it as its inputs change in place.
Captured once, replayed on new contents, results match the oracle."""
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


def test_append_decode_graph_replays_on_new_inputs():
    wa = W.ragged(seed=61, num_seqs=40, max_context=900)
    wb = W.ragged(seed=62, num_seqs=40, max_context=900)
    dev = torch.device("cuda:0")
    # the same fixed-shape buffers serve both batches: pad tables / pools to the larger
    nb = max(wa.num_blocks, wb.num_blocks)
    mb = max(wa.max_blocks_per_seq, wb.max_blocks_per_seq)

    def padded(w):
        bt = torch.full((w.num_seqs, mb), -1, dtype=torch.int32)
        bt[:, :w.max_blocks_per_seq] = w.block_tables
        return bt

    kc = torch.empty(nb, 8, 16, 128, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    q = torch.empty_like(wa.q, device=dev)
    k_new = torch.empty_like(wa.k_new, device=dev)
    v_new = torch.empty_like(wa.v_new, device=dev)
    slots = torch.empty_like(wa.slot_new, device=dev)
    bt = torch.empty(wa.num_seqs, mb, dtype=torch.int32, device=dev)
    cl = torch.empty_like(wa.context_lens, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(q, kc, bt)
    ws = B.workspace(B.pa_decode_workspace_size(sh, 0), dev)

    def load(w):
        kc.view(torch.int16).fill_(W.POOL_SENTINEL_BITS)
        vc.view(torch.int16).fill_(W.POOL_SENTINEL_BITS)
        B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
        q.copy_(w.q)
        k_new.copy_(w.k_new)
        v_new.copy_(w.v_new)
        slots.copy_(w.slot_new)
        bt.copy_(padded(w))
        cl.copy_(w.context_lens)

    def step():
        B.pa_append_decode(k_new, v_new, slots, q, kc, vc, bt, cl, wa.scale, out, lse,
                           workspace=ws)

    load(wa)
    step()  # first call on the device before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for w in (wa, wb, wa):
        load(w)
        g.replay()
        torch.cuda.synchronize()
        assert B.pa_debug_read_error() == 0
        ref, ref_lse = oracle_attention(w)
        assert_attention_close(out, lse, ref, ref_lse, what=f"graph replay seed {w.meta['seed']}")


def test_varlen_graph_replay():
    w = W.mixed(seed=63, num_verify=6, lo=40, hi=600, prefill_chunk=64, prefill_offsets=(0, 80))
    db = DeviceBatch(w)
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.dev)
    sh = B.shape_of(db.q, db.kc, db.block_tables)
    ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, db.q.shape[0], w.max_q_len), db.dev)

    def call():
        B.pa_decode_varlen(db.q, db.kc, db.vc, db.block_tables, db.context_lens, db.cu_seqlens_q,
                           w.max_q_len, w.scale, out, lse, workspace=ws)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="varlen graph")


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_8bit_write_and_decode_graph_replay(fmt):
    # quantising cache write + 8-bit decode captured once; replayed after the
    # new rows and the queries change in place
    w = W.engine(seed=63, num_seqs=24, context=300)
    dev = torch.device("cuda:0")
    fp8 = fmt == "fp8"
    write = B.pa_reshape_and_cache_fp8 if fp8 else B.pa_reshape_and_cache_int8
    decode = B.pa_decode_fp8 if fp8 else B.pa_decode_int8
    ws_size = B.pa_decode_fp8_workspace_size if fp8 else B.pa_decode_int8_workspace_size
    kc, vc = w.empty_pool_f8(dev) if fp8 else w.empty_pool_i8(dev)
    write(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
    k_new, v_new, slots = w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev)
    q, bt, cl = w.q.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(q, kc, bt)
    ws = B.workspace(ws_size(sh, 0), dev)

    def step():
        write(k_new, v_new, slots, kc, vc)
        decode(q, kc, vc, bt, cl, w.scale, out, lse, workspace=ws)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gen = torch.Generator().manual_seed(64)
    k2 = torch.randn(w.k_new.shape, generator=gen).to(torch.bfloat16)
    v2 = torch.randn(w.v_new.shape, generator=gen).to(torch.bfloat16)
    q2 = torch.randn(w.q.shape, generator=gen).to(torch.bfloat16)
    k_new.copy_(k2)
    v_new.copy_(v2)
    q.copy_(q2)
    g.replay()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    w.k_new, w.v_new, w.q = k2, v2, q2
    from tests.pools import oracle_attention_f8, oracle_attention_i8
    ref, ref_lse = oracle_attention_f8(w) if fp8 else oracle_attention_i8(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"{fmt} graph replay")


def test_cascade_graph_replay():
    w = W.shared_prompt(seed=65, num_seqs=24, prefix_tokens=512, hi=200)
    db = DeviceBatch(w)
    sg, cu, mem, pl, mg, mp = [x.to(db.dev) if torch.is_tensor(x) else x
                               for x in W.cascade_groups(w)]
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.dev)
    sh = B.shape_of(db.q, db.kc, db.block_tables)
    ws = B.workspace(B.pa_decode_cascade_workspace_size(sh, pl.shape[0], mem.numel(), mg, mp),
                     db.dev)

    def call():
        B.pa_decode_cascade(db.q, db.kc, db.vc, db.block_tables, db.context_lens, sg, cu, mem,
                            pl, mg, mp, w.scale, out, lse, workspace=ws)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    q2 = torch.randn(w.q.shape, generator=torch.Generator().manual_seed(66)).to(torch.bfloat16)
    db.q.copy_(q2)
    g.replay()
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    w.q = q2
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="cascade graph replay")

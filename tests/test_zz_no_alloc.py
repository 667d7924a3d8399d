"""pa_decode_static_scratch: the decode entry point for callers that cannot
allocate device memory themselves (a plugin inside a runtime that owns every
device allocation, a serving loop whose memory is planned up front). It runs
the same split as pa_decode with a caller workspace, so its results must be
bit-identical to pa_decode's, and they must match the fp64 oracle. Calls in a
row on different batches -- both CTA shapes of the decode grid: the 6-warp
one for many (sequence, KV head) segments, the 8-warp one for few long ones --
check that nothing left in the shared scratch array by one call leaks into
the next. This file is collected last on purpose."""
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


def _no_alloc_call(db):
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.dev)
    B.pa_decode_static_scratch(db.q, db.kc, db.vc, db.block_tables, db.context_lens, db.w.scale,
                               out, lse)
    return out, lse


def test_scratch_need_fits_the_array():
    # every workload shape's balanced split fits the 8 MiB array on this device
    for name in ("tiny", "engine", "ragged", "long"):
        w = W.make(name, seed=1)
        sh = B.make_shape(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                          w.max_blocks_per_seq, w.num_blocks)
        need = B.pa_decode_workspace_size(sh, 0)
        assert 0 < need <= 8 << 20, (name, need)


def test_static_scratch_matches_workspace_entry_point():
    batches = [DeviceBatch(W.engine(seed=41)),
               DeviceBatch(W.ragged(seed=42, num_seqs=96, max_context=3000)),
               DeviceBatch(W.long(seed=43, num_seqs=2, context=8192))]
    refs = [db.decode(0) for db in batches]
    torch.cuda.synchronize()
    for db, (ref_out, ref_lse) in zip(batches, refs):  # calls in a row
        out, lse = _no_alloc_call(db)
        torch.cuda.synchronize()
        assert B.pa_debug_read_error() == 0
        # same split, same arithmetic: the same bits
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)
        oracle_out, oracle_lse = oracle_attention(db.w)
        assert_attention_close(out, lse, oracle_out, oracle_lse, what=db.w.name)

"""pa_decode_static_scratch: the decode entry point for callers that cannot
allocate device memory themselves (a plugin inside a runtime that owns every
device allocation, a serving loop whose memory is planned up front). It must
give the same results as pa_decode with a caller workspace. Two calls in a row
on different batches check that nothing left in the shared scratch array by
one call leaks into the next. This file is collected last on purpose."""
import pytest
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import DeviceBatch, LSE_ATOL, OUT_ATOL, OUT_RTOL

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


def test_static_scratch_matches_workspace_entry_point():
    batches = [DeviceBatch(W.engine(seed=41)),
               DeviceBatch(W.ragged(seed=42, num_seqs=96, max_context=3000))]
    refs = [db.decode(0) for db in batches]
    torch.cuda.synchronize()
    for db, (ref_out, ref_lse) in zip(batches, refs):  # two calls in a row
        out, lse = _no_alloc_call(db)
        torch.cuda.synchronize()
        assert B.pa_debug_read_error() == 0
        o, r = out.float(), ref_out.float()
        assert torch.all((o - r).abs() <= OUT_ATOL + OUT_RTOL * r.abs())
        assert (lse - ref_lse).abs().max().item() <= LSE_ATOL

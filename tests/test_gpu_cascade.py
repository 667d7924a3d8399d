"""CUDA cascade (shared-prefix) decode vs the fp64 oracle. The cascade only
reorganises the work -- shared prefix attended once per group, suffix per
sequence, split-K merge -- so its reference is plain paged attention over
each sequence's whole context: |out - ref| <= 1e-2 + 1e-2 |ref|,
|lse - ref| <= 1e-3. The cases run the cascade's own phases (policy
PA_CASCADE_ALWAYS); the last ones check which path the default policy takes."""
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


def cascade(db, groups=None, with_lse=True, policy=B.PA_CASCADE_ALWAYS):
    w, dev = db.w, db.dev
    sg, cu, mem, pl, mg, mp = W.cascade_groups(w) if groups is None else groups
    sg, cu, mem, pl = sg.to(dev), cu.to(dev), mem.to(dev), pl.to(dev)
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=dev) if with_lse else None
    sh = B.shape_of(db.q, db.kc, db.block_tables)
    ws = B.workspace(B.pa_decode_cascade_workspace_size(sh, pl.shape[0], mem.numel(), mg, mp),
                     dev)
    B.pa_decode_cascade(db.q, db.kc, db.vc, db.block_tables, db.context_lens, sg, cu, mem, pl,
                        mg, mp, w.scale, out, lse, workspace=ws, policy=policy)
    return out, lse


@pytest.mark.parametrize("sizes", [dict(num_seqs=40, max_context=1500), {}])
def test_cascade_ragged_matches_oracle(sizes):
    # the ragged batch: 30% of the sequences share a 512-token prefix
    w = W.ragged(seed=31, **sizes)
    assert w.meta["shared_prefix_seqs"] > 0
    db = DeviceBatch(w)
    out, lse = cascade(db)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"cascade ragged {sizes}")


def _multi_group_workload(seed):
    # contexts: group A (256-token prefix) = seqs 0, 2, 5, 9; group B (64) =
    # 1, 3; group C (32, one member whose context is exactly its prefix plus
    # one token); the rest share nothing. Seq 8's context is a multiple of 16.
    ctx = [300, 65, 257, 700, 40, 1000, 33, 33, 160, 511, 2]
    groups = [([0, 2, 5, 9], 256), ([1, 3], 64), ([6], 32)]
    return W.build("cascade", seed, ctx, [1] * len(ctx), pool_factor=1.3,
                   prefix_groups=groups)


def test_cascade_several_groups():
    w = _multi_group_workload(32)
    db = DeviceBatch(w)
    out, lse = cascade(db)
    out_nl, _ = cascade(db, with_lse=False)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="cascade groups")
    assert torch.equal(out, out_nl)


def test_cascade_prefix_covering_the_whole_context():
    # a one-member group whose prefix is its entire context (empty suffix),
    # and a group listing sequences that really share their first blocks
    w = _multi_group_workload(33)
    sg, cu, mem, pl, mg, mp = W.cascade_groups(w)
    s = 8  # context 160 = 10 blocks, in no group so far
    sg = sg.clone()
    sg[s] = pl.shape[0]
    cu = torch.cat([cu, torch.tensor([cu[-1] + 1], dtype=torch.int32)])
    mem = torch.cat([mem, torch.tensor([s], dtype=torch.int32)])
    pl = torch.cat([pl, torch.tensor([160], dtype=torch.int32)])
    db = DeviceBatch(w)
    out, lse = cascade(db, (sg, cu, mem, pl, max(mg, 1), max(mp, 160)))
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="cascade empty suffix")


def test_cascade_without_groups_equals_decode():
    w = W.tiny(seed=34)
    db = DeviceBatch(w)
    S = w.num_seqs
    groups = (torch.full((S,), -1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
              torch.zeros(0, dtype=torch.int32), torch.zeros(0, dtype=torch.int32), 0, 0)
    out, lse = cascade(db, groups)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what="cascade no groups")


def test_cascade_flags_an_inconsistent_description():
    w = _multi_group_workload(35)
    sg, cu, mem, pl, mg, mp = W.cascade_groups(w)
    sg = sg.clone()
    sg[4] = 0  # claims group 0 without being listed among its members
    db = DeviceBatch(w)
    cascade(db, (sg, cu, mem, pl, mg, mp))
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() & 0x8  # PA_DEVERR_QLEN_RANGE


@pytest.mark.parametrize("sizes", [dict(num_seqs=20, prefix_tokens=1024, hi=300), {}])
def test_cascade_shared_prompt_matches_oracle(sizes):
    # every sequence behind one long prompt (the full size: 128 x 4096 + 1..512);
    # the full-size case checks every row of the first and last 16 sequences
    w = W.shared_prompt(seed=36, **sizes)
    db = DeviceBatch(w)
    out, lse = cascade(db)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"cascade shared prompt {sizes}")


def test_auto_policy_takes_plain_decode_when_the_prefix_is_short():
    # ragged batch: 77 sequences behind a 512-token prefix save at most
    # 76 x 512 x 4 KB = 159 MB of prefix reads, below 256 MiB x 77/64: the
    # default policy runs pa_decode itself (the same bits)
    w = W.ragged(seed=37)
    db = DeviceBatch(w)
    out, lse = cascade(db, policy=B.PA_CASCADE_AUTO)
    ref_out, ref_lse = db.decode(0)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)


def test_auto_policy_takes_the_cascade_behind_a_long_prompt():
    # 128 sequences behind a 4096-token prompt save about 2.1 GB: the default
    # policy runs the cascade (the same bits as forcing it)
    w = W.shared_prompt(seed=38)
    db = DeviceBatch(w)
    out, lse = cascade(db, policy=B.PA_CASCADE_AUTO)
    out2, lse2 = cascade(db, policy=B.PA_CASCADE_ALWAYS)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)

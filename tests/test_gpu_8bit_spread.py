"""8-bit decode when the rows' scales spread far apart: within every block
the even positions hold V rows 2^26 times larger than the odd ones and keys of
zero, while the odd positions hold keys along the sequence's query (both query
heads of a KV head get the same query; scores 25 above the even ones). The
output is then carried by the small rows, whose weights times V scale are
2^-26 of the large rows' scale: a weight normalised by the tile's largest V
scale would vanish in f16. Both 8-bit formats must still match the fp64
oracle over the same dequantised rows within |out - ref| <= 1e-2 + 1e-2 |ref|,
|lse - ref| <= 1e-3."""
import pytest
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from paged_kv_decode_18_gb300 import workloads as W
from tests.gpu_util import Int8Batch, assert_attention_close
from tests.pools import oracle_attention_f8, oracle_attention_i8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


def _spread(w, ratio_log2=26, gap=25.0):
    k = w.k_hist.float().clone()
    v = w.v_hist.float().clone()
    q = w.q.clone()
    q[:, 1::2] = q[:, 0::2]  # both query heads of each KV head ask the same
    w.q = q
    cu = w.cu_hist.tolist()
    for s in range(w.num_seqs):
        n = cu[s + 1] - cu[s]
        even = torch.arange(cu[s], cu[s + 1])[0::2]
        odd = torch.arange(cu[s], cu[s + 1])[1::2]
        for h in range(w.num_kv_heads):
            qv = w.q[s, 2 * h].float()
            alpha = gap / (w.scale * float(qv @ qv))
            k[even, h] = 0.0
            v[even, h] *= 2.0 ** ratio_log2
            k[odd, h] = alpha * qv
        assert n == len(even) + len(odd)
    w.k_hist = k.to(torch.bfloat16)
    w.v_hist = v.to(torch.bfloat16)
    return w


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("num_splits", [0, 1])
def test_8bit_decode_with_far_apart_row_scales(fmt, num_splits):
    w = _spread(W.make("tiny", seed=71))
    db = Int8Batch(w, fp8=fmt == "fp8")
    out, lse = db.decode(num_splits)
    torch.cuda.synchronize()
    assert B.pa_debug_read_error() == 0
    ref, ref_lse = oracle_attention_f8(w) if fmt == "fp8" else oracle_attention_i8(w)
    assert_attention_close(out, lse, ref, ref_lse, what=f"{fmt} spread scales P={num_splits}")

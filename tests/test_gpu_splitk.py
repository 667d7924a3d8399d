"""CUDA split-K merge vs the oracle's merge on random partials, including
empty (-inf) partials and rows whose partials are all empty."""
import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild
from tests.gpu_util import assert_attention_close, device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    B.load()


@pytest.mark.parametrize("P,D", [(1, 128), (5, 128), (33, 128), (64, 128), (16, 64), (3, 256)])
def test_reduce_matches_oracle(P, D):
    dev = device()
    R, H = 9, 16
    g = np.random.default_rng(P * 1000 + D)
    po = g.standard_normal((R, H, P, D)).astype(np.float32)
    pl = (g.standard_normal((R, H, P)) * 4).astype(np.float32)
    if P > 1:
        pl[g.random((R, H, P)) < 0.3] = -np.inf  # empty partials
    pl[2, 3, :] = -np.inf                         # a row with nothing
    out = torch.empty(R, H, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(R, H, dtype=torch.float32, device=dev)
    B.pa_splitk_reduce(torch.from_numpy(po).to(dev), torch.from_numpy(pl).to(dev), out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.splitk_merge(po.reshape(R * H, P, D).astype(np.float64),
                                 pl.reshape(R * H, P).astype(np.float64))
    assert_attention_close(out, lse, ro.reshape(R, H, D), rl.reshape(R, H), what=f"P={P}")
    assert torch.all(out[2, 3] == 0) and torch.isneginf(lse[2, 3])

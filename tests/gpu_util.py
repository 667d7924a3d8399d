"""Helpers for the GPU parity tests: the device side of a workload goes
through the CUDA library only (the pool is written by the CUDA cache-write
kernel); the reference side through the oracle only."""
import numpy as np
import torch

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import workloads as W

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def device():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU test needs CUDA")
    return torch.device("cuda:0")


class DeviceBatch:
    """A workload's tensors on the GPU, with its pool filled by the CUDA cache
    write (history first, then the step's new tokens)."""

    def __init__(self, w, dev=None, write_new=True):
        dev = dev or device()
        self.w = w
        self.dev = dev
        self.kc, self.vc = w.empty_pool(dev)
        self.q = w.q.to(dev)
        self.k_new = w.k_new.to(dev)
        self.v_new = w.v_new.to(dev)
        self.slot_new = w.slot_new.to(dev)
        self.block_tables = w.block_tables.to(dev)
        self.context_lens = w.context_lens.to(dev)
        self.cu_seqlens_q = w.cu_seqlens_q.to(dev)
        if w.k_hist.shape[0]:
            B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev),
                                   self.kc, self.vc)
        if write_new:
            self.write_new()

    def write_new(self):
        B.pa_reshape_and_cache(self.k_new, self.v_new, self.slot_new, self.kc, self.vc)

    def pools_u16(self):
        return (self.kc.cpu().view(torch.int16).numpy().view(np.uint16),
                self.vc.cpu().view(torch.int16).numpy().view(np.uint16))

    def decode(self, num_splits=0, with_lse=True):
        out = torch.empty_like(self.q)
        lse = (torch.empty(self.q.shape[:2], dtype=torch.float32, device=self.dev)
               if with_lse else None)
        sh = B.shape_of(self.q, self.kc, self.block_tables)
        ws = B.workspace(B.pa_decode_workspace_size(sh, num_splits), self.dev)
        B.pa_decode(self.q, self.kc, self.vc, self.block_tables, self.context_lens,
                    self.w.scale, out, lse, num_splits=num_splits, workspace=ws)
        return out, lse

    def varlen(self, causal=True, with_lse=True):
        out = torch.empty_like(self.q)
        lse = (torch.empty(self.q.shape[:2], dtype=torch.float32, device=self.dev)
               if with_lse else None)
        sh = B.shape_of(self.q, self.kc, self.block_tables)
        mq = self.w.max_q_len
        ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, self.q.shape[0], mq), self.dev)
        B.pa_decode_varlen(self.q, self.kc, self.vc, self.block_tables, self.context_lens,
                           self.cu_seqlens_q, mq, self.w.scale, out, lse, causal=causal,
                           workspace=ws)
        return out, lse


def int8_pools_numpy(kc, vc):
    """Device int8 pools in the tile layout -> (k codes, v codes, k scales,
    v scales) numpy arrays, the oracle's form."""
    kcodes, kscales = W.int8_pool_split(kc.cpu())
    vcodes, vscales = W.int8_pool_split(vc.cpu())
    return kcodes.numpy(), vcodes.numpy(), kscales.numpy(), vscales.numpy()


class Int8Batch:
    """A workload on the GPU with its 8-bit pool (int8, or FP8 E4M3 with
    fp8=True) written by the CUDA quantising cache write (history first, then
    the step's new tokens)."""

    def __init__(self, w, fp8=False):
        dev = device()
        self.w, self.dev, self.fp8 = w, dev, fp8
        self.kc, self.vc = w.empty_pool_f8(dev) if fp8 else w.empty_pool_i8(dev)
        write = B.pa_reshape_and_cache_fp8 if fp8 else B.pa_reshape_and_cache_int8
        if w.k_hist.shape[0]:
            write(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), self.kc, self.vc)
        write(w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev), self.kc, self.vc)
        self.q = w.q.to(dev)
        self.bt = w.block_tables.to(dev)
        self.cl = w.context_lens.to(dev)

    def pools(self):
        """(k codes, v codes, k scales, v scales) as numpy, split out of the
        tile layout (FP8 codes as uint8)."""
        kc, vc, ks, vs = int8_pools_numpy(self.kc, self.vc)
        if self.fp8:
            kc, vc = kc.view(np.uint8), vc.view(np.uint8)
        return kc, vc, ks, vs

    def decode(self, num_splits=0, with_lse=True):
        out = torch.empty_like(self.q)
        lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=self.dev) \
            if with_lse else None
        sh = B.shape_of(self.q, self.kc, self.bt)
        if self.fp8:
            ws = B.workspace(B.pa_decode_fp8_workspace_size(sh, num_splits), self.dev)
            B.pa_decode_fp8(self.q, self.kc, self.vc, self.bt, self.cl, self.w.scale, out, lse,
                            num_splits=num_splits, workspace=ws)
        else:
            ws = B.workspace(B.pa_decode_int8_workspace_size(sh, num_splits), self.dev)
            B.pa_decode_int8(self.q, self.kc, self.vc, self.bt, self.cl, self.w.scale, out, lse,
                             num_splits=num_splits, workspace=ws)
        return out, lse


def assert_attention_close(out, lse, ref_out, ref_lse, rows=None, what=""):
    """|gpu - ref| <= 1e-2 + 1e-2 |ref| for out (bf16 vs fp64), |dlse| <= 1e-3."""
    got = out.float().cpu().numpy().astype(np.float64)
    ref_o = ref_out
    if rows is not None:
        got, ref_o = got[rows], ref_o[rows]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref_o)
    tol = OUT_ATOL + OUT_RTOL * np.abs(ref_o)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} out elements beyond tolerance, "
                           f"worst {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    if lse is not None:
        gl = lse.cpu().numpy().astype(np.float64)
        rl = ref_lse
        if rows is not None:
            gl, rl = gl[rows], rl[rows]
        inf = np.isinf(rl)
        assert np.array_equal(np.isinf(gl), inf), f"{what}: -inf rows differ"
        lerr = np.abs(gl[~inf] - rl[~inf])
        assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{what}: lse err {lerr.max():.3e}"

"""fp64 CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module. The product path (the CUDA library in
``paged_kv_decode_18_gb300``) never imports it, and this module imports
nothing from the product package.

It wraps ``pa_oracle.c`` (plain C, fp64, compiled with gcc) through ctypes and
marshals numpy / torch CPU tensors. bf16 tensors travel as their uint16 bit
patterns. See the header of ``pa_oracle.c`` for what each routine computes and
which passage of the source pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")

_lib = None
_lock = threading.Lock()

OK = 0
ERR_ARG = -1
ERR_RANGE = -2
ERR_NOMEM = -3


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into oracle/_build/libpa_oracle.so (gcc, -O2, OpenMP).

    No fast-math: the oracle keeps IEEE fp64 semantics.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", "-Wall",
           "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.pa_oracle_max_threads.restype = i32
        lib.pa_oracle_max_threads.argtypes = []
        lib.pa_oracle_reshape_and_cache.restype = i32
        lib.pa_oracle_reshape_and_cache.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P]
        lib.pa_oracle_attention_dense.restype = i32
        lib.pa_oracle_attention_dense.argtypes = [P, P, P, i64, i32, dbl, i32, i64, P, P]
        lib.pa_oracle_paged_attention.restype = i32
        lib.pa_oracle_paged_attention.argtypes = [
            P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, dbl, i32, i32, i64, i32, P, P]
        lib.pa_oracle_splitk_merge.restype = i32
        lib.pa_oracle_splitk_merge.argtypes = [P, P, i64, i32, i32, P, P]
        lib.pa_oracle_quantize_rows_i8.restype = i32
        lib.pa_oracle_quantize_rows_i8.argtypes = [P, i64, i32, P, P]
        lib.pa_oracle_reshape_and_cache_i8.restype = i32
        lib.pa_oracle_reshape_and_cache_i8.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P,
                                                       P, P]
        lib.pa_oracle_paged_attention_i8.restype = i32
        lib.pa_oracle_paged_attention_i8.argtypes = [
            P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, dbl, i32, i32, P, P]
        lib.pa_oracle_e4m3_values.restype = i32
        lib.pa_oracle_e4m3_values.argtypes = [P, i64, P]
        lib.pa_oracle_e4m3_codes.restype = i32
        lib.pa_oracle_e4m3_codes.argtypes = [P, i64, P]
        lib.pa_oracle_quantize_rows_f8.restype = i32
        lib.pa_oracle_quantize_rows_f8.argtypes = [P, i64, i32, P, P]
        lib.pa_oracle_reshape_and_cache_f8.restype = i32
        lib.pa_oracle_reshape_and_cache_f8.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P,
                                                       P, P]
        lib.pa_oracle_paged_attention_f8.restype = i32
        lib.pa_oracle_paged_attention_f8.argtypes = [
            P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, dbl, i32, i32, P, P]
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise OracleError(f"{what} failed with status {rc}")


def _as_u16(x) -> np.ndarray:
    """bf16 torch tensor / uint16 array -> contiguous uint16 numpy view."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                    .view(np.uint16))
    a = np.asarray(x)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits (uint16), got {a.dtype}")
    return np.ascontiguousarray(a)


def _as(x, dtype) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    a = np.asarray(x)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().pa_oracle_max_threads())


def reshape_and_cache(k, v, slot_mapping, k_cache: np.ndarray, v_cache: np.ndarray,
                      block_size: int) -> None:
    """Slot-mapped cache write, in place on uint16 pools [NB, Hkv, BS, D]."""
    lib = _load()
    k16, v16 = _as_u16(k), _as_u16(v)
    slots = _as(slot_mapping, np.int64)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("pools must be C-contiguous")
    if k_cache.dtype != np.uint16 or v_cache.dtype != np.uint16:
        raise TypeError("pools must be uint16 (bf16 bits)")
    T, Hkv, D = k16.shape
    NB = k_cache.shape[0]
    _check(lib.pa_oracle_reshape_and_cache(_ptr(k16), _ptr(v16), _ptr(slots), T, Hkv, D,
                                           block_size, NB, _ptr(k_cache), _ptr(v_cache)),
           "reshape_and_cache")


def attention_dense(q, K, V, scale: float, online_tile: int = 0):
    """One query [D] over dense keys/values [n, D] -> (out [D] fp64, lse float).

    online_tile == 0: two-pass softmax; > 0: online softmax with that tile.
    """
    lib = _load()
    q16, K16, V16 = _as_u16(q), _as_u16(K), _as_u16(V)
    n, D = K16.shape
    out = np.zeros(D, np.float64)
    lse = np.zeros(1, np.float64)
    mode = 1 if online_tile > 0 else 0
    _check(lib.pa_oracle_attention_dense(_ptr(q16), _ptr(K16), _ptr(V16), n, D, float(scale),
                                         mode, int(online_tile), _ptr(out), _ptr(lse)),
           "attention_dense")
    return out, float(lse[0])


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q,
                    scale: float, causal: bool = True, online_tile: int = 0,
                    num_threads: int = 0):
    """Paged attention in fp64 -> (out [Tq, Hq, D] fp64, lse [Tq, Hq] fp64)."""
    lib = _load()
    q16 = _as_u16(q)
    kc, vc = _as_u16(k_cache), _as_u16(v_cache)
    bt = _as(block_tables, np.int32)
    cl = _as(context_lens, np.int32)
    cu = _as(cu_seqlens_q, np.int32)
    Tq, Hq, D = q16.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.shape != kc.shape:
        raise ValueError("cache shape mismatch")
    S = cl.shape[0]
    if bt.ndim != 2 or bt.shape[0] != S or cu.shape[0] != S + 1 or int(cu[-1]) != Tq:
        raise ValueError("table / length shape mismatch")
    out = np.zeros((Tq, Hq, D), np.float64)
    lse = np.zeros((Tq, Hq), np.float64)
    mode = 1 if online_tile > 0 else 0
    rc = lib.pa_oracle_paged_attention(
        _ptr(q16), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), _ptr(cu), S, Hq, Hkv, D, BS,
        bt.shape[1], NB, float(scale), 1 if causal else 0, mode, int(online_tile),
        int(num_threads), _ptr(out), _ptr(lse))
    _check(rc, "paged_attention")
    return out, lse


def splitk_merge(part_out: np.ndarray, part_lse: np.ndarray):
    """part_out [rows, P, D] fp64, part_lse [rows, P] fp64 -> (out [rows, D], lse [rows])."""
    lib = _load()
    po = np.ascontiguousarray(part_out, np.float64)
    pl = np.ascontiguousarray(part_lse, np.float64)
    rows, P, D = po.shape
    if pl.shape != (rows, P):
        raise ValueError("part_lse shape mismatch")
    out = np.zeros((rows, D), np.float64)
    lse = np.zeros(rows, np.float64)
    _check(lib.pa_oracle_splitk_merge(_ptr(po), _ptr(pl), rows, P, D, _ptr(out), _ptr(lse)),
           "splitk_merge")
    return out, lse


def quantize_rows_i8(x):
    """Quantise rows of bf16 values (last axis = one group) -> (codes int8, scales fp32).

    Rule (see pa_oracle.c): amax = max |x|; inv = fl32(127 / amax);
    code = clamp(rint(fl32(x * inv)), -127, 127); scale = fl32(amax / 127).
    """
    lib = _load()
    x16 = _as_u16(x)
    D = x16.shape[-1]
    rows = x16.size // D
    codes = np.zeros(x16.shape, np.int8)
    scales = np.zeros(x16.shape[:-1], np.float32)
    _check(lib.pa_oracle_quantize_rows_i8(_ptr(x16), rows, D, _ptr(codes), _ptr(scales)),
           "quantize_rows_i8")
    return codes, scales


def reshape_and_cache_i8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> None:
    """Quantising cache write into int8 pools (numpy arrays, updated in place)."""
    lib = _load()
    k16, v16 = _as_u16(k), _as_u16(v)
    sm = _as(slot_mapping, np.int64)
    for a, dt in ((k_cache, np.int8), (v_cache, np.int8), (k_scale, np.float32),
                  (v_scale, np.float32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise ValueError("int8 pool arrays must be contiguous int8 / float32")
    T, Hkv, D = k16.shape
    NB, Hkv2, BS, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or k_scale.shape != (NB, Hkv, BS):
        raise ValueError("cache shape mismatch")
    _check(lib.pa_oracle_reshape_and_cache_i8(_ptr(k16), _ptr(v16), _ptr(sm), T, Hkv, D, BS, NB,
                                              _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                              _ptr(v_scale)), "reshape_and_cache_i8")


def paged_attention_i8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                       cu_seqlens_q, scale: float, causal: bool = True, num_threads: int = 0):
    """Paged attention in fp64 over int8 pools (rows dequantised as code * scale)."""
    lib = _load()
    q16 = _as_u16(q)
    kc, vc = _as(k_cache, np.int8), _as(v_cache, np.int8)
    ks, vs = _as(k_scale, np.float32), _as(v_scale, np.float32)
    bt = _as(block_tables, np.int32)
    cl = _as(context_lens, np.int32)
    cu = _as(cu_seqlens_q, np.int32)
    Tq, Hq, D = q16.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.shape != kc.shape or ks.shape != (NB, Hkv, BS) or vs.shape != ks.shape:
        raise ValueError("cache shape mismatch")
    S = cl.shape[0]
    if bt.ndim != 2 or bt.shape[0] != S or cu.shape[0] != S + 1 or int(cu[-1]) != Tq:
        raise ValueError("table / length shape mismatch")
    out = np.zeros((Tq, Hq, D), np.float64)
    lse = np.zeros((Tq, Hq), np.float64)
    rc = lib.pa_oracle_paged_attention_i8(
        _ptr(q16), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(cl), _ptr(cu), S, Hq,
        Hkv, D, BS, bt.shape[1], NB, float(scale), 1 if causal else 0, int(num_threads),
        _ptr(out), _ptr(lse))
    _check(rc, "paged_attention_i8")
    return out, lse


# ---------------------------------------------------------------------------
# FP8 (E4M3) pool: codes as uint8, one fp32 scale per (token, KV head) row
# ---------------------------------------------------------------------------

def e4m3_values(codes) -> np.ndarray:
    """The value of each E4M3 code (uint8), fp64; NaN for the NaN codes."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, np.float64)
    _check(_load().pa_oracle_e4m3_values(_ptr(c), c.size, _ptr(out)), "e4m3_values")
    return out


def e4m3_codes(y) -> np.ndarray:
    """The finite E4M3 code nearest to each fp32 value (ties to the even code,
    saturating at +-448)."""
    a = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.zeros(a.shape, np.uint8)
    _check(_load().pa_oracle_e4m3_codes(_ptr(a), a.size, _ptr(out)), "e4m3_codes")
    return out


def quantize_rows_f8(x):
    """bf16 rows [..., D] -> (codes uint8 [..., D], scales fp32 [...])."""
    lib = _load()
    x16 = _as_u16(x)
    D = x16.shape[-1]
    rows = x16.size // D
    codes = np.zeros(x16.shape, np.uint8)
    scales = np.zeros(x16.shape[:-1], np.float32)
    _check(lib.pa_oracle_quantize_rows_f8(_ptr(x16), rows, D, _ptr(codes), _ptr(scales)),
           "quantize_rows_f8")
    return codes, scales


def reshape_and_cache_f8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> None:
    """Quantising cache write into fp8 pools (numpy arrays, updated in place)."""
    lib = _load()
    k16, v16 = _as_u16(k), _as_u16(v)
    sm = _as(slot_mapping, np.int64)
    for a, dt in ((k_cache, np.uint8), (v_cache, np.uint8), (k_scale, np.float32),
                  (v_scale, np.float32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise ValueError("fp8 pool arrays must be contiguous uint8 / float32")
    T, Hkv, D = k16.shape
    NB, Hkv2, BS, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or k_scale.shape != (NB, Hkv, BS):
        raise ValueError("cache shape mismatch")
    _check(lib.pa_oracle_reshape_and_cache_f8(_ptr(k16), _ptr(v16), _ptr(sm), T, Hkv, D, BS, NB,
                                              _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                              _ptr(v_scale)), "reshape_and_cache_f8")


def paged_attention_f8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                       cu_seqlens_q, scale: float, causal: bool = True, num_threads: int = 0):
    """Paged attention in fp64 over fp8 pools (rows dequantised as value(code) * scale)."""
    lib = _load()
    q16 = _as_u16(q)
    kc, vc = _as(k_cache, np.uint8), _as(v_cache, np.uint8)
    ks, vs = _as(k_scale, np.float32), _as(v_scale, np.float32)
    bt = _as(block_tables, np.int32)
    cl = _as(context_lens, np.int32)
    cu = _as(cu_seqlens_q, np.int32)
    Tq, Hq, D = q16.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.shape != kc.shape or ks.shape != (NB, Hkv, BS) or vs.shape != ks.shape:
        raise ValueError("cache shape mismatch")
    S = cl.shape[0]
    if bt.ndim != 2 or bt.shape[0] != S or cu.shape[0] != S + 1 or int(cu[-1]) != Tq:
        raise ValueError("table / length shape mismatch")
    out = np.zeros((Tq, Hq, D), np.float64)
    lse = np.zeros((Tq, Hq), np.float64)
    rc = lib.pa_oracle_paged_attention_f8(
        _ptr(q16), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(cl), _ptr(cu), S, Hq,
        Hkv, D, BS, bt.shape[1], NB, float(scale), 1 if causal else 0, int(num_threads),
        _ptr(out), _ptr(lse))
    _check(rc, "paged_attention_f8")
    return out, lse

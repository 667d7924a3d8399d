"""Thin Python binding of libpagedattn's C ABI (include/pa.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
dtype / contiguity / device, passes raw device pointers, the shape struct and
the current CUDA stream to the C entry point of the same name, and raises
``PAError`` on a non-zero status. All arithmetic runs in the library's CUDA
kernels; there is no fallback. If the library has not been built the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpagedattn.so")

PA_OK = 0
PA_ERR_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_WORKSPACE = -3
PA_ERR_CUDA = -4
PA_ERR_DEVICE = -5

PA_DEVERR_SLOT_RANGE = 0x1
PA_DEVERR_BLOCK_RANGE = 0x2
PA_DEVERR_CONTEXT_RANGE = 0x4
PA_DEVERR_QLEN_RANGE = 0x8
PA_DEVERR_PIPE_TIMEOUT = 0x10
PA_DEVERR_PLAN_OVERFLOW = 0x20

# every symbol include/pa.h declares
EXPORTED = (
    "pa_reshape_and_cache",
    "pa_decode",
    "pa_decode_workspace_size",
    "pa_decode_static_scratch",
    "pa_append_decode",
    "pa_decode_varlen",
    "pa_decode_varlen_workspace_size",
    "pa_reshape_and_cache_int8",
    "pa_decode_int8",
    "pa_decode_int8_workspace_size",
    "pa_reshape_and_cache_fp8",
    "pa_decode_fp8",
    "pa_decode_fp8_workspace_size",
    "pa_decode_cascade",
    "pa_decode_cascade_ex",
    "pa_decode_cascade_workspace_size",
    "pa_splitk_reduce",
    "pa_status_string",
    "pa_debug_read_error",
    "pa_debug_inject_missing_copy",
    "pa_version",
)


class pa_shape(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("block_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int),
        ("num_blocks", ctypes.c_int64),
    ]


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {pa_status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load the library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libpagedattn.so not found at {p}; build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        V, S = ctypes.c_void_p, ctypes.POINTER(pa_shape)
        i32, i64, f32, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.pa_reshape_and_cache.restype = i32
        lib.pa_reshape_and_cache.argtypes = [V, V, V, i64, V, V, S, V]
        lib.pa_decode.restype = i32
        lib.pa_decode.argtypes = [V, V, V, V, V, f32, V, V, S, i32, V, sz, V]
        lib.pa_decode_workspace_size.restype = sz
        lib.pa_decode_workspace_size.argtypes = [S, i32]
        lib.pa_append_decode.restype = i32
        lib.pa_append_decode.argtypes = [V, V, V, i64, V, V, V, V, V, f32, V, V, S, V, sz, V]
        lib.pa_decode_static_scratch.restype = i32
        lib.pa_decode_static_scratch.argtypes = [V, V, V, V, V, f32, V, V, S, V]
        lib.pa_decode_varlen.restype = i32
        lib.pa_decode_varlen.argtypes = [V, V, V, V, V, V, i64, i32, i32, f32, V, V, S, V, sz, V]
        lib.pa_decode_varlen_workspace_size.restype = sz
        lib.pa_decode_varlen_workspace_size.argtypes = [S, i64, i32]
        lib.pa_reshape_and_cache_int8.restype = i32
        lib.pa_reshape_and_cache_int8.argtypes = [V, V, V, i64, V, V, S, V]
        lib.pa_decode_int8.restype = i32
        lib.pa_decode_int8.argtypes = [V, V, V, V, V, f32, V, V, S, i32, V, sz, V]
        lib.pa_decode_int8_workspace_size.restype = sz
        lib.pa_decode_int8_workspace_size.argtypes = [S, i32]
        lib.pa_reshape_and_cache_fp8.restype = i32
        lib.pa_reshape_and_cache_fp8.argtypes = [V, V, V, i64, V, V, S, V]
        lib.pa_decode_fp8.restype = i32
        lib.pa_decode_fp8.argtypes = [V, V, V, V, V, f32, V, V, S, i32, V, sz, V]
        lib.pa_decode_fp8_workspace_size.restype = sz
        lib.pa_decode_fp8_workspace_size.argtypes = [S, i32]
        lib.pa_decode_cascade.restype = i32
        lib.pa_decode_cascade.argtypes = [V, V, V, V, V, V, i32, V, V, V, i32, i32, i32, f32,
                                          V, V, S, V, sz, V]
        lib.pa_decode_cascade_ex.restype = i32
        lib.pa_decode_cascade_ex.argtypes = [V, V, V, V, V, V, i32, V, V, V, i32, i32, i32, f32,
                                             V, V, S, i32, V, sz, V]
        lib.pa_decode_cascade_workspace_size.restype = sz
        lib.pa_decode_cascade_workspace_size.argtypes = [S, i32, i32, i32, i32]
        lib.pa_splitk_reduce.restype = i32
        lib.pa_splitk_reduce.argtypes = [V, V, i64, i32, i32, i32, V, V, V]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [i32]
        lib.pa_debug_read_error.restype = i32
        lib.pa_debug_read_error.argtypes = [V]
        lib.pa_debug_inject_missing_copy.restype = i32
        lib.pa_debug_inject_missing_copy.argtypes = [i32]
        lib.pa_version.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _check(rc: int, what: str):
    if rc != PA_OK:
        raise PAError(rc, what)


def make_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
               num_blocks) -> pa_shape:
    return pa_shape(int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim),
                    int(block_size), int(max_blocks_per_seq), int(num_blocks))


# bytes of one (block, KV head) tile of the int8 and FP8 pools: 16 x 128
# one-byte codes, then the 16 rows' fp32 scales
PA_INT8_TILE_BYTES = 2112
INT8_BLOCK, INT8_HEAD_DIM = 16, 128


def shape_of(q, k_cache, block_tables, num_seqs=None) -> pa_shape:
    """Shape struct from the tensors: q [*, Hq, D], k_cache [NB, Hkv, BS, D]
    (bf16) or [NB, Hkv, PA_INT8_TILE_BYTES] (uint8, the int8 or FP8 pool),
    block_tables [S, max_blocks]."""
    if k_cache.dim() == 3 and k_cache.dtype == torch.uint8:
        if k_cache.shape[2] != PA_INT8_TILE_BYTES:
            raise ValueError(f"8-bit pool tiles must be {PA_INT8_TILE_BYTES} bytes")
        NB, Hkv = k_cache.shape[:2]
        BS, D = INT8_BLOCK, INT8_HEAD_DIM
    else:
        NB, Hkv, BS, D = k_cache.shape
    S = block_tables.shape[0] if num_seqs is None else num_seqs
    return make_shape(S, q.shape[1], Hkv, D, BS, block_tables.shape[1], NB)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def pa_version() -> str:
    return load().pa_version().decode()


def pa_debug_read_error(stream=None) -> int:
    rc = load().pa_debug_read_error(_stream(stream))
    if rc < 0:
        raise PAError(rc, "pa_debug_read_error")
    return rc


def pa_debug_inject_missing_copy(flat_tile: int) -> None:
    """Failure-detection hook: the next decode launch leaves out the copy of
    one tile, so its bounded wait expires and flags PA_DEVERR_PIPE_TIMEOUT."""
    _check(load().pa_debug_inject_missing_copy(int(flat_tile)), "pa_debug_inject_missing_copy")


def pa_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    if k.shape != v.shape or k_cache.shape != v_cache.shape:
        raise ValueError("k/v or cache shapes differ")
    if slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("slot_mapping length != number of tokens")
    NB, Hkv, BS, D = k_cache.shape
    if k.shape[1:] != (Hkv, D):
        raise ValueError("k rows do not match the cache's [Hkv, D]")
    sh = make_shape(0, Hkv, Hkv, D, BS, 0, NB)
    _check(load().pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0],
                                       _ptr(k_cache), _ptr(v_cache), ctypes.byref(sh),
                                       _stream(stream)), "pa_reshape_and_cache")


def pa_decode_workspace_size(shape: pa_shape, num_splits: int = 0) -> int:
    return int(load().pa_decode_workspace_size(ctypes.byref(shape), int(num_splits)))


def _cache_write_q8(name, k, v, slot_mapping, k_cache, v_cache, stream):
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_cache, "k_cache", torch.uint8, 3)
    _need(v_cache, "v_cache", torch.uint8, 3)
    if k.shape != v.shape or k_cache.shape != v_cache.shape:
        raise ValueError("k/v or cache shapes differ")
    if slot_mapping.shape[0] != k.shape[0]:
        raise ValueError("slot_mapping length != number of tokens")
    sh = shape_of(k, k_cache, torch.empty((0, 0)))
    if k.shape[1:] != (sh.num_kv_heads, sh.head_dim):
        raise ValueError("k rows do not match the cache")
    _check(getattr(load(), name)(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0],
                                 _ptr(k_cache), _ptr(v_cache), ctypes.byref(sh),
                                 _stream(stream)), name)


def pa_reshape_and_cache_int8(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Quantising cache write into the int8 pool (uint8 tiles [NB, Hkv, 2112]:
    a tile's 16 x 128 codes, then its 16 fp32 row scales)."""
    _cache_write_q8("pa_reshape_and_cache_int8", k, v, slot_mapping, k_cache, v_cache, stream)


def pa_reshape_and_cache_fp8(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Quantising cache write into the FP8 (E4M3) pool (same tiles as int8)."""
    _cache_write_q8("pa_reshape_and_cache_fp8", k, v, slot_mapping, k_cache, v_cache, stream)


def pa_decode_cascade_workspace_size(shape: pa_shape, num_groups: int, num_members: int,
                                     max_group_size: int, max_prefix_len: int) -> int:
    return int(load().pa_decode_cascade_workspace_size(ctypes.byref(shape), int(num_groups),
                                                       int(num_members), int(max_group_size),
                                                       int(max_prefix_len)))


PA_CASCADE_AUTO = 0
PA_CASCADE_ALWAYS = 1
PA_CASCADE_PLAIN = 2


def pa_decode_cascade(q, k_cache, v_cache, block_tables, context_lens, seq_group, cu_group,
                      group_members, prefix_lens, max_group_size, max_prefix_len, scale, out,
                      lse=None, workspace=None, stream=None, policy=PA_CASCADE_AUTO) -> None:
    """Decode with shared prefixes attended once per group (same result as
    pa_decode). policy: PA_CASCADE_AUTO (the library decides whether the
    cascade pays), PA_CASCADE_ALWAYS or PA_CASCADE_PLAIN."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(seq_group, "seq_group", torch.int32, 1)
    _need(cu_group, "cu_group", torch.int32, 1)
    _need(prefix_lens, "prefix_lens", torch.int32, 1)
    if group_members.numel():
        _need(group_members, "group_members", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    sh = shape_of(q, k_cache, block_tables)
    G = prefix_lens.shape[0]
    if cu_group.shape[0] != G + 1 or seq_group.shape[0] != sh.num_seqs:
        raise ValueError("group description shapes do not match")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode_cascade_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), _ptr(context_lens), _ptr(seq_group),
                                       G, _ptr(cu_group),
                                       _ptr(group_members) if group_members.numel() else None,
                                       _ptr(prefix_lens), int(group_members.numel()),
                                       int(max_group_size), int(max_prefix_len), float(scale),
                                       _ptr(out), _ptr(lse), ctypes.byref(sh), int(policy),
                                       _ptr(workspace), ws_bytes, _stream(stream)),
           "pa_decode_cascade")


def pa_decode_int8_workspace_size(shape: pa_shape, num_splits: int = 0) -> int:
    return int(load().pa_decode_int8_workspace_size(ctypes.byref(shape), int(num_splits)))


def pa_decode_fp8_workspace_size(shape: pa_shape, num_splits: int = 0) -> int:
    return int(load().pa_decode_fp8_workspace_size(ctypes.byref(shape), int(num_splits)))


def _decode_q8(name, q, k_cache, v_cache, block_tables, context_lens, scale, out, lse,
               num_splits, workspace, stream):
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 3)
    _need(v_cache, "v_cache", torch.uint8, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k / v cache shapes differ")
    sh = shape_of(q, k_cache, block_tables)
    if q.shape[0] != sh.num_seqs or context_lens.shape[0] != sh.num_seqs:
        raise ValueError("q / context_lens rows != number of sequences")
    if out.shape != q.shape:
        raise ValueError("out shape != q shape")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(getattr(load(), name)(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 _ptr(context_lens), float(scale), _ptr(out), _ptr(lse),
                                 ctypes.byref(sh), int(num_splits), _ptr(workspace), ws_bytes,
                                 _stream(stream)), name)


def pa_decode_int8(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse=None,
                   num_splits: int = 0, workspace=None, stream=None) -> None:
    """Decode over the int8 pool with the dequantisation fused."""
    _decode_q8("pa_decode_int8", q, k_cache, v_cache, block_tables, context_lens, scale, out,
               lse, num_splits, workspace, stream)


def pa_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse=None,
                  num_splits: int = 0, workspace=None, stream=None) -> None:
    """Decode over the FP8 (E4M3) pool with the dequantisation fused."""
    _decode_q8("pa_decode_fp8", q, k_cache, v_cache, block_tables, context_lens, scale, out,
               lse, num_splits, workspace, stream)


def _prepared(cfn, args, stream, what, keep):
    """A zero-argument callable that makes one C-ABI call with arguments that
    were checked and converted once (the tensors in `keep` stay referenced).
    The stream goes last: fixed now when one was given, else the current
    torch stream at each call (so the call can also be captured in a graph)."""
    if stream is not None:
        full = args + (_stream(stream),)

        def call():
            rc = cfn(*full)
            if rc != PA_OK:
                raise PAError(rc, what)
    else:
        def call():
            rc = cfn(*args, _stream(None))
            if rc != PA_OK:
                raise PAError(rc, what)
    call.keep = keep
    return call


def prepare_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse=None,
                   num_splits: int = 0, workspace=None, stream=None):
    """pa_decode with its arguments checked and marshalled now; the returned
    callable makes the call each time it is invoked, on `stream` if one is
    given, else on the torch stream current at that moment. For serving loops
    that issue the same call on fixed buffers."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    sh = shape_of(q, k_cache, block_tables)
    if q.shape[0] != sh.num_seqs or context_lens.shape[0] != sh.num_seqs:
        raise ValueError("q / context_lens rows != number of sequences")
    if out.shape != q.shape:
        raise ValueError("out shape != q shape")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
            ctypes.c_float(scale), _ptr(out), _ptr(lse), ctypes.byref(sh),
            ctypes.c_int(num_splits), _ptr(workspace), ctypes.c_size_t(ws_bytes))
    keep = (q, k_cache, v_cache, block_tables, context_lens, out, lse, workspace, sh)
    return _prepared(load().pa_decode, args, stream, "pa_decode", keep)


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse=None,
              num_splits: int = 0, workspace=None, stream=None) -> None:
    prepare_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse,
                   num_splits, workspace, stream)()


def prepare_append_decode(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                          context_lens, scale, out, lse=None, workspace=None, stream=None):
    """pa_append_decode with its arguments checked and marshalled now (see
    prepare_decode)."""
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if k_new.shape != v_new.shape or slot_mapping.shape[0] != k_new.shape[0]:
        raise ValueError("k_new / v_new / slot_mapping disagree")
    sh = shape_of(q, k_cache, block_tables)
    if q.shape[0] != sh.num_seqs or context_lens.shape[0] != sh.num_seqs:
        raise ValueError("q / context_lens rows != number of sequences")
    if out.shape != q.shape:
        raise ValueError("out shape != q shape")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), ctypes.c_int64(k_new.shape[0]),
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
            ctypes.c_float(scale), _ptr(out), _ptr(lse), ctypes.byref(sh), _ptr(workspace),
            ctypes.c_size_t(ws_bytes))
    keep = (k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables, context_lens, out,
            lse, workspace, sh)
    return _prepared(load().pa_append_decode, args, stream, "pa_append_decode", keep)


def pa_append_decode(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                     context_lens, scale, out, lse=None, workspace=None, stream=None) -> None:
    """Cache write of the step's new K/V rows, then decode (balanced split), as
    one call whose decode preparation overlaps the write."""
    prepare_append_decode(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                          context_lens, scale, out, lse, workspace, stream)()


def pa_decode_static_scratch(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                             lse=None, stream=None) -> None:
    """pa_decode (balanced split) without a workspace, for callers that cannot
    allocate device memory: the split scratch is a fixed 8 MiB array inside the
    library. Calls that may overlap on the GPU share that array and race."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    sh = shape_of(q, k_cache, block_tables)
    if q.shape[0] != sh.num_seqs or context_lens.shape[0] != sh.num_seqs:
        raise ValueError("q / context_lens rows != number of sequences")
    if out.shape != q.shape:
        raise ValueError("out shape != q shape")
    _check(load().pa_decode_static_scratch(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(block_tables), _ptr(context_lens), float(scale),
                                           _ptr(out), _ptr(lse), ctypes.byref(sh),
                                           _stream(stream)), "pa_decode_static_scratch")


def pa_decode_varlen_workspace_size(shape: pa_shape, num_q_tokens: int, max_q_len: int) -> int:
    return int(load().pa_decode_varlen_workspace_size(ctypes.byref(shape), int(num_q_tokens),
                                                      int(max_q_len)))


def pa_decode_varlen(q, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q, max_q_len,
                     scale, out, lse=None, causal: bool = True, workspace=None,
                     stream=None) -> None:
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    sh = shape_of(q, k_cache, block_tables)
    if context_lens.shape[0] != sh.num_seqs or cu_seqlens_q.shape[0] != sh.num_seqs + 1:
        raise ValueError("context_lens / cu_seqlens_q length mismatch")
    if out.shape != q.shape:
        raise ValueError("out shape != q shape")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pa_decode_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), _ptr(cu_seqlens_q), q.shape[0],
                                   int(max_q_len), 1 if causal else 0, float(scale), _ptr(out),
                                   _ptr(lse), ctypes.byref(sh), _ptr(workspace), ws_bytes,
                                   _stream(stream)), "pa_decode_varlen")


def pa_splitk_reduce(part_out, part_lse, out, lse=None, stream=None) -> None:
    """part_out [rows, heads, P, D] fp32, part_lse [rows, heads, P] fp32 ->
    out [rows, heads, D] bf16, lse [rows, heads] fp32."""
    _need(part_out, "part_out", torch.float32, 4)
    _need(part_lse, "part_lse", torch.float32, 3)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    R, H, P, D = part_out.shape
    if part_lse.shape != (R, H, P) or out.shape != (R, H, D):
        raise ValueError("split-K shapes disagree")
    _check(load().pa_splitk_reduce(_ptr(part_out), _ptr(part_lse), R, H, P, D, _ptr(out),
                                   _ptr(lse), _stream(stream)), "pa_splitk_reduce")


# ---------------------------------------------------------------------------
# workspace convenience
# ---------------------------------------------------------------------------

def workspace(nbytes: int, device=None):
    """A device byte buffer of at least nbytes (256-byte aligned by torch's
    allocator), or None when nbytes is 0."""
    if nbytes <= 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")

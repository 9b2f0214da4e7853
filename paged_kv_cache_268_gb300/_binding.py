"""ctypes binding over libpkv.so (include/pkv.h).

Argument marshalling only: every step of the append and decode paths runs in
the library's CUDA kernels.  torch tensors supply device pointers and the
current stream; nothing here computes attention, and there is no CPU
fallback — a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

_LIB = None

PKV_F16, PKV_BF16 = 0, 1
_DT = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
HEADER = os.path.join(_build.INCLUDE, "pkv.h")


class PkvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "block_size",
        "num_blocks", "max_blocks_per_seq", "max_context_len", "dtype",
        "split_tokens")]


class Plan(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int32), ("split_tokens", ctypes.c_int32),
                ("num_splits", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("warps_per_cta", ctypes.c_int32),
                ("stages_per_warp", ctypes.c_int32), ("grid_ctas", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


def library_path() -> str:
    """libpkv.so to load: $PKV_LIBRARY if set, else the in-tree build."""
    return os.environ.get("PKV_LIBRARY") or _build.LIB


def load_library(path: str | None = None):
    """Load libpkv.so; raises if it has not been built (run build())."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(
            f"libpkv.so not found at {p}: build it first with "
            "`python -m paged_kv_cache_268_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(p)
    vp, i32, i32p, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_size_t
    sp = ctypes.POINTER(Shape)
    lib.pkv_kv_cache_append.argtypes = [sp, vp, vp, vp, i32, vp, vp, vp]
    lib.pkv_kv_cache_append.restype = ctypes.c_int
    lib.pkv_paged_attn_decode.argtypes = [sp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.pkv_paged_attn_decode.restype = ctypes.c_int
    lib.pkv_decode_step.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.pkv_decode_step.restype = ctypes.c_int
    lib.pkv_decode_plan.argtypes = [sp, ctypes.POINTER(Plan)]
    lib.pkv_decode_plan.restype = ctypes.c_int
    lib.pkv_workspace_bytes.argtypes = [sp, ctypes.POINTER(sz)]
    lib.pkv_workspace_bytes.restype = ctypes.c_int
    lib.pkv_get_device_error.argtypes = [i32p, vp]
    lib.pkv_get_device_error.restype = ctypes.c_int
    lib.pkv_strerror.argtypes = [ctypes.c_int]
    lib.pkv_strerror.restype = ctypes.c_char_p
    lib.pkv_launch_count.argtypes = []
    lib.pkv_launch_count.restype = ctypes.c_uint64
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = ctypes.c_int
    if path is None:
        _LIB = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions include/pkv.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pkv_\w+)\s*\(", text, flags=re.M)


def strerror(code: int) -> str:
    try:
        return load_library().pkv_strerror(code).decode()
    except RuntimeError:
        return "libpkv not loaded"


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check(fn: str, rc: int):
    if rc != 0:
        raise PkvError(fn, rc)


def make_shape(*, num_seqs=0, num_q_heads=1, num_kv_heads=1, head_dim=128, block_size=16,
               num_blocks=1, max_blocks_per_seq=1, max_context_len=1, dtype=PKV_F16,
               split_tokens=0) -> Shape:
    return Shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                 max_blocks_per_seq, max_context_len, dtype, split_tokens)


def _cache_shape(k_cache: torch.Tensor) -> tuple[int, int, int, int]:
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    return tuple(k_cache.shape)


def _dense(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def kv_cache_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """Scatter new K/V rows [T, Hkv, D] into the paged caches at slot_mapping [T]."""
    NB, Hkv, bs, D = _cache_shape(k_cache)
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dense(t, n, k_cache.dtype)
    _dense(slot_mapping, "slot_mapping", torch.int32)
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("k, v must be [T, Hkv, D] matching the caches")
    T = k.shape[0]
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [T]")
    shape = make_shape(num_kv_heads=Hkv, head_dim=D, block_size=bs, num_blocks=NB,
                       dtype=_DT[k_cache.dtype])
    lib = load_library()
    _check("pkv_kv_cache_append",
           lib.pkv_kv_cache_append(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(slot_mapping), T,
                                   _ptr(k_cache), _ptr(v_cache), _stream_ptr(stream)))


def decode_shape(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                 max_context_len: int | None = None, split_tokens: int = 0) -> Shape:
    NB, Hkv, bs, D = _cache_shape(k_cache)
    B, Hq, Dq = q.shape
    MB = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = MB * bs        # always a valid bound; needs no host sync
    return make_shape(num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                      num_blocks=NB, max_blocks_per_seq=MB, max_context_len=int(max_context_len),
                      dtype=_DT[q.dtype], split_tokens=int(split_tokens))


def decode_plan(shape: Shape) -> Plan:
    plan = Plan()
    _check("pkv_decode_plan", load_library().pkv_decode_plan(ctypes.byref(shape), ctypes.byref(plan)))
    return plan


def workspace_bytes(shape: Shape) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_workspace_bytes", load_library().pkv_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return int(n.value)


def alloc_workspace(shape: Shape, device=None) -> torch.Tensor | None:
    n = workspace_bytes(shape)
    if n == 0:
        return None
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=device or "cuda")


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: torch.Tensor | None = None, *, max_context_len: int | None = None,
                      split_tokens: int = 0, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """softmax(q . K^T * scale) . V per (sequence, query head) over the paged cache.

    q [B, Hq, D]; caches [NB, Hkv, bs, D]; block_tables [B, MB] int32;
    context_lens [B] int32.  Returns out [B, Hq, D] (allocated if not given).
    split_tokens: 0 = library's choice, > 0 = partition size, -1 = persistent
    schedule.
    """
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dense(t, n, q.dtype)
    _dense(block_tables, "block_tables", torch.int32)
    _dense(context_lens, "context_lens", torch.int32)
    if v_cache.shape != k_cache.shape or q.dim() != 3 or q.shape[2] != k_cache.shape[3]:
        raise ValueError("q must be [B, Hq, D]; caches [NB, Hkv, bs, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != q.shape[0] or context_lens.shape != (q.shape[0],):
        raise ValueError("block_tables must be [B, MB]; context_lens [B]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _dense(out, "out", q.dtype)
    shape = decode_shape(q, k_cache, block_tables, max_context_len, split_tokens)
    if workspace is None:
        workspace = alloc_workspace(shape, q.device)
    lib = load_library()
    _check("pkv_paged_attn_decode",
           lib.pkv_paged_attn_decode(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_tables), _ptr(context_lens), float(scale),
                                     _ptr(out), _ptr(workspace),
                                     0 if workspace is None else workspace.numel(),
                                     _stream_ptr(stream)))
    return out


def decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                context_lens: torch.Tensor, scale: float, out: torch.Tensor | None = None, *,
                max_context_len: int | None = None, split_tokens: int = 0,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Append this step's token (k_new, v_new: [B, Hkv, D]) at position L-1 of
    every sequence and run decode attention, in one launch (plus the reduce)."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"),
                 (v_cache, "v_cache")):
        _dense(t, n, q.dtype)
    _dense(block_tables, "block_tables", torch.int32)
    _dense(context_lens, "context_lens", torch.int32)
    NB, Hkv, bs, D = _cache_shape(k_cache)
    if k_new.shape != (q.shape[0], Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new, v_new must be [B, Hkv, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _dense(out, "out", q.dtype)
    shape = decode_shape(q, k_cache, block_tables, max_context_len, split_tokens)
    if workspace is None:
        workspace = alloc_workspace(shape, q.device)
    _check("pkv_decode_step",
           load_library().pkv_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k_new), _ptr(v_new),
                                          _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                          _ptr(context_lens), float(scale), _ptr(out),
                                          _ptr(workspace),
                                          0 if workspace is None else workspace.numel(),
                                          _stream_ptr(stream)))
    return out


def get_device_error(stream=None) -> int:
    """Read and clear the library's device-side error word (synchronises)."""
    code = ctypes.c_int32(0)
    _check("pkv_get_device_error",
           load_library().pkv_get_device_error(ctypes.byref(code), _stream_ptr(stream)))
    return int(code.value)


def launch_count() -> int:
    return int(load_library().pkv_launch_count())

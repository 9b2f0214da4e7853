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
        "split_tokens", "kernel")]


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
    lib.pkv_set_workspace.argtypes = [vp, sz]
    lib.pkv_set_workspace.restype = ctypes.c_int
    lib.pkv_paged_attn_decode.argtypes = [sp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.pkv_paged_attn_decode.restype = ctypes.c_int
    lib.pkv_decode_step.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.pkv_decode_step.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [sp, vp, vp, i32, vp, vp, i32, vp, i32, vp]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.pkv_bm_create.argtypes = [i32, i32, i32]
    lib.pkv_bm_create.restype = vp
    lib.pkv_bm_destroy.argtypes = [vp]
    lib.pkv_bm_destroy.restype = None
    lib.pkv_bm_add_sequence.argtypes = [vp, i64, i32]
    lib.pkv_bm_fork.argtypes = [vp, i64, i64]
    lib.pkv_bm_append_token.argtypes = [vp, i64, i32p, i32p, i32p]
    lib.pkv_bm_free_sequence.argtypes = [vp, i64]
    lib.pkv_bm_swap_out.argtypes = [vp, i64, i32, i32p, i32, i32p]
    lib.pkv_bm_swap_in.argtypes = [vp, i64, i32p, i32, i32p]
    lib.pkv_bm_num_free.argtypes = [vp, i32p, i32p]
    lib.pkv_bm_seq_info.argtypes = [vp, i64, i32p, i32p, i32p]
    lib.pkv_bm_block_tables.argtypes = [vp, ctypes.POINTER(i64), i32, i32, i32p, i32p]
    for n in ("add_sequence", "fork", "append_token", "free_sequence", "swap_out", "swap_in",
              "num_free", "seq_info", "block_tables"):
        getattr(lib, "pkv_bm_" + n).restype = ctypes.c_int
    lib.pkv_decode_plan.argtypes = [sp, ctypes.POINTER(Plan)]
    lib.pkv_decode_plan.restype = ctypes.c_int
    lib.pkv_decode_plan_for.argtypes = [sp, i32, ctypes.POINTER(Plan)]
    lib.pkv_decode_plan_for.restype = ctypes.c_int
    lib.pkv_workspace_bytes.argtypes = [sp, ctypes.POINTER(sz)]
    lib.pkv_workspace_bytes.restype = ctypes.c_int
    lib.pkv_get_device_error.argtypes = [i32p, vp]
    lib.pkv_get_device_error.restype = ctypes.c_int
    lib.pkv_selftest_wait_timeout.argtypes = [i32, vp]
    lib.pkv_selftest_wait_timeout.restype = ctypes.c_int
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


def _stream_ptr(stream, device=None) -> int:
    """The stream handle to launch on: `stream`, or the current stream of
    `device` (of the current device when None)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return int(stream.cuda_stream)


def _one_device(**tensors) -> torch.device:
    """The CUDA device every given tensor lives on (None entries skipped).
    The library launches on the current device with that device's TMA
    descriptors, so tensors of another GPU must never reach it."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, expected {dev} like the other tensors")
    return dev


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check(fn: str, rc: int):
    if rc != 0:
        raise PkvError(fn, rc)


def make_shape(*, num_seqs=0, num_q_heads=1, num_kv_heads=1, head_dim=128, block_size=16,
               num_blocks=1, max_blocks_per_seq=1, max_context_len=1, dtype=PKV_F16,
               split_tokens=0, kernel=0) -> Shape:
    return Shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                 max_blocks_per_seq, max_context_len, dtype, split_tokens, kernel)


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
    dev = _one_device(k=k, v=v, slot_mapping=slot_mapping, k_cache=k_cache, v_cache=v_cache)
    lib = load_library()
    with torch.cuda.device(dev):
        _check("pkv_kv_cache_append",
               lib.pkv_kv_cache_append(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                       T, _ptr(k_cache), _ptr(v_cache), _stream_ptr(stream, dev)))


def decode_shape(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                 max_context_len: int | None = None, split_tokens: int = 0,
                 kernel: int = 0) -> Shape:
    NB, Hkv, bs, D = _cache_shape(k_cache)
    B, Hq, Dq = q.shape
    MB = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = MB * bs        # always a valid bound; needs no host sync
    return make_shape(num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                      num_blocks=NB, max_blocks_per_seq=MB, max_context_len=int(max_context_len),
                      dtype=_DT[q.dtype], split_tokens=int(split_tokens), kernel=int(kernel))


def decode_plan(shape: Shape, num_sms: int | None = None) -> Plan:
    """How a decode call will run on the current device, or, with `num_sms`,
    on a device with that many SMs (host only, no GPU needed)."""
    plan = Plan()
    lib = load_library()
    if num_sms is None:
        _check("pkv_decode_plan", lib.pkv_decode_plan(ctypes.byref(shape), ctypes.byref(plan)))
    else:
        _check("pkv_decode_plan_for",
               lib.pkv_decode_plan_for(ctypes.byref(shape), int(num_sms), ctypes.byref(plan)))
    return plan


def workspace_bytes(shape: Shape) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_workspace_bytes", load_library().pkv_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)))
    return int(n.value)


def alloc_workspace(shape: Shape, device=None) -> torch.Tensor | None:
    """A workspace tensor for `shape` on `device` (None when none is needed).
    The size is planned on that device."""
    dev = torch.device(device or "cuda")
    with torch.cuda.device(dev):
        n = workspace_bytes(shape)
    if n == 0:
        return None
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=dev)


# Workspaces set with set_workspace, by device index (kept alive here).
_SET_WS: dict[int, torch.Tensor] = {}


def set_workspace(workspace: torch.Tensor | None, device=None) -> None:
    """Make `workspace` (a contiguous CUDA tensor) the workspace that decode
    calls on its device use when they are given none (pkv_set_workspace);
    None clears the setting of `device` (default: the current device)."""
    lib = load_library()
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        with torch.cuda.device(dev):
            _check("pkv_set_workspace", lib.pkv_set_workspace(None, 0))
        _SET_WS.pop(dev.index, None)
        return
    _dense(workspace, "workspace")
    with torch.cuda.device(workspace.device):
        _check("pkv_set_workspace", lib.pkv_set_workspace(_ptr(workspace), _nbytes(workspace)))
    _SET_WS[workspace.device.index] = workspace


def _workspace_for(shape: Shape, dev: torch.device, workspace):
    """The workspace tensor to pass: the given one, none when a workspace is
    set for `dev` (the library then uses that one), else a new one."""
    if workspace is not None:
        _dense(workspace, "workspace")
        return workspace
    if dev.index in _SET_WS:
        return None
    return alloc_workspace(shape, dev)


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: torch.Tensor | None = None, *, max_context_len: int | None = None,
                      split_tokens: int = 0, kernel: int = 0,
                      workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """softmax(q . K^T * scale) . V per (sequence, query head) over the paged cache.

    q [B, Hq, D]; caches [NB, Hkv, bs, D]; block_tables [B, MB] int32;
    context_lens [B] int32.  Returns out [B, Hq, D] (allocated if not given).
    split_tokens: 0 = library's choice, > 0 = tokens per split-KV partition.
    kernel: 0 = library's choice, 1 CUDA cores, 2 mma.sync, 3 tcgen05.
    workspace: the split-KV scratch.  None uses the one set with
    set_workspace for q's device, else allocates one of the planned size;
    pass or set one to keep allocation off the decode path.
    """
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dense(t, n, q.dtype)
    _dense(block_tables, "block_tables", torch.int32)
    _dense(context_lens, "context_lens", torch.int32)
    _check_decode_extents(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    else:
        _dense(out, "out", q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape [B, Hq, D]")
    dev = _one_device(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                      context_lens=context_lens, out=out, workspace=workspace)
    shape = decode_shape(q, k_cache, block_tables, max_context_len, split_tokens, kernel)
    workspace = _workspace_for(shape, dev, workspace)
    lib = load_library()
    with torch.cuda.device(dev):
        _check("pkv_paged_attn_decode",
               lib.pkv_paged_attn_decode(ctypes.byref(shape), _ptr(q), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
                                         float(scale), _ptr(out), _ptr(workspace),
                                         _nbytes(workspace), _stream_ptr(stream, dev)))
    return out


def _check_decode_extents(q, k_cache, v_cache, block_tables, context_lens):
    """The library sees only pointers and the shape it is given, so the
    tensors' extents must agree with that shape before any launch."""
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [NB, Hkv, bs, D] tensors of one shape")
    if q.dim() != 3 or q.shape[2] != k_cache.shape[3]:
        raise ValueError("q must be [B, Hq, D] with the caches' head_dim")
    if (block_tables.dim() != 2 or block_tables.shape[0] != q.shape[0]
            or context_lens.shape != (q.shape[0],)):
        raise ValueError("block_tables must be [B, MB]; context_lens [B]")


def _nbytes(t: torch.Tensor | None) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                context_lens: torch.Tensor, scale: float, out: torch.Tensor | None = None, *,
                max_context_len: int | None = None, split_tokens: int = 0, kernel: int = 0,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Append this step's token (k_new, v_new: [B, Hkv, D]) at position L-1 of
    every sequence and run decode attention, in one launch (plus the reduce).
    split_tokens and kernel as for paged_attn_decode."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"),
                 (v_cache, "v_cache")):
        _dense(t, n, q.dtype)
    _dense(block_tables, "block_tables", torch.int32)
    _dense(context_lens, "context_lens", torch.int32)
    _check_decode_extents(q, k_cache, v_cache, block_tables, context_lens)
    NB, Hkv, bs, D = _cache_shape(k_cache)
    if k_new.shape != (q.shape[0], Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new, v_new must be [B, Hkv, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _dense(out, "out", q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape [B, Hq, D]")
    dev = _one_device(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                      block_tables=block_tables, context_lens=context_lens, out=out,
                      workspace=workspace)
    shape = decode_shape(q, k_cache, block_tables, max_context_len, split_tokens, kernel)
    workspace = _workspace_for(shape, dev, workspace)
    with torch.cuda.device(dev):
        _check("pkv_decode_step",
               load_library().pkv_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k_new),
                                              _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                              _ptr(block_tables), _ptr(context_lens),
                                              float(scale), _ptr(out), _ptr(workspace),
                                              _nbytes(workspace), _stream_ptr(stream, dev)))
    return out


def copy_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                dst_v: torch.Tensor, pairs: torch.Tensor, stream=None) -> None:
    """Copy block pairs[i, 0] of (src_k, src_v) to block pairs[i, 1] of
    (dst_k, dst_v).  Pools are [NB, Hkv, bs, D] tensors on the GPU or in
    pinned host memory; pairs is an int32 [n, 2] tensor the GPU can read."""
    for t, n in ((src_k, "src_k"), (src_v, "src_v"), (dst_k, "dst_k"), (dst_v, "dst_v")):
        if not t.is_contiguous() or t.dim() != 4 or t.dtype != src_k.dtype:
            raise ValueError(f"{n} must be a contiguous [NB, Hkv, bs, D] tensor of one dtype")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must live on the GPU or in pinned host memory")
    if src_k.shape[1:] != dst_k.shape[1:] or src_v.shape != src_k.shape or dst_v.shape != dst_k.shape:
        raise ValueError("pools must share the block shape")
    if pairs.dtype != torch.int32 or not pairs.is_contiguous() or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be a contiguous int32 [n, 2] tensor")
    if not (pairs.is_cuda or pairs.is_pinned()):
        raise ValueError("pairs must live on the GPU or in pinned host memory")
    _, Hkv, bs, D = src_k.shape
    shape = make_shape(num_kv_heads=Hkv, head_dim=D, block_size=bs, num_blocks=src_k.shape[0],
                       dtype=_DT[src_k.dtype])
    on_gpu = {n: t for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k),
                                ("dst_v", dst_v), ("pairs", pairs)) if t.is_cuda}
    dev = _one_device(**on_gpu) if on_gpu else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check("pkv_copy_blocks",
               load_library().pkv_copy_blocks(ctypes.byref(shape), _ptr(src_k), _ptr(src_v),
                                              src_k.shape[0], _ptr(dst_k), _ptr(dst_v),
                                              dst_k.shape[0], _ptr(pairs), pairs.shape[0],
                                              _stream_ptr(stream, dev)))


class BlockManager:
    """Host-side block manager of the C library (pkv_bm_* in include/pkv.h)."""

    def __init__(self, num_gpu_blocks: int, num_cpu_blocks: int, block_size: int):
        self._lib = load_library()
        self._h = self._lib.pkv_bm_create(num_gpu_blocks, num_cpu_blocks, block_size)
        if not self._h:
            raise ValueError("bad block manager sizes")
        self.block_size = block_size

    def close(self):
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def _call(self, name, *args):
        _check("pkv_bm_" + name, getattr(self._lib, "pkv_bm_" + name)(self._h, *args))

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        self._call("add_sequence", seq_id, num_tokens)

    def fork(self, parent: int, child: int) -> None:
        self._call("fork", parent, child)

    def append_token(self, seq_id: int) -> tuple[int, int, int]:
        """(slot, copy_src, copy_dst); copy_* are -1 unless a shared block was copied."""
        s, a, b = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._call("append_token", seq_id, ctypes.byref(s), ctypes.byref(a), ctypes.byref(b))
        return s.value, a.value, b.value

    def free_sequence(self, seq_id: int) -> None:
        self._call("free_sequence", seq_id)

    def _pairs(self, name, *args, cap=1 << 16):
        import numpy as np
        buf = (ctypes.c_int32 * (2 * cap))()
        n = ctypes.c_int32()
        self._call(name, *args, buf, cap, ctypes.byref(n))
        return np.array(buf[: 2 * n.value], dtype=np.int32).reshape(-1, 2)

    def swap_out(self, seq_id: int, gpu_window: int):
        """(gpu id, cpu id) pairs [n, 2] of the blocks moved to the CPU pool."""
        return self._pairs("swap_out", seq_id, gpu_window)

    def swap_in(self, seq_id: int):
        """(cpu id, gpu id) pairs [n, 2] of the blocks moved back to the GPU."""
        return self._pairs("swap_in", seq_id)

    def num_free(self) -> tuple[int, int]:
        g, c = ctypes.c_int32(), ctypes.c_int32()
        self._call("num_free", ctypes.byref(g), ctypes.byref(c))
        return g.value, c.value

    def seq_info(self, seq_id: int) -> tuple[int, int, int]:
        a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._call("seq_info", seq_id, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
        return a.value, b.value, c.value

    def block_tables(self, seq_ids, max_blocks_per_seq: int):
        """(block_tables [n, MB] int32, context_lens [n] int32) as numpy arrays."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = ids.shape[0]
        tables = np.zeros((n, max_blocks_per_seq), dtype=np.int32)
        lens = np.zeros(n, dtype=np.int32)
        i32p = ctypes.POINTER(ctypes.c_int32)
        self._call("block_tables", ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                   max_blocks_per_seq, tables.ctypes.data_as(i32p), lens.ctypes.data_as(i32p))
        return tables, lens


def get_device_error(stream=None) -> int:
    """Read and clear the library's device-side error word (synchronises)."""
    code = ctypes.c_int32(0)
    _check("pkv_get_device_error",
           load_library().pkv_get_device_error(ctypes.byref(code), _stream_ptr(stream)))
    return int(code.value)


def selftest_wait_timeout(limit_us: int = 50_000, stream=None) -> None:
    """Run the bounded-wait self-test: a warp waits on an mbarrier nothing
    arrives on and gives up after limit_us, recording PKV_DEV_TIMEOUT (read it
    with get_device_error)."""
    _check("pkv_selftest_wait_timeout",
           load_library().pkv_selftest_wait_timeout(int(limit_us), _stream_ptr(stream)))


def launch_count() -> int:
    return int(load_library().pkv_launch_count())

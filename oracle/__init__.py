"""CPU oracle for paged decode attention and the KV append scatter.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library and its Python binding never import it, and it shares no code with
them: the arithmetic lives in ``pkv_oracle.c`` (plain C, fp64, no blocking or
reordering), compiled here with gcc into ``liboracle.so`` and called through
ctypes.

What it computes and which passage each step follows is written at the top of
``pkv_oracle.c``: softmax(q . K^T * scale) . V per (sequence, query head)
(second page, section 3.1, scaled_dot_product_attention), with K/V reached
through the block table by indirect addressing (third page, "PagedAttention"),
and the slot scatter of new K/V rows (first page, section 4.2 block manager;
third page, "continuous batching").

Pins (tests/test_oracle_pins.py) tie it to things other than itself:
closed forms, a hand-worked softmax, a library attention routine on contiguous
data, exhaustive format decoding, invariances, and planted-mistake checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, no vector ISA
    flags, so it gives the same results on x86 and Arm)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def load(path: str | None = None):
    """Load liboracle.so (building it first when missing or stale)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.pkv_oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.pkv_oracle_half_to_double.restype = ctypes.c_double
    lib.pkv_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.pkv_oracle_bf16_to_double.restype = ctypes.c_double
    lib.pkv_oracle_decode.argtypes = [i, i, i, i, i, i, i, i, u16p, u16p, u16p,
                                      i32p, i32p, ctypes.c_double, f64p]
    lib.pkv_oracle_decode.restype = i
    lib.pkv_oracle_decode_rows.argtypes = [i, i, i, i, i, i, i, u16p, u16p, u16p,
                                           i32p, i32p, ctypes.c_double, i32p, i,
                                           f64p]
    lib.pkv_oracle_decode_rows.restype = i
    lib.pkv_oracle_append.argtypes = [i, i, i, i, i, u16p, u16p, i32p, u16p,
                                      u16p]
    lib.pkv_oracle_append.restype = i
    lib.pkv_oracle_copy_blocks.argtypes = [i, i, i, i, i, i, u16p, u16p, i32p]
    lib.pkv_oracle_copy_blocks.restype = i
    return lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit element patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def widen(bits, dtype: int, lib=None) -> np.ndarray:
    """Exact widening of 16-bit patterns to float64 (the oracle's converter)."""
    lib = lib or load()
    bits = np.asarray(bits, dtype=np.uint16).ravel()
    fn = lib.pkv_oracle_half_to_double if dtype == F16 else lib.pkv_oracle_bf16_to_double
    return np.array([fn(int(b)) for b in bits], dtype=np.float64)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
           dtype: int, lib=None) -> np.ndarray:
    """out[B, Hq, D] (float64) for every sequence and query head.

    q: [B, Hq, D]; k_cache, v_cache: [NB, Hkv, bs, D] (16-bit patterns);
    block_tables: [B, MB] int32; context_lens: [B] int32."""
    lib = lib or load()
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = kc.shape
    assert D2 == D and vc.shape == kc.shape and bt.shape[0] == B and cl.shape == (B,)
    MB = bt.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    bad = lib.pkv_oracle_decode(B, Hq, Hkv, D, bs, NB, MB, dtype,
                                _ptr(q, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16),
                                _ptr(vc, ctypes.c_uint16), _ptr(bt, ctypes.c_int32),
                                _ptr(cl, ctypes.c_int32), float(scale),
                                _ptr(out, ctypes.c_double))
    if bad != 0:
        raise ValueError(f"oracle: {bad} rows break the input contract")
    return out


def decode_rows(rows, q, k_cache, v_cache, block_tables, context_lens,
                scale: float, dtype: int, lib=None) -> np.ndarray:
    """out[R, D] (float64) for the listed (sequence, query head) pairs."""
    lib = lib or load()
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    MB = bt.shape[1]
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    bad = lib.pkv_oracle_decode_rows(Hq, Hkv, D, bs, NB, MB, dtype,
                                     _ptr(q, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16),
                                     _ptr(vc, ctypes.c_uint16), _ptr(bt, ctypes.c_int32),
                                     _ptr(cl, ctypes.c_int32), float(scale),
                                     _ptr(rows, ctypes.c_int32), rows.shape[0],
                                     _ptr(out, ctypes.c_double))
    if bad != 0:
        raise ValueError(f"oracle: {bad} rows break the input contract")
    return out


def append(k, v, slot_mapping, k_cache, v_cache, lib=None):
    """Return copies of (k_cache, v_cache) with the new rows scattered in.

    k, v: [T, Hkv, D] 16-bit patterns; slot_mapping: [T] int32 (negative = skip).
    """
    lib = lib or load()
    k, v = _u16(k), _u16(v)
    sm = _i32(slot_mapping)
    kc = _u16(k_cache).copy()
    vc = _u16(v_cache).copy()
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = kc.shape
    assert Hkv2 == Hkv and D2 == D and sm.shape == (T,)
    bad = lib.pkv_oracle_append(T, Hkv, D, bs, NB, _ptr(k, ctypes.c_uint16),
                                _ptr(v, ctypes.c_uint16), _ptr(sm, ctypes.c_int32),
                                _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16))
    if bad != 0:
        raise ValueError(f"oracle: {bad} slots outside the pool")
    return kc, vc


def copy_blocks(src, dst, pairs, lib=None):
    """Return a copy of pool `dst` with block pairs[i, 0] of pool `src` copied
    to block pairs[i, 1] (pools [NB, Hkv, bs, D] of 16-bit patterns)."""
    lib = lib or load()
    src = _u16(src)
    out = _u16(dst).copy()
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    _, Hkv, bs, D = src.shape
    bad = lib.pkv_oracle_copy_blocks(pr.shape[0], Hkv, bs, D, src.shape[0], out.shape[0],
                                     _ptr(src, ctypes.c_uint16), _ptr(out, ctypes.c_uint16),
                                     _ptr(pr, ctypes.c_int32))
    if bad != 0:
        raise ValueError(f"oracle: {bad} pairs outside the pools")
    return out

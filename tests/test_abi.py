"""The C-ABI library loads, exports every symbol include/pkv.h declares, and
rejects bad arguments on the host (CPU only: no call here reaches a GPU)."""
import ctypes

import pytest

from paged_kv_cache_268_gb300 import _binding as B
from paged_kv_cache_268_gb300 import build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load_library()


def test_exports_every_declared_function(lib):
    names = B.header_functions()
    assert {"pkv_kv_cache_append", "pkv_paged_attn_decode", "pkv_workspace_bytes",
            "pkv_set_workspace", "pkv_decode_step", "pkv_decode_plan", "pkv_get_device_error",
            "pkv_strerror", "pkv_launch_count", "pkv_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_and_version(lib):
    assert lib.pkv_version() >= 100
    for code in range(0, -8, -1):
        assert lib.pkv_strerror(code)
    assert b"unknown" in lib.pkv_strerror(-99)
    assert lib.pkv_launch_count() == 0


def _shape(**kw):
    base = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                num_blocks=64, max_blocks_per_seq=8, max_context_len=100, dtype=0)
    base.update(kw)
    return B.make_shape(**base)


FAKE = 0x10000  # 16-byte aligned non-null address; never dereferenced on the host


def _decode(lib, shape, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, cl=FAKE, out=FAKE, ws=None, wsb=0):
    return lib.pkv_paged_attn_decode(ctypes.byref(shape) if shape is not None else None,
                                     q, kc, vc, bt, cl, 0.1, out, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=6, num_kv_heads=4), -2),          # Hq % Hkv != 0
    (dict(num_kv_heads=0), -2),
    (dict(num_seqs=-1), -2),
    (dict(max_context_len=0), -2),
    (dict(max_context_len=129), -2),                     # > MB * bs
    (dict(split_tokens=-2), -2),
    (dict(split_tokens=-1), -2),                         # no persistent schedule
    (dict(head_dim=96), -3),
    (dict(block_size=8), -3),
    (dict(dtype=5), -3),
    (dict(num_q_heads=66, num_kv_heads=2), -3),          # group of 33 not built
    (dict(num_blocks=1 << 24, num_kv_heads=8, num_q_heads=8), -3),  # rows overflow int32
])
def test_decode_rejects_bad_shapes(lib, kw, code):
    assert _decode(lib, _shape(**kw)) == code


def test_decode_null_and_alignment(lib):
    assert _decode(lib, None) == -1
    assert _decode(lib, _shape(), q=None) == -1
    assert _decode(lib, _shape(), out=None) == -1
    assert _decode(lib, _shape(), q=FAKE + 2) == -4
    assert _decode(lib, _shape(), bt=FAKE + 2) == -4
    # an empty batch is a no-op that never touches the GPU
    assert _decode(lib, _shape(num_seqs=0), q=None) == 0


def test_append_rejects_bad_args(lib):
    s = _shape()
    f = lib.pkv_kv_cache_append
    assert f(None, FAKE, FAKE, FAKE, 1, FAKE, FAKE, None) == -1
    assert f(ctypes.byref(s), None, FAKE, FAKE, 1, FAKE, FAKE, None) == -1
    assert f(ctypes.byref(s), FAKE, FAKE, FAKE, -1, FAKE, FAKE, None) == -2
    assert f(ctypes.byref(s), FAKE + 8, FAKE, FAKE, 1, FAKE, FAKE, None) == -4
    assert f(ctypes.byref(_shape(head_dim=80)), FAKE, FAKE, FAKE, 1, FAKE, FAKE, None) == -3
    assert f(ctypes.byref(s), None, None, None, 0, None, None, None) == 0   # no tokens: no-op
    assert lib.pkv_launch_count() == 0


def test_set_workspace_rejects_bad_args_before_device(lib):
    f = lib.pkv_set_workspace
    assert f(FAKE, 0) == -2                 # a workspace of no bytes
    assert f(FAKE + 4, 4096) == -4          # not 16-byte aligned
    # well-formed calls need the current device, which this host lacks
    assert f(FAKE, 4096) == -6
    assert f(None, 0) == -6


def test_selftest_rejects_bad_limit_before_device(lib):
    assert lib.pkv_selftest_wait_timeout(0, None) == -2
    assert lib.pkv_selftest_wait_timeout(1000001, None) == -2


def test_plan_rejects_before_device(lib):
    p = B.Plan()
    assert lib.pkv_decode_plan(None, ctypes.byref(p)) == -1
    assert lib.pkv_decode_plan(ctypes.byref(_shape(head_dim=48)), ctypes.byref(p)) == -3
    n = ctypes.c_size_t(0)
    assert lib.pkv_workspace_bytes(ctypes.byref(_shape()), None) == -1
    assert lib.pkv_workspace_bytes(ctypes.byref(_shape(num_kv_heads=3)), ctypes.byref(n)) == -2


# ---------------------------------------------------------------- binding extents
# The library sees only pointers and the shape built from the tensors, so the
# binding must reject tensors whose extents disagree before anything launches.
# On the CPU the CUDA-tensor check is lifted to reach the extent checks; a call
# with consistent extents then reaches the library, which finds no device.
def _decode_args(B=2, Hq=8, Hkv=2, D=64, bs=16, NB=8, MB=4):
    import torch
    f16 = torch.float16
    return dict(q=torch.zeros(B, Hq, D, dtype=f16), k_cache=torch.zeros(NB, Hkv, bs, D, dtype=f16),
                v_cache=torch.zeros(NB, Hkv, bs, D, dtype=f16),
                block_tables=torch.zeros(B, MB, dtype=torch.int32),
                context_lens=torch.ones(B, dtype=torch.int32))


@pytest.mark.parametrize("bad", ["q_head_dim", "v_cache", "tables_rows", "lens_len", "out_shape",
                                 "k_new"])
def test_binding_rejects_mismatched_extents(lib, monkeypatch, bad):
    import torch
    monkeypatch.setattr(B, "_dense", lambda *a, **k: None)
    a = _decode_args()
    out = None
    if bad == "q_head_dim":
        a["q"] = torch.zeros(2, 8, 128, dtype=torch.float16)
    elif bad == "v_cache":
        a["v_cache"] = torch.zeros(8, 2, 32, 64, dtype=torch.float16)
    elif bad == "tables_rows":
        a["block_tables"] = torch.zeros(3, 4, dtype=torch.int32)
    elif bad == "lens_len":
        a["context_lens"] = torch.ones(1, dtype=torch.int32)
    elif bad == "out_shape":
        out = torch.zeros(2, 8, 32, dtype=torch.float16)
    k_new = torch.zeros(2, 2, 64 if bad != "k_new" else 32, dtype=torch.float16)
    if bad != "k_new":
        with pytest.raises(ValueError):
            B.paged_attn_decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"],
                                a["context_lens"], 0.125, out, max_context_len=16)
    with pytest.raises(ValueError):
        B.decode_step(a["q"], k_new, k_new.clone(), a["k_cache"], a["v_cache"], a["block_tables"],
                      a["context_lens"], 0.125, out, max_context_len=16)


class _NoDevice:
    """Stands in for torch.cuda.device on a host without CUDA."""

    def __init__(self, dev):
        pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def test_binding_passes_consistent_extents_to_the_library(lib, monkeypatch):
    import torch
    monkeypatch.setattr(B, "_dense", lambda *a, **k: None)
    monkeypatch.setattr(B, "_one_device", lambda **t: torch.device("cuda", 0))
    monkeypatch.setattr(B.torch.cuda, "device", _NoDevice)
    a = _decode_args()
    with pytest.raises(B.PkvError) as e:      # no GPU here: the library reports it
        B.paged_attn_decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"],
                            a["context_lens"], 0.125, max_context_len=16)
    assert e.value.code == -6


# ---------------------------------------------------------------- binding devices
# Every tensor of a call must live on one GPU: the library launches on the
# current device with that device's TMA descriptors, so another GPU's memory
# must never reach it.  The rejection is host logic, checked here with
# stand-ins for CUDA tensors and streams.
class _FakeCuda:
    def __init__(self, index):
        import torch
        self.is_cuda = True
        self.device = torch.device("cuda", index)


def test_one_device_rejects_mixed_and_host_tensors():
    import torch
    assert B._one_device(q=_FakeCuda(1), out=None, k_cache=_FakeCuda(1)) == torch.device("cuda", 1)
    with pytest.raises(ValueError, match="k_cache is on cuda:1"):
        B._one_device(q=_FakeCuda(0), k_cache=_FakeCuda(1))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        B._one_device(q=_FakeCuda(0), block_tables=torch.zeros(2, dtype=torch.int32))


def test_stream_of_another_device_is_rejected():
    import torch

    class S:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    with pytest.raises(ValueError, match="stream is on cuda:1"):
        B._stream_ptr(S(), torch.device("cuda", 0))


def test_every_call_checks_all_its_tensors_for_one_device(lib, monkeypatch):
    import torch
    monkeypatch.setattr(B, "_dense", lambda *a, **k: None)
    seen = {}

    class Stop(Exception):
        pass

    def spy(**tensors):
        seen.update(tensors)
        raise Stop

    monkeypatch.setattr(B, "_one_device", spy)
    a = _decode_args()
    out = torch.zeros_like(a["q"])
    ws = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(Stop):
        B.paged_attn_decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"],
                            a["context_lens"], 0.125, out, max_context_len=16, workspace=ws)
    assert set(seen) == {"q", "k_cache", "v_cache", "block_tables", "context_lens", "out",
                         "workspace"}
    seen.clear()
    k_new = torch.zeros(2, 2, 64, dtype=torch.float16)
    with pytest.raises(Stop):
        B.decode_step(a["q"], k_new, k_new.clone(), a["k_cache"], a["v_cache"],
                      a["block_tables"], a["context_lens"], 0.125, out, max_context_len=16,
                      workspace=ws)
    assert set(seen) == {"q", "k_new", "v_new", "k_cache", "v_cache", "block_tables",
                         "context_lens", "out", "workspace"}
    seen.clear()
    with pytest.raises(Stop):
        B.kv_cache_append(k_new, k_new.clone(), torch.zeros(2, dtype=torch.int32),
                          a["k_cache"][:, :, :, :], a["v_cache"])
    assert set(seen) == {"k", "v", "slot_mapping", "k_cache", "v_cache"}

"""Guard regions (GPU, through the C ABI): a decode call writes only its out
rows, at most pkv_plan.workspace_bytes of workspace and, for the fused step,
only slots inside the cache pools.  Each of those buffers sits inside a larger
allocation whose margins hold a canary pattern that must survive the call."""
from __future__ import annotations

import pytest
import torch

from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, oracle_decode, widen_out

pytestmark = pytest.mark.gpu

CANARY16 = 0x5A5A          # 16-bit pattern around out and the caches
CANARY8 = 0xA5             # byte pattern around the workspace
PAD = 4096                 # elements (8 KB of 16-bit values) on each side
WPAD = 4096                # bytes on each side of the workspace

SMALL = {
    "tiny_mha": W.WORKLOADS["tiny_mha"],
    "llama7b_mha": W.scaled(W.WORKLOADS["llama7b_mha"], 6, 1300),
    "llama3_8b_gqa": W.scaled(W.WORKLOADS["llama3_8b_gqa"], 8, 1500, min_len=16),
    "long_ctx_gqa": W.scaled(W.WORKLOADS["long_ctx_gqa"], 2, 2600, lens="fixed"),
    "cont_batch": W.scaled(W.WORKLOADS["cont_batch"], 16, 700),
}


def _guarded(like: torch.Tensor):
    """A tensor shaped like `like` inside a canary-filled allocation, and the
    allocation."""
    n = like.numel()
    buf = torch.empty(n + 2 * PAD, dtype=like.dtype, device=like.device)
    buf.view(torch.int16).fill_(CANARY16)
    t = buf[PAD:PAD + n].view(like.shape)
    return t, buf


def _margins_intact(buf: torch.Tensor, n: int) -> bool:
    b = buf.view(torch.int16)
    return bool(torch.all(b[:PAD] == CANARY16)) and bool(torch.all(b[PAD + n:] == CANARY16))


@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", W.ORDER)
def test_writes_stay_inside_their_buffers(pkv, name, fused, kernel):
    w = W.make(SMALL[name], seed=5)
    if kernel == 3 and w.spec.head_dim != 128:
        pytest.skip("the tcgen05 kernel is built for head_dim 128")
    if kernel == 3 and fused and w.spec.dtype != W.BF16:
        pytest.skip("the tcgen05 fused step is covered for bfloat16 caches")
    d = device_inputs(w)
    q = d["q"]
    out, obuf = _guarded(q)
    shape = pkv.decode_shape(q, d["k_cache"], d["block_tables"], w.max_context_len, 0, kernel)
    nbytes = pkv.workspace_bytes(shape)
    wbuf = torch.full((nbytes + 2 * WPAD,), CANARY8, dtype=torch.uint8, device=q.device)
    ws = wbuf[WPAD:WPAD + nbytes] if nbytes else None
    if fused:
        kc, kbuf = _guarded(d["k_cache"])
        vc, vbuf = _guarded(d["v_cache"])
        kc.copy_(d["k_cache"])
        vc.copy_(d["v_cache"])
        pkv.decode_step(q, w.k_new.cuda(), w.v_new.cuda(), kc, vc, d["block_tables"],
                        d["context_lens"], w.scale, out, max_context_len=w.max_context_len,
                        kernel=kernel, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert _margins_intact(kbuf, kc.numel()) and _margins_intact(vbuf, vc.numel())
        # the fused step equals append-then-decode bit for bit
        ref = pkv.paged_attn_decode(q, kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                    max_context_len=w.max_context_len, kernel=kernel)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    else:
        pkv.paged_attn_decode(q, d["k_cache"], d["v_cache"], d["block_tables"],
                              d["context_lens"], w.scale, out, max_context_len=w.max_context_len,
                              kernel=kernel, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), oracle_decode(w), f"{name} kernel {kernel}")
    assert _margins_intact(obuf, q.numel())
    if nbytes:
        assert bool(torch.all(wbuf[:WPAD] == CANARY8))
        assert bool(torch.all(wbuf[WPAD + nbytes:] == CANARY8))

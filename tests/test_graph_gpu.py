"""The decode path inside a CUDA graph: capture decode_step (append fused)
and paged_attn_decode, replay, and compare bit for bit with eager calls.
Host-side planning, descriptor encoding and kernel attributes happen at
capture time; the first (eager) call sets the kernels up."""
from __future__ import annotations

import pytest
import torch

from paged_kv_cache_268_gb300 import workloads as W
from parity import device_inputs
from test_decode_gpu import SMALL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("name", ["llama7b_mha", "llama3_8b_gqa", "long_ctx_gqa"])
def test_graph_replay_matches_eager(pkv, name, kernel):
    """kernel 0: the library's choice; 3: the tcgen05 kernel (its own
    programmatic launch and fused append inside the graph)."""
    w = W.make(SMALL[name], seed=3)
    d = device_inputs(w)
    kn, vn = w.k_new.cuda(), w.v_new.cuda()
    shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], w.max_context_len, 0,
                             kernel)
    ws = pkv.alloc_workspace(shape)

    def step(kc, vc, out, out2):
        pkv.decode_step(d["q"], kn, vn, kc, vc, d["block_tables"], d["context_lens"], w.scale,
                        out, max_context_len=w.max_context_len, kernel=kernel, workspace=ws)
        pkv.paged_attn_decode(d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                              out2, max_context_len=w.max_context_len, kernel=kernel,
                              workspace=ws)

    kc_e, vc_e = d["k_cache"].clone(), d["v_cache"].clone()
    o_e, o2_e = torch.empty_like(d["q"]), torch.empty_like(d["q"])
    step(kc_e, vc_e, o_e, o2_e)                     # eager (also sets the kernels up)
    torch.cuda.synchronize()

    kc_g, vc_g = d["k_cache"].clone(), d["v_cache"].clone()
    o_g, o2_g = torch.full_like(d["q"], float("nan")), torch.full_like(d["q"], float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(kc_g, vc_g, o_g, o2_g)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    same = lambda a, b: torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert same(o_g, o_e) and same(o2_g, o2_e)
    assert same(kc_g, kc_e) and same(vc_g, vc_e)

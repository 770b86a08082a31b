"""A multi-layer decode step (fused append + decode per layer) captured in a
CUDA graph replays bit-identically to eager execution.  The library's first
call on a device caches device properties, so it runs once before capture."""
import pytest
import torch

import workloads
from tests.gpu_fill import fill_gpu, step_tokens

pytestmark = pytest.mark.gpu


def test_graph_captured_layer_loop_matches_eager(pkv, cuda_device):
    wl = workloads.Workload(80, "graph", [500, 37, 1200, 64], 1, 16, 4, 16, seed=12)
    layers = []
    for layer in range(3):
        f = fill_gpu(wl, layer, cuda_device, step_append=False)
        k, v = step_tokens(wl, layer, cuda_device)
        layers.append((f, k, v))
    n = pkv.pkv_decode_workspace_size(wl.batch, wl.hq, wl.hkv, 128, wl.max_pages * wl.page_size, wl.page_size)
    ws = torch.zeros(n, dtype=torch.uint8, device=cuda_device)
    outs = [torch.empty(wl.batch, wl.hq, 128, dtype=torch.bfloat16, device=cuda_device) for _ in layers]

    def step():
        for (f, k, v), o in zip(layers, outs):
            pkv.pkv_append_decode_fp8(k, v, f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, o, ws)

    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for o, e in zip(outs, eager):
            assert torch.equal(o, e)

"""The allocation-free decode entry point, for callers that may not call
cudaMalloc (an engine that owns all device memory through its own pool, a
plugin that must not bypass its host runtime's allocator, a latency-critical
loop).  It keeps its split-K scratch in a fixed array inside the library; this
checks, through the C ABI, that it returns what pkv_paged_gqa_decode returns
with a caller workspace, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result)."""
import pytest
import torch

import workloads
from tests.gpu_fill import assert_close, fill_gpu

pytestmark = pytest.mark.gpu


def _ref(pkv, f, out_dtype):
    wl = f.wl
    n = pkv.pkv_decode_workspace_size(wl.batch, wl.hq, wl.hkv, 128, wl.max_pages * wl.page_size, wl.page_size)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=f.q.device)
    out = torch.empty(f.q.shape, dtype=out_dtype, device=f.q.device)
    pkv.pkv_paged_gqa_decode(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out, ws)
    return out


def _noalloc(pkv, f, out_dtype):
    out = torch.empty(f.q.shape, dtype=out_dtype, device=f.q.device)
    pkv.pkv_paged_gqa_decode_noalloc(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out)
    return out


def test_noalloc_matches_workspace_entry_point_twice(pkv, cuda_device):
    assert pkv.pkv_decode_noalloc_scratch_bytes() == 16 << 20
    # two different workloads back to back: the second call runs on scratch
    # that still holds the first call's partial states
    for cfg, page in [(1, 16), (0, 32), (1, 16)]:
        wl = workloads.config(cfg, page_size=page)
        f = fill_gpu(wl, 0, cuda_device)
        for _ in range(2):
            ref = _ref(pkv, f, torch.float32)
            got = _noalloc(pkv, f, torch.float32)
            torch.cuda.synchronize()
            assert_close(got.double().cpu().numpy(), ref.double().cpu().numpy(), f"config {cfg}")
            assert torch.equal(got, ref)        # same kernels, same split: identical bits
        assert torch.equal(_noalloc(pkv, f, torch.bfloat16), _ref(pkv, f, torch.bfloat16))


def test_noalloc_rejects_sizes_beyond_its_scratch(pkv, cuda_device):
    B, Hq, Hkv = 4096, 64, 8                  # 32768 segments: far more partial slots than fit
    q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device=cuda_device)
    kc = torch.zeros(1, Hkv, 16, 128, dtype=torch.uint8, device=cuda_device)
    s = torch.ones(Hkv, device=cuda_device)
    bt = torch.zeros(B, 1, dtype=torch.int32, device=cuda_device)
    lens = torch.ones(B, dtype=torch.int32, device=cuda_device)
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_gqa_decode_noalloc(q, kc, kc, s, s, bt, lens, out)
    assert e.value.status == 5                # PKV_ERR_WORKSPACE

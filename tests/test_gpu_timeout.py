"""Failure detection on the GPU without a fault: a decode worker is told
(test facility pkv_test_withhold_load) never to load its first page, so its
bounded pipeline wait runs out; the kernel must report PKV_DEVERR_TIMEOUT,
drain, return within seconds, and leave the context usable."""
import time

import pytest
import torch

import workloads
from tests.gpu_fill import assert_close, fill_gpu
from tests.test_gpu_decode import _full_oracle

pytestmark = pytest.mark.gpu


def test_withheld_load_times_out_and_context_survives(pkv, cuda_device):
    wl = workloads.Workload(70, "timeout", [300, 77], 0, 8, 2, 16, seed=4)
    f = fill_gpu(wl, 0, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.pkv_test_withhold_load(0)
    try:
        t0 = time.time()
        pkv.paged_gqa_decode(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out_dtype=torch.float32,
                             device_error=err, max_ctas=4)
        torch.cuda.synchronize()
        dt = time.time() - t0
    finally:
        pkv.pkv_test_withhold_load(-1)
    assert int(err.item()) & pkv.DEVERR_TIMEOUT
    assert 1.5 < dt < 20.0
    err.zero_()
    out = pkv.paged_gqa_decode(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out_dtype=torch.float32,
                               device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.double().cpu().numpy(), _full_oracle(wl, f), "after timeout")


def test_prefill_withheld_tile_times_out_and_context_survives(pkv, cuda_device):
    """Prefill CTA 0 (the heaviest query tile) never gets its first K tile: its
    MMA warp's wait runs out, every role drains its own copies and MMAs, TMEM
    is freed, the call reports PKV_DEVERR_TIMEOUT, and the next call is exact."""
    from tests.test_gpu_prefill import _oracle_pools
    import numpy as np
    import oracle
    wl = workloads.Workload(71, "prefill-timeout", [400], 0, 8, 1, 16, seed=5)
    f = fill_gpu(wl, 0, cuda_device)
    q = wl.q_rows(0, 40)
    cu = torch.tensor([0, 40], dtype=torch.int32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.pkv_test_withhold_load(0)
    try:
        t0 = time.time()
        pkv.paged_prefill(q.to(cuda_device), cu, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, 40,
                          out_dtype=torch.float32, device_error=err)
        torch.cuda.synchronize()
        dt = time.time() - t0
    finally:
        pkv.pkv_test_withhold_load(-1)
    assert int(err.item()) & pkv.DEVERR_TIMEOUT
    assert 1.5 < dt < 20.0
    err.zero_()
    out = pkv.paged_prefill(q.to(cuda_device), cu, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, 40,
                            out_dtype=torch.float32, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kco, vco, ks, vs = _oracle_pools(wl)
    ref = oracle.paged_prefill(q.view(torch.uint16).numpy(), np.array([0, 40], np.int32), kco, vco, ks, vs,
                               wl.block_table().numpy(), np.array(wl.seq_lens, np.int32), threads=8)
    assert_close(out.double().cpu().numpy(), ref, "prefill after timeout")

"""pkv_kv_calibrate on the GPU against the oracle: running maxima and scales
bit-exact (a maximum is exact; the division is IEEE)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def test_batches_fold_into_running_max(pkv, cuda_device):
    g = torch.Generator().manual_seed(7)
    rk = torch.zeros(8, device=cuda_device)
    rv = torch.zeros(8, device=cuda_device)
    ks = torch.empty(8, device=cuda_device)
    vs = torch.empty(8, device=cuda_device)
    ork = np.zeros(8, np.float32)
    orv = np.zeros(8, np.float32)
    for T in (1, 37, 1000, 5000):
        k = torch.randn(T, 8, 128, generator=g) * torch.rand(1, 8, 1, generator=g) * 30
        v = torch.randn(T, 8, 128, generator=g) * 3
        if T == 37:
            k[3, 2, 9] = float("nan")
        pkv.pkv_kv_calibrate(k.to(cuda_device), v.to(cuda_device), rk, rv, ks, vs)
        oracle.kv_absmax_update(k.numpy(), ork)
        oracle.kv_absmax_update(v.numpy(), orv)
    torch.cuda.synchronize()
    assert np.array_equal(rk.cpu().numpy(), ork) and np.array_equal(rv.cpu().numpy(), orv)
    assert np.array_equal(ks.cpu().numpy(), oracle.kv_scale_from_max(ork))
    assert np.array_equal(vs.cpu().numpy(), oracle.kv_scale_from_max(orv))


def test_bf16_and_empty_batch(pkv, cuda_device):
    x = (torch.randn(64, 2, 128) * 11).to(torch.bfloat16)
    rk = torch.zeros(2, device=cuda_device)
    rv = torch.full((2,), 5.0, device=cuda_device)
    pkv.pkv_kv_calibrate(x.to(cuda_device), x.to(cuda_device), rk, rv)
    empty = torch.zeros(0, 2, 128, device=cuda_device)
    ks = torch.empty(2, device=cuda_device)
    vs = torch.empty(2, device=cuda_device)
    pkv.pkv_kv_calibrate(empty, empty, rk, rv, ks, vs)
    torch.cuda.synchronize()
    o = np.zeros(2, np.float32)
    oracle.kv_absmax_update(x.view(torch.uint16).numpy(), o)
    assert np.array_equal(rk.cpu().numpy(), o)
    assert np.array_equal(rv.cpu().numpy(), np.maximum(o, 5.0))
    assert np.array_equal(ks.cpu().numpy(), oracle.kv_scale_from_max(o))


def test_prefill_calibration_reproduces_workload_scales(pkv, cuda_device):
    """Calibrating over the 8B-layer workload's prefill gives the scales the
    workload recipe states (absmax / 448 over the prefill tokens)."""
    wl = workloads.config(1)
    rk = torch.zeros(wl.hkv, device=cuda_device)
    rv = torch.zeros(wl.hkv, device=cuda_device)
    ks = torch.empty(wl.hkv, device=cuda_device)
    vs = torch.empty(wl.hkv, device=cuda_device)
    for b, L in enumerate(wl.prefill_lens):
        pkv.pkv_kv_calibrate(wl.kv_rows(0, 0, b, 0, L, device=cuda_device),
                             wl.kv_rows(0, 1, b, 0, L, device=cuda_device), rk, rv, ks, vs)
    ek, ev = wl.scales(0, device=cuda_device)
    torch.cuda.synchronize()
    assert torch.equal(ks, ek) and torch.equal(vs, ev)

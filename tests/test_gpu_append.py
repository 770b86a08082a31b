"""kv_append_fp8 on the GPU against the oracle: bit-exact page bytes."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_fill import fill_gpu, oracle_pages

pytestmark = pytest.mark.gpu
THREADS = max(1, min(32, len(os.sched_getaffinity(0))))


def _encode_on_gpu(pkv, y: torch.Tensor, scale: float, dev) -> np.ndarray:
    """Codes the kernel writes for the fp32 values y (length multiple of 2048)."""
    n = y.numel()
    T = n // 128
    x = y.view(T, 1, 128)
    slots = torch.arange(T, dtype=torch.int64, device=dev)
    s = torch.tensor([scale], dtype=torch.float32, device=dev)
    kc = torch.empty((T // 16, 1, 16, 128), dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    pkv.kv_append_fp8(x, x, slots, s, s, kc, vc)
    assert torch.equal(kc, vc)
    return kc.view(-1).cpu().numpy()


def _compare_codes(y_cpu: np.ndarray, got: np.ndarray, exp: np.ndarray):
    nan = np.isnan(y_cpu)
    assert np.array_equal(got[~nan], exp[~nan])
    assert np.all((got[nan] & 0x7F) == 0x7F)          # any NaN code for NaN input


def test_exhaustive_fp32_sweep(pkv, cuda_device):
    """All 2^32 fp32 bit patterns, scale 1: kernel codes == oracle codes."""
    chunk = 1 << 27
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device=cuda_device)
        y = torch.where(bits >= 1 << 31, bits - (1 << 32), bits).to(torch.int32).view(torch.float32)
        got = _encode_on_gpu(pkv, y, 1.0, cuda_device)
        y_cpu = y.cpu().numpy()
        exp = oracle.e4m3_encode(y_cpu, threads=THREADS)
        _compare_codes(y_cpu, got, exp)


def test_random_scales_division(pkv, cuda_device):
    """1M values with random scales: the division must be IEEE x / s."""
    g = torch.Generator().manual_seed(11)
    n = 1 << 20
    for trial in range(8):
        scale = float(torch.rand(1, generator=g) * 3 + 1e-3)
        y = (torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 3)).float()
        got = _encode_on_gpu(pkv, y.to(cuda_device), scale, cuda_device)
        s32 = np.float32(scale)
        exp = oracle.e4m3_encode((y.numpy() / s32).astype(np.float32), threads=THREADS)
        assert np.array_equal(got, exp), trial


def test_bf16_inputs(pkv, cuda_device):
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 4, 128, generator=g) * 20).to(torch.bfloat16)
    slots = torch.randperm(8 * 16, generator=g)[:64].to(torch.int64)
    scale = torch.tensor([0.05, 0.3, 1.0, 7.0])
    kc = torch.zeros((8, 4, 16, 128), dtype=torch.uint8, device=cuda_device)
    vc = torch.zeros_like(kc)
    pkv.kv_append_fp8(x.to(cuda_device), x.to(cuda_device), slots.to(cuda_device), scale.to(cuda_device),
                      scale.to(cuda_device), kc, vc)
    ref = np.zeros((8, 4, 16, 128), np.uint8)
    oracle.kv_append(x.view(torch.uint16).numpy(), slots.numpy(), scale.numpy(), ref)
    assert np.array_equal(kc.cpu().numpy(), ref)


def test_skipped_and_out_of_pool_slots(pkv, cuda_device):
    x = torch.ones(4, 2, 128, device=cuda_device)
    slots = torch.tensor([-1, 3, 64, 1 << 40], dtype=torch.int64, device=cuda_device)
    s = torch.ones(2, device=cuda_device)
    kc = torch.full((4, 2, 16, 128), 0xAB, dtype=torch.uint8, device=cuda_device)
    vc = torch.full_like(kc, 0xAB)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.kv_append_fp8(x, x, slots, s, s, kc, vc, err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEVERR_SLOT
    ref = np.full((4, 2, 16, 128), 0xAB, np.uint8)
    oracle.kv_append(np.ones((4, 2, 128), np.float32), slots.cpu().numpy(), np.ones(2, np.float32), ref)
    assert np.array_equal(kc.cpu().numpy(), ref)


def test_empty_append_is_noop(pkv, cuda_device):
    x = torch.zeros(0, 2, 128, device=cuda_device)
    kc = torch.zeros((1, 2, 16, 128), dtype=torch.uint8, device=cuda_device)
    pkv.kv_append_fp8(x, x, torch.zeros(0, dtype=torch.int64, device=cuda_device), torch.ones(2, device=cuda_device),
                      torch.ones(2, device=cuda_device), kc, kc.clone())
    assert int(kc.sum()) == 0


@pytest.mark.parametrize("cfg,page", [(0, 16), (1, 16), (0, 32), (1, 32), (0, 64), (0, 256)])
def test_pages_bit_exact_small_configs(pkv, cuda_device, cfg, page):
    wl = workloads.config(cfg, page_size=page)
    f = fill_gpu(wl, 0, cuda_device, tail_fill=0)
    assert int(f.err.item()) == 0
    ks, vs = wl.scales(0)
    assert torch.equal(ks, f.ks.cpu()) and torch.equal(vs, f.vs.cpu())     # generator: same on both devices
    ref_k = np.zeros(tuple(f.kc.shape), np.uint8)
    ref_v = np.zeros_like(ref_k)
    for b, L in enumerate(wl.seq_lens):
        slots = wl.slots(b, 0, L).numpy()
        oracle.kv_append(wl.kv_rows(0, 0, b, 0, L).numpy(), slots, ks.numpy(), ref_k)
        oracle.kv_append(wl.kv_rows(0, 1, b, 0, L).numpy(), slots, vs.numpy(), ref_v)
    assert np.array_equal(f.kc.cpu().numpy(), ref_k)
    assert np.array_equal(f.vc.cpu().numpy(), ref_v)


@pytest.mark.parametrize("cfg,page", [(2, 16), (3, 16), (4, 16), (4, 32)])
def test_pages_bit_exact_large_configs_sampled(pkv, cuda_device, cfg, page):
    """Full-size caches; the pages of sampled (sequence, kv head) pairs are
    compared with oracle pages built from host-generated inputs."""
    wl = workloads.config(cfg, page_size=page)
    f = fill_gpu(wl, 0, cuda_device)
    assert int(f.err.item()) == 0
    ks, vs = f.ks.cpu().numpy(), f.vs.cpu().numpy()
    bt = wl.block_table()
    for b, h in [(0, 0), (wl.batch - 1, wl.hkv - 1), (wl.batch // 2, 3)]:
        kc_o, vc_o = oracle_pages(wl, 0, b, h, float(ks[h]), float(vs[h]))
        pages = bt[b, :wl.pages_per_seq[b]].long()
        L = wl.seq_lens[b]
        P = wl.page_size
        got_k = f.kc[pages.to(cuda_device), h].cpu().numpy().reshape(-1, 128)[:L]
        got_v = f.vc[pages.to(cuda_device), h].cpu().numpy().reshape(-1, 128)[:L]
        exp_k = kc_o[pages.numpy(), 0].reshape(-1, 128)[:L]
        exp_v = vc_o[pages.numpy(), 0].reshape(-1, 128)[:L]
        assert np.array_equal(got_k, exp_k), (b, h)
        assert np.array_equal(got_v, exp_v), (b, h)
        assert P * len(pages) >= L
    del f
    torch.cuda.empty_cache()

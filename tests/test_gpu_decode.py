"""paged_gqa_decode on the GPU against the fp64 oracle.

Tolerance (fp32 output mode): max-abs <= 2e-3 and relative L2 <= 1e-3 of
the oracle's fp64 attention over the same dequantised cache.  The bf16
output must equal the round-to-nearest-even bf16 of the fp32 output bit for
bit, and lie within one bf16 ulp of the oracle rounded to bf16.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_fill import (assert_close, bf16_ulp, fill_gpu, oracle_rows, sample_pairs)

pytestmark = pytest.mark.gpu


def _poisoned_workspace(pkv, f, max_ctas):
    """A workspace full of NaN bytes: reading a slot nobody wrote shows up."""
    wl = f.wl
    n = pkv.pkv_decode_workspace_size(wl.batch, wl.hq, wl.hkv, 128, wl.page_size, max_ctas)
    return torch.full((n,), 0xFF, dtype=torch.uint8, device=f.q.device)


def _decode(pkv, f, out_dtype=torch.float32, max_ctas=0, err=None, bt=None, lens=None, kc=None, vc=None):
    out = pkv.paged_gqa_decode(f.q, f.kc if kc is None else kc, f.vc if vc is None else vc, f.ks, f.vs,
                               f.bt if bt is None else bt, f.lens if lens is None else lens,
                               out_dtype=out_dtype, device_error=err if err is not None else f.err,
                               max_ctas=max_ctas, workspace=_poisoned_workspace(pkv, f, max_ctas))
    torch.cuda.synchronize()
    return out


def _full_oracle(wl, f):
    kc = f.kc.cpu().numpy() * 0   # shapes only; oracle pools are rebuilt from host inputs
    ks, vs = wl.scales(0)
    kco = np.zeros(kc.shape, np.uint8)
    vco = np.zeros(kc.shape, np.uint8)
    for b, L in enumerate(wl.seq_lens):
        slots = wl.slots(b, 0, L).numpy()
        oracle.kv_append(wl.kv_rows(0, 0, b, 0, L).numpy(), slots, ks.numpy(), kco)
        oracle.kv_append(wl.kv_rows(0, 1, b, 0, L).numpy(), slots, vs.numpy(), vco)
    ref = oracle.paged_decode(wl.q().view(torch.uint16).numpy(), kco, vco, ks.numpy(), vs.numpy(),
                              wl.block_table().numpy(), np.array(wl.seq_lens, np.int32), threads=8)
    return ref.reshape(wl.batch, wl.hq, wl.head_dim)


@pytest.mark.parametrize("page", [16, 32, 64, 256])
def test_tiny_config_all_rows(pkv, cuda_device, page):
    wl = workloads.config(0, page_size=page)
    f = fill_gpu(wl, 0, cuda_device)
    got = _decode(pkv, f).double().cpu().numpy()
    assert int(f.err.item()) == 0
    ref = _full_oracle(wl, f)
    assert_close(got, ref, "tiny fp32")
    # bf16 output == RNE(fp32 output), and within 1 bf16 ulp of the oracle
    got32 = _decode(pkv, f)
    got16 = _decode(pkv, f, out_dtype=torch.bfloat16)
    assert torch.equal(got16, got32.to(torch.bfloat16))
    ref16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert np.all(np.abs(got16.double().cpu().numpy() - ref16) <= bf16_ulp(ref) * 1.0001)


@pytest.mark.parametrize("lens,hq,hkv,page", [
    ([1, 2, 15, 16, 17, 31, 33], 8, 1, 16),
    ([0, 5, 0, 300], 16, 2, 16),              # empty sequences give zero rows
    ([1, 100, 257, 64], 4, 4, 32),
    ([1000, 3, 47], 32, 8, 16),               # G = 4
    ([513, 2049], 2, 2, 32),                  # G = 1
    ([77, 1], 16, 8, 16),                     # G = 2
    ([4097, 1, 999], 64, 8, 32),
    ([1, 63, 64, 65, 200], 8, 2, 64),         # 64-token pages (chunks of 16 inside a page)
    ([129, 1000, 5], 16, 2, 128),
    ([255, 256, 257, 3000], 64, 8, 256),      # 256-token pages
])
def test_ragged_shapes(pkv, cuda_device, lens, hq, hkv, page):
    wl = workloads.Workload(50, "ragged", lens, 0, hq, hkv, page, pool_factor=1.5, seed=21)
    f = fill_gpu(wl, 0, cuda_device)
    ref = _full_oracle(wl, f)
    for ctas in (0, 1, 3, 7):
        got = _decode(pkv, f, max_ctas=ctas).double().cpu().numpy()
        assert int(f.err.item()) == 0
        assert_close(got, ref, f"ctas={ctas}")
        for b, L in enumerate(wl.seq_lens):
            if L == 0:
                assert np.all(got[b] == 0)


def test_deterministic_and_page_permutation_invariant(pkv, cuda_device):
    wl = workloads.Workload(51, "perm", [700, 33, 1601, 16], 0, 16, 2, 16, pool_factor=2.0, seed=5)
    f = fill_gpu(wl, 0, cuda_device)
    a = _decode(pkv, f)
    b = _decode(pkv, f)
    assert torch.equal(a, b)                                   # run to run
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(wl.num_pages, generator=g).to(cuda_device)   # page p moves to perm[p]
    kc2 = torch.empty_like(f.kc)
    vc2 = torch.empty_like(f.vc)
    kc2[perm] = f.kc
    vc2[perm] = f.vc
    bt2 = torch.where(f.bt >= 0, perm[f.bt.clamp(min=0).long()].to(torch.int32), f.bt)
    c = _decode(pkv, f, bt=bt2, kc=kc2, vc=vc2)
    assert torch.equal(a, c)                                   # bit-identical


def test_tail_garbage_does_not_matter(pkv, cuda_device):
    """Unused rows of the last page filled with NaN codes (0x7F) or zeros give
    bit-identical output."""
    wl = workloads.Workload(52, "tail", [37, 100, 5, 250], 0, 8, 1, 16, seed=8)
    fa = fill_gpu(wl, 0, cuda_device, tail_fill=0x7F)
    fb = fill_gpu(wl, 0, cuda_device, tail_fill=0x00)
    assert torch.equal(_decode(pkv, fa), _decode(pkv, fb))
    assert not torch.isnan(_decode(pkv, fa)).any()


def test_closed_forms(pkv, cuda_device):
    """V = 1 everywhere gives o = 1; one-token contexts give dequant(V) exactly."""
    dev = cuda_device
    B, Hq, Hkv, P, L = 3, 16, 2, 16, 333
    npg = (L + P - 1) // P
    kc = torch.randint(0, 256, (B * npg, Hkv, P, 128), dtype=torch.uint8, device=dev)
    kc[(kc & 0x7F) == 0x7F] = 0x30
    vc = torch.full_like(kc, 0x38)                             # E4M3 1.0
    bt = torch.arange(B * npg, dtype=torch.int32, device=dev).view(B, npg)
    q = torch.randn(B, Hq, 128, device=dev).to(torch.bfloat16)
    ks = torch.tensor([0.01, 0.02], device=dev)
    vs = torch.ones(2, device=dev)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    out = pkv.paged_gqa_decode(q, kc, vc, ks, vs, bt, lens, out_dtype=torch.float32)
    assert torch.allclose(out, torch.ones_like(out), rtol=0, atol=1e-5)
    # one-token contexts
    vc = torch.randint(0, 256, kc.shape, dtype=torch.uint8, device=dev)
    vc[(vc & 0x7F) == 0x7F] = 0x41
    vs = torch.tensor([0.3, 1.7], device=dev)
    lens = torch.ones(B, dtype=torch.int32, device=dev)
    out = pkv.paged_gqa_decode(q, kc, vc, ks, vs, bt, lens, out_dtype=torch.float32)
    v0 = vc[bt[:, 0].long()][:, :, 0, :].cpu()                 # [B, Hkv, 128] codes of token 0
    vals = torch.from_numpy(oracle.e4m3_value(v0.numpy())).float() * vs.cpu().view(1, 2, 1)
    exp = vals.repeat_interleave(Hq // Hkv, dim=1)
    assert torch.equal(out.cpu(), exp)


def test_device_errors_without_faults(pkv, cuda_device):
    wl = workloads.Workload(53, "err", [40, 70], 0, 8, 2, 16, seed=1)
    f = fill_gpu(wl, 0, cuda_device)
    bt = f.bt.clone()
    bt[1, 2] = wl.num_pages + 5                               # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    _decode(pkv, f, err=err, bt=bt)
    assert int(err.item()) & pkv.DEVERR_PAGE
    err.zero_()
    lens = f.lens.clone()
    lens[0] = bt.shape[1] * wl.page_size + 100                 # beyond the table
    _decode(pkv, f, err=err, lens=lens)
    assert int(err.item()) & pkv.DEVERR_SEQLEN
    err.zero_()
    out = _decode(pkv, f, err=err)                             # and a clean call afterwards
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()


@pytest.mark.parametrize("cfg,page,n_bh", [(1, 16, 6), (2, 16, 5), (3, 16, 3), (4, 16, 4), (4, 32, 4),
                                           (2, 64, 3), (4, 256, 3)])
def test_full_size_configs_sampled(pkv, cuda_device, cfg, page, n_bh):
    """Full-size workloads in the benchmark's launch configuration; sampled
    (sequence, kv head) groups checked against the oracle."""
    wl = workloads.config(cfg, page_size=page)
    f = fill_gpu(wl, 0, cuda_device)
    got32 = _decode(pkv, f)
    got16 = _decode(pkv, f, out_dtype=torch.bfloat16)
    assert int(f.err.item()) == 0
    assert torch.equal(got16, got32.to(torch.bfloat16))
    pairs = sample_pairs(wl, n_bh, seed=cfg)
    exp = oracle_rows(wl, 0, pairs, f.ks.cpu().numpy(), f.vs.cpu().numpy())
    got = got32.double().cpu().numpy()
    g = np.stack([got[b, i] for (b, i) in pairs])
    r = np.stack([exp[p] for p in pairs])
    assert_close(g, r, f"config {cfg} P={page}")
    del f
    torch.cuda.empty_cache()

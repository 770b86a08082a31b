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
    n = pkv.pkv_decode_workspace_size(wl.batch, wl.hq, wl.hkv, 128, f.max_len, wl.page_size, max_ctas)
    return torch.full((n,), 0xFF, dtype=torch.uint8, device=f.q.device)


def _decode(pkv, f, out_dtype=torch.float32, max_ctas=0, err=None, bt=None, lens=None, kc=None, vc=None,
            psz=None):
    out = pkv.paged_gqa_decode(f.q, f.kc if kc is None else kc, f.vc if vc is None else vc, f.ks, f.vs,
                               f.bt if bt is None else bt, f.lens if lens is None else lens,
                               out_dtype=out_dtype, device_error=err if err is not None else f.err,
                               max_ctas=max_ctas, workspace=_poisoned_workspace(pkv, f, max_ctas),
                               max_seq_len=f.max_len, seq_page_sizes=f.psz if psz is None else psz)
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
    psz = np.array(wl.page_sizes, np.int32) if wl.page_sizes is not None else None
    ref = oracle.paged_decode(wl.q().view(torch.uint16).numpy(), kco, vco, ks.numpy(), vs.numpy(),
                              wl.block_table().numpy(), np.array(wl.seq_lens, np.int32), threads=8,
                              seq_page_sizes=psz)
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


@pytest.mark.parametrize("cfg,page,n_bh,layer,dyn", [
    (1, 16, 6, 0, False), (2, 16, 5, 0, False), (3, 16, 3, 0, False), (4, 16, 4, 0, False),
    (4, 16, 3, 40, False), (4, 16, 3, 79, False), (4, 32, 4, 0, False), (2, 64, 3, 0, False),
    (4, 256, 3, 0, False), (4, 16, 4, 0, True), (4, 16, 3, 79, True)])
def test_full_size_configs_sampled(pkv, cuda_device, cfg, page, n_bh, layer, dyn):
    """Full-size workloads in the benchmark's launch configuration (for the
    mixed batch also layers 40 and 79, and 64-token pages above 8192 tokens);
    sampled (sequence, kv head) groups checked against the oracle, the bf16
    output also within one bf16 ulp of the oracle."""
    wl = workloads.config(cfg, page_size=page, dynamic_pages=dyn)
    f = fill_gpu(wl, layer, cuda_device)
    got32 = _decode(pkv, f)
    got16 = _decode(pkv, f, out_dtype=torch.bfloat16)
    assert int(f.err.item()) == 0
    assert torch.equal(got16, got32.to(torch.bfloat16))
    pairs = sample_pairs(wl, n_bh, seed=cfg + layer)
    exp = oracle_rows(wl, layer, pairs, f.ks.cpu().numpy(), f.vs.cpu().numpy())
    got = got32.double().cpu().numpy()
    g = np.stack([got[b, i] for (b, i) in pairs])
    r = np.stack([exp[p] for p in pairs])
    assert_close(g, r, f"config {cfg} P={page} layer {layer}")
    # within one bf16 ulp of the oracle rounded to bf16 wherever that ulp
    # (>= 2^-12 for |o| >= 2^-4) is well above the fp32-mode error; nearer to
    # zero the absolute tolerance governs (an ulp there can be smaller than
    # the fp32 rounding of a long accumulation)
    g16 = got16.double().cpu().numpy()
    g16 = np.stack([g16[b, i] for (b, i) in pairs])
    r16 = torch.from_numpy(r).to(torch.bfloat16).double().numpy()
    big = np.abs(r) >= 2.0 ** -4
    assert big.any()
    assert np.all(np.abs(g16 - r16)[big] <= bf16_ulp(r)[big] * 1.0001)
    assert np.abs(g16 - r).max() <= 2e-3 + 0.5 * bf16_ulp(r).max()
    del f
    torch.cuda.empty_cache()


@pytest.mark.parametrize("lens,hq,hkv,page,ctas", [
    ([8200, 8200, 3000, 9000], 16, 2, 16, 1),     # about 890 chunks per worker: 6 folds
    ([16384] * 4, 8, 2, 32, 1),                  # 2048 chunks per worker: 15 folds
    ([16384, 40, 16384, 1, 12000], 32, 8, 16, 3),
])
def test_accumulation_chain_is_folded(pkv, cuda_device, lens, hq, hkv, page, ctas):
    """With few workers each one's range spans thousands of chunks; every 128
    chunks a worker adds its tensor-core accumulator into its piece's slot in
    fp32 and restarts it, so no accumulation chain is longer than 128 chunks.
    All rows against the oracle, the same calls with many workers alike."""
    wl = workloads.Workload(54, "chain", lens, 0, hq, hkv, page, pool_factor=1.2, seed=23)
    f = fill_gpu(wl, 0, cuda_device)
    ref = _full_oracle(wl, f)
    for c in (ctas, 0):
        got = _decode(pkv, f, max_ctas=c).double().cpu().numpy()
        assert int(f.err.item()) == 0
        assert_close(got, ref, f"ctas={c}")
        diff = np.abs(got - ref).max()
        assert diff <= 1e-4, diff


@pytest.mark.parametrize("lens,sizes,hq,hkv,page", [
    ([37, 100, 1, 300, 64, 0], [16, 64, 32, 64, 16, 256], 16, 2, 16),
    ([1000, 3, 2049, 513], [256, 32, 64, 32], 64, 8, 32),
    ([9000, 700, 20000], [64, 16, 64], 32, 8, 16),          # the notes' 16 / 64 split by length
])
def test_per_sequence_page_sizes(pkv, cuda_device, lens, sizes, hq, hkv, page):
    """Sequences with their own page size (runs of P_b / P pool pages): all
    rows against the oracle for several splits, and bit-identical to the same
    cache read through the equivalent table of pool pages."""
    wl = workloads.Workload(55, "varpage", lens, 0, hq, hkv, page, pool_factor=1.3, seed=29, page_sizes=sizes)
    f = fill_gpu(wl, 0, cuda_device)
    ref = _full_oracle(wl, f)
    outs = []
    for ctas in (0, 1, 5):
        got = _decode(pkv, f, max_ctas=ctas)
        assert int(f.err.item()) == 0
        assert_close(got.double().cpu().numpy(), ref, f"ctas={ctas}")
        outs.append(got)
    bt = wl.block_table().numpy()
    wide = np.full((wl.batch, max(1, max((L + page - 1) // page for L in wl.seq_lens))), -1, np.int32)
    for b, L in enumerate(wl.seq_lens):
        for t in range(0, L, page):
            wide[b, t // page] = bt[b, t // sizes[b]] + (t % sizes[b]) // page
    n = pkv.pkv_decode_workspace_size(wl.batch, hq, hkv, 128, f.max_len, page)
    ws = torch.empty(n, dtype=torch.uint8, device=cuda_device)
    plain = pkv.paged_gqa_decode(f.q, f.kc, f.vc, f.ks, f.vs, torch.from_numpy(wide).to(cuda_device), f.lens,
                                 out_dtype=torch.float32, workspace=ws, max_seq_len=f.max_len)
    torch.cuda.synchronize()
    assert torch.equal(plain, outs[0])


def test_invalid_page_size_flags_error(pkv, cuda_device):
    wl = workloads.Workload(56, "badpage", [40, 70], 0, 8, 2, 32, seed=1, page_sizes=[32, 64])
    f = fill_gpu(wl, 0, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for bad in (16, 48, 512):                      # below the pool page, not a power of two, above 256
        err.zero_()
        psz = torch.tensor([32, bad], dtype=torch.int32, device=cuda_device)
        out = _decode(pkv, f, err=err, psz=psz)
        assert int(err.item()) & pkv.DEVERR_PAGESIZE
        assert torch.all(out[1] == 0)              # the sequence reads as empty
    err.zero_()
    _decode(pkv, f, err=err)
    assert int(err.item()) == 0


def test_closed_forms_uniform_and_one_hot_weights(pkv, cuda_device):
    """K = 0 gives uniform weights, so o = mean_t dequant(V_t); V one-hot per
    token (V_t = e_t, t < 128) returns the softmax weights, compared with the
    oracle's weights."""
    dev = cuda_device
    B, Hq, Hkv, P = 2, 16, 2, 16
    L = 100
    npg = (L + P - 1) // P
    bt = torch.arange(B * npg, dtype=torch.int32, device=dev).view(B, npg)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, Hq, 128, generator=g).to(torch.bfloat16).to(dev)
    ks = torch.tensor([0.05, 0.02], device=dev)
    vs = torch.tensor([0.3, 1.7], device=dev)
    # K = 0: mean of the dequantised V
    kc = torch.zeros(B * npg, Hkv, P, 128, dtype=torch.uint8, device=dev)
    vc = torch.randint(0, 256, kc.shape, dtype=torch.uint8, generator=None, device=dev)
    vc[(vc & 0x7F) == 0x7F] = 0x33
    out = pkv.paged_gqa_decode(q, kc, vc, ks, vs, bt, lens, out_dtype=torch.float32)
    vals = oracle.e4m3_value(vc.cpu().numpy()) * vs.cpu().numpy().reshape(1, Hkv, 1, 1)
    bt_np = bt.cpu().numpy()
    for b in range(B):
        rows = np.concatenate([vals[bt_np[b, p]] for p in range(npg)], axis=1)[:, :L]   # [Hkv, L, 128]
        mean = rows.mean(axis=1)
        exp = np.repeat(mean, Hq // Hkv, axis=0)
        assert np.abs(out[b].double().cpu().numpy() - exp).max() <= 1e-5 * max(1.0, np.abs(exp).max())
    # one-hot V: code 0x38 (1.0) at dim t of token t, zero elsewhere; v_scale 1
    kc = torch.randint(0, 256, kc.shape, dtype=torch.uint8, device=dev)
    kc[(kc & 0x7F) == 0x7F] = 0x30
    vc = torch.zeros_like(kc)
    for b in range(B):
        for t in range(L):
            vc[bt_np[b, t // P], :, t % P, t] = 0x38
    ones = torch.ones(Hkv, device=dev)
    out = pkv.paged_gqa_decode(q, kc, vc, ks, ones, bt, lens, out_dtype=torch.float32)
    _, w = oracle.paged_decode(q.cpu().view(torch.uint16).numpy(), kc.cpu().numpy(), vc.cpu().numpy(),
                               ks.cpu().numpy(), ones.cpu().numpy(), bt_np, lens.cpu().numpy(), want_weights=True)
    w = w.reshape(B, Hq, L)
    got = out.double().cpu().numpy()
    assert np.abs(got[:, :, :L] - w).max() <= 2e-6
    assert np.all(got[:, :, L:] == 0)


def test_page_sizes_and_batches_interleaved(pkv, cuda_device):
    """Every page size runs the same kernel, whose shared memory grows with
    the batch: a call with another page size and a smaller batch in between
    must not lower the limit a larger batch needs."""
    big = workloads.Workload(53, "big", [1, 2, 15, 16, 17, 31, 33, 40, 90], 0, 8, 1, 16, seed=2)
    small = workloads.Workload(54, "small", [4097, 1, 999], 0, 64, 8, 32, seed=3)
    fb = fill_gpu(big, 0, cuda_device)
    fs = fill_gpu(small, 0, cuda_device)
    ref_b, ref_s = _full_oracle(big, fb), _full_oracle(small, fs)
    for _ in range(2):
        assert_close(_decode(pkv, fb, max_ctas=7).double().cpu().numpy(), ref_b, "P=16, batch 9")
        assert_close(_decode(pkv, fs, max_ctas=7).double().cpu().numpy(), ref_s, "P=32, batch 3")

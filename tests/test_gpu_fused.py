"""pkv_append_decode_fp8 (append fused into the decode launch) on the GPU:
page bytes and outputs bit-identical to pkv_kv_append_fp8 + pkv_paged_gqa_decode,
and within tolerance of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_fill import assert_close, fill_gpu, step_tokens
from tests.test_gpu_decode import _full_oracle

pytestmark = pytest.mark.gpu


def _ws(pkv, wl, dev, max_ctas=0):
    n = pkv.pkv_decode_workspace_size(wl.batch, wl.hq, wl.hkv, 128, wl.max_len, wl.page_size, max_ctas)
    return torch.full((n,), 0xFF, dtype=torch.uint8, device=dev)


def _separate(pkv, wl, dev, dtype, max_ctas=0):
    f = fill_gpu(wl, 0, dev, step_append=False)
    k, v = step_tokens(wl, 0, dev)
    k, v = k.to(dtype), v.to(dtype)
    slots = torch.cat([wl.slots(b, L, L + wl.append) for b, L in enumerate(wl.prefill_lens)]).to(dev)
    pkv.pkv_kv_append_fp8(k.reshape(-1, wl.hkv, 128), v.reshape(-1, wl.hkv, 128), slots, f.ks, f.vs, f.kc, f.vc,
                          f.err)
    out = torch.empty(f.q.shape, dtype=torch.float32, device=dev)
    pkv.pkv_paged_gqa_decode(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out, _ws(pkv, wl, dev, max_ctas), None,
                             f.err, max_ctas, max_seq_len=f.max_len, seq_page_sizes=f.psz)
    torch.cuda.synchronize()
    return f, out


def _fused(pkv, wl, dev, dtype, max_ctas=0):
    f = fill_gpu(wl, 0, dev, step_append=False)
    k, v = step_tokens(wl, 0, dev)
    out = torch.empty(f.q.shape, dtype=torch.float32, device=dev)
    pkv.pkv_append_decode_fp8(k.to(dtype), v.to(dtype), f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out,
                              _ws(pkv, wl, dev, max_ctas), None, f.err, max_ctas, max_seq_len=f.max_len,
                              seq_page_sizes=f.psz)
    torch.cuda.synchronize()
    return f, out


@pytest.mark.parametrize("lens,append,hq,hkv,page", [
    ([36, 99], 1, 8, 1, 16),           # the tiny workload's shape with one new token
    ([15, 16, 31, 1], 2, 8, 2, 16),     # new tokens crossing page boundaries
    ([100, 7, 64], 3, 16, 4, 32),
    ([4096] * 4, 1, 32, 8, 16),
    ([0, 5], 1, 4, 1, 16),              # a sequence made of its new token only
    ([63, 100, 17], 2, 16, 2, 64),      # 64-token pages: new tokens in chunks inside a page
    ([255, 30], 1, 8, 8, 256),
])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_equals_separate(pkv, cuda_device, lens, append, hq, hkv, page, dtype):
    _fused_vs_separate(pkv, cuda_device, lens, append, hq, hkv, page, dtype, None)


@pytest.mark.parametrize("lens,append,hq,hkv,sizes", [
    ([63, 100, 17, 300], 2, 16, 2, [64, 16, 32, 64]),     # new tokens inside runs of pool pages
    ([1000, 5, 250], 1, 64, 8, [256, 16, 64]),
])
def test_fused_equals_separate_per_sequence_pages(pkv, cuda_device, lens, append, hq, hkv, sizes):
    _fused_vs_separate(pkv, cuda_device, lens, append, hq, hkv, 16, torch.float32, sizes)


def _fused_vs_separate(pkv, cuda_device, lens, append, hq, hkv, page, dtype, sizes):
    wl = workloads.Workload(60, "fused", lens, append, hq, hkv, page, pool_factor=1.5, seed=31, page_sizes=sizes)
    for ctas in (0, 3):
        fs, out_s = _separate(pkv, wl, cuda_device, dtype, ctas)
        ff, out_f = _fused(pkv, wl, cuda_device, dtype, ctas)
        assert int(fs.err.item()) == 0 and int(ff.err.item()) == 0
        assert torch.equal(fs.kc, ff.kc) and torch.equal(fs.vc, ff.vc)
        assert torch.equal(out_s, out_f)
    if dtype == torch.float32:
        assert_close(out_f.double().cpu().numpy(), _full_oracle(wl, ff), "fused vs oracle")


def test_fused_llama3_8b_layer_matches_oracle_pages(pkv, cuda_device):
    wl = workloads.config(1)
    f, out = _fused(pkv, wl, cuda_device, torch.float32)
    ks, vs = f.ks.cpu().numpy(), f.vs.cpu().numpy()
    for b in (0, wl.batch - 1):
        L = wl.seq_lens[b]
        t = L - 1
        phys = int(wl.block_table()[b, t // 16])
        for h in (0, wl.hkv - 1):
            exp_k = oracle.e4m3_encode(wl.kv_head_values(0, 0, b, h, t, t + 1).numpy().ravel() / ks[h])
            exp_v = oracle.e4m3_encode(wl.kv_head_values(0, 1, b, h, t, t + 1).numpy().ravel() / vs[h])
            assert np.array_equal(f.kc[phys, h, t % 16].cpu().numpy(), exp_k)
            assert np.array_equal(f.vc[phys, h, t % 16].cpu().numpy(), exp_v)


def test_fused_short_sequence_flags_error(pkv, cuda_device):
    wl = workloads.Workload(61, "short", [0, 40], 0, 8, 1, 16, seed=2)
    f = fill_gpu(wl, 0, cuda_device)
    k = torch.ones(2, 2, 1, 128, device=cuda_device)
    out = torch.empty(f.q.shape, dtype=torch.float32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.pkv_append_decode_fp8(k, k, f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out, _ws(pkv, wl, cuda_device),
                              None, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_SEQLEN

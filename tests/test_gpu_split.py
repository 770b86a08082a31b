"""The weighted decode split on the GPU.

Per-CTA weights change only how the list of chunks is cut among the workers,
never the math: outputs stay within the tolerance of the oracle (max-abs <=
2e-3, rel-L2 <= 1e-3), pages written by the fused append are bit-identical,
equal weights reproduce the even split bit for bit, and weights installed
for another grid size are ignored.  Covers ranges long enough to fold their
accumulator (more than 128 chunks) and lists shorter than the workers'
shares (empty ranges).
"""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_fill import assert_close, fill_gpu, oracle_rows, sample_pairs, step_tokens
from tests.test_gpu_decode import _decode, _full_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _even_split(pkv, cuda_device):
    pkv.pkv_decode_set_split_weights(None)
    yield
    pkv.pkv_decode_set_split_weights(None)


def _weights(n, seed):
    return np.random.default_rng(seed).integers(768, 1281, n).tolist()


@pytest.mark.parametrize("ctas", [1, 7, 50])
@pytest.mark.parametrize("value", [768, 1024, 1280])
def test_equal_weights_are_the_even_split(pkv, cuda_device, ctas, value):
    wl = workloads.Workload(60, "eq", [700, 33, 1601, 16, 0, 4097], 0, 32, 8, 16, pool_factor=1.5, seed=3)
    f = fill_gpu(wl, 0, cuda_device)
    even = _decode(pkv, f, max_ctas=ctas)
    pkv.pkv_decode_set_split_weights([value] * ctas)
    assert pkv.pkv_decode_get_split_weights() == [value] * ctas
    same = _decode(pkv, f, max_ctas=ctas)
    assert torch.equal(even, same)
    assert int(f.err.item()) == 0


def test_weights_for_another_grid_are_ignored(pkv, cuda_device):
    wl = workloads.Workload(61, "other", [900, 5, 2500], 0, 16, 2, 16, seed=4)
    f = fill_gpu(wl, 0, cuda_device)
    even = _decode(pkv, f, max_ctas=7)
    pkv.pkv_decode_set_split_weights(_weights(5, 1))
    assert torch.equal(even, _decode(pkv, f, max_ctas=7))
    pkv.pkv_decode_set_split_weights(_weights(7, 1))
    weighted = _decode(pkv, f, max_ctas=7)
    assert_close(weighted.double().cpu().numpy(), even.double().cpu().numpy(), "weighted vs even")


@pytest.mark.parametrize("lens,hq,hkv,page", [
    ([1, 2, 15, 16, 17, 31, 33], 8, 1, 16),
    ([0, 5, 0, 300], 16, 2, 16),
    ([1000, 3, 47], 32, 8, 16),
    ([4097, 1, 999], 64, 8, 32),
    ([255, 256, 257, 3000], 64, 8, 256),
])
@pytest.mark.parametrize("ctas", [2, 7, 50])
def test_random_weights_match_the_oracle(pkv, cuda_device, lens, hq, hkv, page, ctas):
    wl = workloads.Workload(62, "wragged", lens, 0, hq, hkv, page, pool_factor=1.5, seed=22)
    f = fill_gpu(wl, 0, cuda_device)
    ref = _full_oracle(wl, f)
    for seed in range(3):
        pkv.pkv_decode_set_split_weights(_weights(ctas, seed))
        got = _decode(pkv, f, max_ctas=ctas).double().cpu().numpy()
        assert int(f.err.item()) == 0
        assert_close(got, ref, f"ctas={ctas} seed={seed}")
        for b, L in enumerate(wl.seq_lens):
            if L == 0:
                assert np.all(got[b] == 0)


def test_lists_shorter_than_the_shares(pkv, cuda_device):
    """Ten chunk-heads over 200 workers: most ranges are empty."""
    wl = workloads.Workload(63, "short", [37, 100], 0, 8, 1, 16, seed=7)
    f = fill_gpu(wl, 0, cuda_device)
    ref = _full_oracle(wl, f)
    for seed in range(4):
        pkv.pkv_decode_set_split_weights(_weights(50, seed))
        assert_close(_decode(pkv, f, max_ctas=50).double().cpu().numpy(), ref, f"seed={seed}")


def test_long_ranges_fold_their_accumulators(pkv, cuda_device):
    """Two CTAs at weights 768 and 1280: the second CTA's warps take about 680
    chunks each, folded every 128."""
    wl = workloads.Workload(64, "long", [40000, 30000], 0, 8, 1, 16, seed=9)
    f = fill_gpu(wl, 0, cuda_device)
    ref = _full_oracle(wl, f)
    even = _decode(pkv, f, max_ctas=2).double().cpu().numpy()
    assert_close(even, ref, "even")
    for w in ([768, 1280], [1280, 768], [1200, 800]):
        pkv.pkv_decode_set_split_weights(w)
        assert_close(_decode(pkv, f, max_ctas=2).double().cpu().numpy(), ref, f"weights={w}")


def test_fused_append_with_weights(pkv, cuda_device):
    """The fused step writes the same pages with or without weights (every
    chunk still has exactly one owner) and its output matches the oracle."""
    wl = workloads.Workload(65, "wfused", [511, 1, 2048, 77, 4000], 2, 32, 8, 16, pool_factor=1.5, seed=12)
    fa = fill_gpu(wl, 0, cuda_device, step_append=False)
    fb = fill_gpu(wl, 0, cuda_device, step_append=False)
    k_new, v_new = step_tokens(wl, 0, cuda_device)
    outs = []
    for f, weights in ((fa, None), (fb, _weights(7, 5))):
        pkv.pkv_decode_set_split_weights(weights)
        outs.append(pkv.append_decode_fp8(k_new, v_new, f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens,
                                          out_dtype=torch.float32, device_error=f.err, max_ctas=7,
                                          max_seq_len=f.max_len))
        torch.cuda.synchronize()
        assert int(f.err.item()) == 0
    assert torch.equal(fa.kc, fb.kc) and torch.equal(fa.vc, fb.vc)
    ref = _full_oracle(wl, fb)
    for out in outs:
        assert_close(out.double().cpu().numpy(), ref, "fused")


def test_calibrate_installs_weights_and_stays_deterministic(pkv, cuda_device):
    wl = workloads.config(1)
    f = fill_gpu(wl, 0, cuda_device)
    out = torch.empty(f.q.shape, dtype=torch.float32, device=cuda_device)
    ws = pkv.decode_workspace(wl.batch, wl.hq, wl.hkv, wl.page_size, cuda_device, 0, f.max_len)
    w = pkv.pkv_decode_calibrate_split(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out, ws, rounds=2,
                                       max_seq_len=f.max_len)
    assert len(w) > 0 and all(768 <= x <= 1280 for x in w)
    assert pkv.pkv_decode_get_split_weights() == w
    a = _decode(pkv, f)
    b = _decode(pkv, f)
    assert torch.equal(a, b)
    ks, vs = wl.scales(0)
    pairs = sample_pairs(wl, 6)
    exp = oracle_rows(wl, 0, pairs, ks.numpy(), vs.numpy())
    got = np.stack([a[b_, i].double().cpu().numpy() for b_, i in pairs])
    assert_close(got, np.stack([exp[p] for p in pairs]), "calibrated")
    # the weights can be saved and restored
    pkv.pkv_decode_set_split_weights(None)
    assert pkv.pkv_decode_get_split_weights() == []
    pkv.pkv_decode_set_split_weights(w)
    assert torch.equal(_decode(pkv, f), a)

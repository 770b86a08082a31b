"""Pins for the oracle's paged decode attention (CPU only).

  * brute force: dense fp64 softmax attention over logical-order tokens,
    quantised through torch's float8 cast (tests/dense_ref.py), on the tiny
    workload and on random small shapes (ragged lengths, G in 1..8, P 16/32);
  * closed forms: a 1-token context returns dequant(V) exactly; K = 0 gives
    the mean of V; a 2-token case gives sigmoid weights; L = 0 gives zeros;
  * invariants: softmax weights sum to 1; a random permutation of physical
    pages (block table permuted alike) leaves every output bit unchanged;
  * per-sequence page sizes (a P_b-token page is a run of P_b / P pool
    pages): dense brute force on mixed 16/32/64/256-token pages, and the same
    result as the uniform P-token table that lists every pool page of the
    runs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.dense_ref import dense_attention, dequant_torch, quantize_torch

SM = 1.0 / math.sqrt(128.0)


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b))))


def _fill(wl, layer=0):
    ks, vs = wl.scales(layer)
    P, H, D = wl.page_size, wl.hkv, wl.head_dim
    kc = np.full((wl.num_pages, H, P, D), 0x7F, np.uint8)        # NaN in unused slots
    vc = np.full_like(kc, 0x7F)
    dense_k, dense_v = [], []
    for b, L in enumerate(wl.seq_lens):
        slots = wl.slots(b, 0, L)
        k = wl.kv_rows(layer, 0, b, 0, L)
        v = wl.kv_rows(layer, 1, b, 0, L)
        oracle.kv_append(k.numpy(), slots.numpy(), ks.numpy(), kc)
        oracle.kv_append(v.numpy(), slots.numpy(), vs.numpy(), vc)
        dense_k.append(dequant_torch(quantize_torch(k, ks), ks))
        dense_v.append(dequant_torch(quantize_torch(v, vs), vs))
    return kc, vc, ks.numpy(), vs.numpy(), dense_k, dense_v


def _check_dense(wl, tol=1e-12):
    kc, vc, ks, vs, dk, dv = _fill(wl)
    q = wl.q()
    bt = wl.block_table().numpy()
    lens = np.array(wl.seq_lens, np.int32)
    psz = np.array(wl.page_sizes, np.int32) if wl.page_sizes is not None else None
    out = oracle.paged_decode(q.view(torch.uint16).numpy(), kc, vc, ks, vs, bt, lens, seq_page_sizes=psz)
    out = out.reshape(wl.batch, wl.hq, wl.head_dim)
    for b in range(wl.batch):
        ref = dense_attention(q[b].double().numpy(), dk[b], dv[b], SM)
        assert _rel(out[b], ref) < tol, b
    return out


def test_tiny_workload_matches_dense_brute_force():
    _check_dense(workloads.config(0))


@pytest.mark.parametrize("lens,hq,hkv,P", [
    ([1, 2, 15, 16, 17], 8, 1, 16),
    ([31, 32, 33, 64, 5], 4, 2, 32),
    ([50, 7], 2, 2, 16),
    ([3, 40, 100], 16, 4, 16),
    ([77], 64, 8, 32),
])
def test_random_small_shapes_match_dense(lens, hq, hkv, P):
    wl = workloads.Workload(90, "adhoc", lens, 0, hq, hkv, P, pool_factor=1.5, seed=7)
    _check_dense(wl)


def test_planted_mistakes_are_caught_by_dense_pin():
    """Feeding the oracle a wrong head map, a wrong scale or a block-table
    entry from another sequence changes its result enough for the dense pin to fail."""
    wl = workloads.Workload(91, "adhoc", [40, 23], 0, 8, 2, 16, seed=3)
    kc, vc, ks, vs, dk, dv = _fill(wl)
    q = wl.q()
    bt = wl.block_table().numpy()
    lens = np.array(wl.seq_lens, np.int32)
    qb = q.view(torch.uint16).numpy()
    ref = dense_attention(q[0].double().numpy(), dk[0], dv[0], SM)
    good = oracle.paged_decode(qb, kc, vc, ks, vs, bt, lens).reshape(2, 8, 128)[0]
    assert _rel(good, ref) < 1e-12
    bad_scale = oracle.paged_decode(qb, kc, vc, ks, vs, bt, lens, sm_scale=1.0).reshape(2, 8, 128)[0]
    assert _rel(bad_scale, ref) > 1e-3
    qperm = qb[:, [1, 0, 2, 3, 4, 5, 6, 7], :].copy()        # heads 0/1 swapped: wrong q->kv map
    ref_perm = dense_attention(q[0].double().numpy()[[1, 0, 2, 3, 4, 5, 6, 7]], dk[0], dv[0], SM)
    out_perm = oracle.paged_decode(qperm, kc, vc, ks, vs, bt, lens).reshape(2, 8, 128)[0]
    assert _rel(out_perm, ref_perm) < 1e-12                   # relabelled consistently: fine
    assert _rel(out_perm, ref) > 1e-3                         # but not equal to the true map
    bt_wrong = bt.copy()
    bt_wrong[0, 0] = bt[1, 0]                                 # gather a page of the other sequence
    out_wrong = oracle.paged_decode(qb, kc, vc, ks, vs, bt_wrong, lens).reshape(2, 8, 128)[0]
    assert _rel(out_wrong, ref) > 1e-3
    vs_wrong = vs * 1.01
    out_vs = oracle.paged_decode(qb, kc, vc, ks, vs_wrong, bt, lens).reshape(2, 8, 128)[0]
    assert _rel(out_vs, ref) > 1e-3


def test_one_token_context_returns_dequantised_v_exactly():
    wl = workloads.Workload(92, "adhoc", [1, 1, 1], 0, 8, 2, 16, seed=11)
    kc, vc, ks, vs, dk, dv = _fill(wl)
    q = wl.q().view(torch.uint16).numpy()
    out = oracle.paged_decode(q, kc, vc, ks, vs, wl.block_table().numpy(),
                              np.array(wl.seq_lens, np.int32)).reshape(3, 8, 128)
    for b in range(3):
        for i in range(8):
            assert np.array_equal(out[b, i], dv[b][0, i // 4])


def test_zero_keys_give_mean_of_values():
    P, L, D = 16, 45, 128
    npg = (L + P - 1) // P
    rng = np.random.default_rng(0)
    kc = np.zeros((npg, 1, P, D), np.uint8)                      # code 0 = +0.0
    vc = rng.integers(0, 256, size=kc.shape, dtype=np.uint8)
    vc[(vc & 0x7F) == 0x7F] = 0x10                               # no NaN codes
    bt = np.arange(npg, dtype=np.int32)[None]
    q = torch.randn(1, 4, D).to(torch.bfloat16).view(torch.uint16).numpy()
    vs = np.array([0.25], np.float32)
    out = oracle.paged_decode(q, kc, vc, np.ones(1, np.float32), vs, bt, np.array([L], np.int32))
    vals = oracle.e4m3_value(vc.reshape(-1, D)[:L]) * 0.25
    mean = vals.sum(axis=0) / L
    for i in range(4):
        assert np.max(np.abs(out[i] - mean)) < 1e-12 * max(1.0, np.abs(mean).max())


def test_two_token_closed_form():
    """K rows e_0 * a and e_0 * c (codes chosen exactly), q = e_0: weights are
    sigmoid((a - c) * sm_scale), output is the weighted mix of two V rows."""
    D, P = 128, 16
    kc = np.zeros((1, 1, P, D), np.uint8)
    vc = np.zeros_like(kc)
    kc[0, 0, 0, 0] = 0x48      # 2^(9-7) * 1 = 4
    kc[0, 0, 1, 0] = 0xB8      # -1
    vc[0, 0, 0, :] = 0x38      # +1
    vc[0, 0, 1, :] = 0x40      # +2
    q = np.zeros((1, 1, D), np.uint16)
    q[0, 0, 0] = 0x3F80        # bf16 1.0
    out, w = oracle.paged_decode(q, kc, vc, np.array([0.5], np.float32), np.array([3.0], np.float32),
                                 np.zeros((1, 1), np.int32), np.array([2], np.int32), want_weights=True)
    s0, s1 = 4 * 0.5 * SM, -1 * 0.5 * SM
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert abs(w[0, 0] - w0) < 1e-15 and abs(w[0, 1] - (1 - w0)) < 1e-15
    assert np.allclose(out[0], 3.0 * (w0 * 1 + (1 - w0) * 2), rtol=0, atol=1e-14)


def test_weights_sum_to_one_and_empty_sequence_is_zero():
    wl = workloads.Workload(93, "adhoc", [0, 33, 200], 0, 4, 1, 16, seed=2)
    kc, vc, ks, vs, dk, dv = _fill(wl)
    out, w = oracle.paged_decode(wl.q().view(torch.uint16).numpy(), kc, vc, ks, vs,
                                 wl.block_table().numpy(), np.array(wl.seq_lens, np.int32),
                                 want_weights=True)
    out = out.reshape(3, 4, 128)
    w = w.reshape(3, 4, -1)
    assert (out[0] == 0).all() and (w[0] == 0).all()
    for b, L in [(1, 33), (2, 200)]:
        assert np.all(np.abs(w[b, :, :L].sum(axis=1) - 1) < 1e-12)
        assert (w[b, :, L:] == 0).all()


def test_page_permutation_invariance():
    wl = workloads.Workload(94, "adhoc", [70, 129, 16], 0, 8, 2, 16, pool_factor=2.0, seed=4)
    kc, vc, ks, vs, _, _ = _fill(wl)
    q = wl.q().view(torch.uint16).numpy()
    bt = wl.block_table().numpy()
    lens = np.array(wl.seq_lens, np.int32)
    base = oracle.paged_decode(q, kc, vc, ks, vs, bt, lens)
    perm = np.random.default_rng(8).permutation(wl.num_pages)     # new home of page p = perm[p]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    moved = oracle.paged_decode(q, kc2, vc2, ks, vs, bt2, lens)
    assert np.array_equal(base, moved)


def test_threaded_equals_single_thread():
    wl = workloads.Workload(95, "adhoc", [300, 41, 90, 17], 0, 16, 2, 32, seed=6)
    kc, vc, ks, vs, _, _ = _fill(wl)
    args = (wl.q().view(torch.uint16).numpy(), kc, vc, ks, vs, wl.block_table().numpy(),
            np.array(wl.seq_lens, np.int32))
    assert np.array_equal(oracle.paged_decode(*args, threads=1), oracle.paged_decode(*args, threads=5))


def test_bad_block_table_entry_is_reported():
    kc = np.zeros((2, 1, 16, 128), np.uint8)
    with pytest.raises(ValueError):
        oracle.paged_decode(np.zeros((1, 1, 128), np.uint16), kc, kc, np.ones(1, np.float32),
                            np.ones(1, np.float32), np.array([[5]], np.int32), np.array([3], np.int32))


@pytest.mark.parametrize("lens,sizes,P", [
    ([37, 100, 1, 300, 64], [16, 64, 32, 64, 16], 16),
    ([200, 513, 31], [32, 256, 64], 32),
    ([1000, 17], [256, 16], 16),
])
def test_per_sequence_page_sizes_match_dense(lens, sizes, P):
    wl = workloads.Workload(92, "varpage", lens, 0, 16, 2, P, pool_factor=1.5, seed=13, page_sizes=sizes)
    _check_dense(wl)


def test_per_sequence_page_sizes_equal_expanded_uniform_table():
    """A table of P_b-token pages reads exactly what a table of P-token pages
    reads when it lists, for every logical page, its P_b / P pool pages in
    order."""
    lens, sizes, P = [300, 77, 129, 5], [64, 16, 32, 64], 16
    wl = workloads.Workload(93, "varpage", lens, 0, 8, 2, P, pool_factor=1.25, seed=17, page_sizes=sizes)
    kc, vc, ks, vs, _, _ = _fill(wl)
    bt = wl.block_table().numpy()
    wide = np.full((wl.batch, max((L + P - 1) // P for L in wl.seq_lens)), -1, np.int32)
    for b, L in enumerate(wl.seq_lens):
        for t in range(0, L, P):                                # pool page of every P-token block
            wide[b, t // P] = bt[b, t // sizes[b]] + (t % sizes[b]) // P
    q = wl.q().view(torch.uint16).numpy()
    lens_np = np.array(wl.seq_lens, np.int32)
    a = oracle.paged_decode(q, kc, vc, ks, vs, bt, lens_np, seq_page_sizes=np.array(sizes, np.int32))
    b_ = oracle.paged_decode(q, kc, vc, ks, vs, wide, lens_np)
    assert np.array_equal(a, b_)
    # reading the table as if every page had P tokens (a planted mistake: the
    # logical page index taken with P) differs on the sequences with P_b > P
    short = np.minimum(lens_np, bt.shape[1] * P).astype(np.int32)
    a_s = oracle.paged_decode(q, kc, vc, ks, vs, bt, short, seq_page_sizes=np.array(sizes, np.int32))
    c = oracle.paged_decode(q, kc, vc, ks, vs, bt, short).reshape(wl.batch, wl.hq, -1)
    a_s = a_s.reshape(wl.batch, wl.hq, -1)
    for b in range(wl.batch):
        same = np.allclose(a_s[b], c[b], rtol=1e-6, atol=1e-9)
        assert same == (sizes[b] == P or short[b] <= P), b

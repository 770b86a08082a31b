"""Pins for the oracle's kv_append (CPU only).

The oracle writes pages with its own scalar codec and slot arithmetic; the
pin rebuilds the same pool with torch's float8 cast and torch index
arithmetic (different code, a library codec) and demands identical bytes.
"""
import numpy as np
import torch

import oracle
import workloads
from tests.dense_ref import quantize_torch


def _torch_pool(x, slots, scale, num_pages, P):
    """Reference pool [num_pages, Hkv, P, D] built with torch ops."""
    T, H, D = x.shape
    pool = torch.zeros(num_pages * P, H, D, dtype=torch.uint8)        # [slot, h, d]
    keep = slots >= 0
    pool[slots[keep]] = quantize_torch(x[keep], scale)
    return pool.view(num_pages, P, H, D).permute(0, 2, 1, 3).contiguous()


def _fill_oracle(wl, layer=0):
    ks, vs = wl.scales(layer)
    P, H, D = wl.page_size, wl.hkv, wl.head_dim
    kc = np.zeros((wl.num_pages, H, P, D), np.uint8)
    vc = np.zeros_like(kc)
    xs, ss = [], []
    for b, L in enumerate(wl.prefill_lens):
        slots = wl.slots(b, 0, L)
        k = wl.kv_rows(layer, 0, b, 0, L)
        v = wl.kv_rows(layer, 1, b, 0, L)
        assert oracle.kv_append(k.numpy(), slots.numpy(), ks.numpy(), kc) == 0
        assert oracle.kv_append(v.numpy(), slots.numpy(), vs.numpy(), vc) == 0
        xs.append((k, v))
        ss.append(slots)
    return kc, vc, xs, ss, ks, vs


def test_tiny_pool_matches_torch_route():
    wl = workloads.config(0)
    kc, vc, xs, ss, ks, vs = _fill_oracle(wl)
    k_all = torch.cat([k for k, _ in xs])
    v_all = torch.cat([v for _, v in xs])
    slots = torch.cat(ss)
    assert np.array_equal(kc, _torch_pool(k_all, slots, ks, wl.num_pages, wl.page_size).numpy())
    assert np.array_equal(vc, _torch_pool(v_all, slots, vs, wl.num_pages, wl.page_size).numpy())


def test_random_shapes_and_skips_match_torch_route():
    g = torch.Generator().manual_seed(5)
    for P, H, T in [(16, 1, 5), (16, 3, 40), (32, 2, 70), (32, 8, 33)]:
        D = 128
        num_pages = (T + P - 1) // P + 3
        slots = torch.randperm(num_pages * P, generator=g)[:T].to(torch.int64)
        slots[::7] = -1                                   # skipped tokens
        x = torch.randn(T, H, D, generator=g) * 30
        scale = torch.rand(H, generator=g) * 0.5 + 0.01
        cache = np.full((num_pages, H, P, D), 0xAB, np.uint8)
        untouched = cache.copy()
        assert oracle.kv_append(x.numpy(), slots.numpy(), scale.numpy(), cache) == 0
        ref = _torch_pool(x, slots, scale, num_pages, P).numpy()
        written = np.zeros(num_pages * P, bool)
        written[slots[slots >= 0].numpy()] = True
        written = written.reshape(num_pages, P)[:, None, :, None]
        written = np.broadcast_to(written, cache.shape)
        assert np.array_equal(cache[written], ref[written])
        assert np.array_equal(cache[~written], untouched[~written])   # nothing else touched


def test_out_of_pool_slots_are_counted_and_skipped():
    x = np.ones((3, 1, 128), np.float32)
    cache = np.zeros((2, 1, 16, 128), np.uint8)
    bad = oracle.kv_append(x, np.array([0, 32, 99], np.int64), np.ones(1, np.float32), cache)
    assert bad == 2
    assert (cache[0, 0, 0] == 0x38).all() and cache.sum() == 0x38 * 128


def test_bf16_input_equals_fp32_of_widened_values():
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(9, 2, 128, generator=g) * 10).to(torch.bfloat16)
    slots = torch.arange(9, dtype=torch.int64)
    scale = np.array([0.03, 0.2], np.float32)
    c1 = np.zeros((1, 2, 16, 128), np.uint8)
    c2 = np.zeros_like(c1)
    oracle.kv_append(x.view(torch.uint16).numpy(), slots.numpy(), scale, c1)
    oracle.kv_append(x.float().numpy(), slots.numpy(), scale, c2)
    assert np.array_equal(c1, c2)


def test_division_not_reciprocal_multiply():
    """x / s and x * (1/s) can round to different fp32 values; near an E4M3
    rounding midpoint that changes the code.  Builds such inputs next to every
    midpoint and checks that the oracle follows the division."""
    s = np.float32(0.0373)
    mags = np.sort(np.unique(np.abs(oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8)))))
    mids = (mags[:-1] + mags[1:]) / 2
    base = (mids * np.float64(s)).astype(np.float32)
    cand = np.concatenate([(base.view(np.uint32).astype(np.int64) + d).astype(np.uint32).view(np.float32)
                           for d in range(-4, 5)])
    div = cand / s
    mul = cand * (np.float32(1) / s)
    differ = oracle.e4m3_encode(div) != oracle.e4m3_encode(mul)
    assert differ.any()                                 # the distinction matters
    xs = cand[differ][:64]
    cache = np.zeros((4, 1, 16, 128), np.uint8)
    xx = np.zeros((len(xs), 1, 128), np.float32)
    xx[:, 0, 0] = xs
    oracle.kv_append(xx, np.arange(len(xs), dtype=np.int64), np.array([s]), cache)
    got = cache.reshape(-1, 128)[: len(xs), 0]
    assert np.array_equal(got, oracle.e4m3_encode(xs / s))
    assert not np.array_equal(got, oracle.e4m3_encode(xs * (np.float32(1) / s)))

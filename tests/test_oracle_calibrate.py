"""Pins for the oracle's KV-scale calibration (CPU only): the running maximum
agrees with numpy's max over |x| (a library reduction), merges batches like a
single pass, skips NaN, and the scale follows the pages' recipe max/448 with
the 1e-12 floor (exact cases checked by hand)."""
import numpy as np
import torch

import oracle
import workloads


def test_running_max_matches_numpy_and_batches_merge():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((300, 8, 128)) * rng.choice([0.1, 3.0, 40.0], (300, 8, 1))).astype(np.float32)
    rm = np.zeros(8, np.float32)
    oracle.kv_absmax_update(x, rm)
    assert np.array_equal(rm, np.abs(x).max(axis=(0, 2)))
    rm2 = np.zeros(8, np.float32)
    for t0 in range(0, 300, 70):                       # running max over prefill batches
        oracle.kv_absmax_update(x[t0:t0 + 70], rm2)
    assert np.array_equal(rm, rm2)


def test_running_max_keeps_previous_and_skips_nan():
    x = np.ones((4, 2, 128), np.float32)
    x[1, 0, 5] = np.nan
    x[2, 1, 7] = -9.5
    rm = np.array([3.0, 1.0], np.float32)              # previous batches saw up to 3.0 on head 0
    oracle.kv_absmax_update(x, rm)
    assert list(rm) == [3.0, 9.5]


def test_bf16_rows_widen_exactly():
    x = (torch.randn(50, 4, 128) * 7).to(torch.bfloat16)
    rm_a = np.zeros(4, np.float32)
    rm_b = np.zeros(4, np.float32)
    oracle.kv_absmax_update(x.view(torch.uint16).numpy(), rm_a)
    oracle.kv_absmax_update(x.float().numpy(), rm_b)
    assert np.array_equal(rm_a, rm_b)


def test_scale_recipe():
    rm = np.array([448.0, 896.0, 0.0, 1e-10, 3.0], np.float32)
    s = oracle.kv_scale_from_max(rm)
    assert s[0] == 1.0 and s[1] == 2.0                 # absmax / 448
    assert s[2] == np.float32(1e-12)                   # the clamp(min=1e-12) floor
    assert s[3] == np.float32(1e-12)                   # 1e-10/448 < 1e-12
    assert s[4] == np.float32(np.float32(3.0) / np.float32(448.0))


def test_matches_workload_scales():
    """The workload generator's scale recipe (absmax/448 over the prefill) is
    what calibrating over the same prefill batches gives."""
    wl = workloads.config(0)
    ks, vs = wl.scales(0)
    rk = np.zeros(wl.hkv, np.float32)
    rv = np.zeros(wl.hkv, np.float32)
    for b, L in enumerate(wl.prefill_lens):
        oracle.kv_absmax_update(wl.kv_rows(0, 0, b, 0, L).numpy(), rk)
        oracle.kv_absmax_update(wl.kv_rows(0, 1, b, 0, L).numpy(), rv)
    assert np.array_equal(oracle.kv_scale_from_max(rk), ks.numpy())
    assert np.array_equal(oracle.kv_scale_from_max(rv), vs.numpy())

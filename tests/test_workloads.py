"""Checks of the seeded input generators and of the byte/page accounting
(CPU only).  The accounting is pinned to the sizes the pages print
(tests/golden/kv_cache_sizes.txt)."""
import os

import numpy as np
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_sizes.txt")


def _golden_rows():
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        yield line.split()


def test_kv_formula_matches_pages():
    seen = 0
    for row in _golden_rows():
        if row[0] != "kv_bytes":
            continue
        layers, kvh, hd, tokens, bpe = map(int, row[1:6])
        expected, tol = float(row[6]), float(row[7])
        wl = workloads.Workload(99, "acct", [tokens], 0, kvh * 8, kvh, 16)
        assert wl.head_dim == hd
        # kv_bytes counts FP8 (1 byte) per element for one layer
        total = wl.kv_bytes() * layers * bpe
        assert abs(total - expected) / expected <= tol, (tokens, total, expected)
        seen += 1
    assert seen == 2


def test_page_counts_match_pages():
    seen = 0
    for row in _golden_rows():
        if row[0] != "pages":
            continue
        tokens, P, expected = map(int, row[1:4])
        wl = workloads.Workload(99, "acct", [tokens], 0, 8, 8, P)
        assert wl.pages_per_seq == [expected]
        if expected * P == tokens:
            assert tokens % P == 0          # last page exactly full
        seen += 1
    assert seen == 2


def test_config_shapes():
    c = [workloads.config(i) for i in range(5)]
    assert c[0].seq_lens == [37, 100] and (c[0].hq, c[0].hkv, c[0].group) == (8, 1, 8)
    assert c[1].seq_lens == [4097] * 32 and (c[1].hq, c[1].hkv) == (32, 8)
    assert c[2].seq_lens == [16385] * 16 and (c[2].hq, c[2].hkv) == (64, 8)
    assert c[3].seq_lens == [127984] * 4 and c[3].pages_per_seq == [7999] * 4
    assert c[3].num_pages == int(np.ceil(4 * 7999 * 1.25))
    assert len(c[4].seq_lens) == 64 and c[4].layers == 80
    assert min(c[4].prefill_lens) >= 512 and max(c[4].prefill_lens) <= 131072
    assert workloads.config(4, page_size=32).page_size == 32


def test_block_table_is_a_partial_permutation():
    for i in (0, 1, 3):
        wl = workloads.config(i)
        bt = wl.block_table()
        used = []
        for b, n in enumerate(wl.pages_per_seq):
            assert (bt[b, :n] >= 0).all() and (bt[b, n:] == -1).all()
            used.append(bt[b, :n])
        used = torch.cat(used)
        assert used.unique().numel() == used.numel() == wl.needed_pages
        assert int(used.max()) < wl.num_pages
        assert not torch.equal(used, torch.arange(used.numel(), dtype=torch.int32))   # shuffled


def test_generator_is_deterministic_and_slice_consistent():
    wl = workloads.config(1)
    a = wl.kv_head_values(0, 0, 3, 5, 100, 300)
    b = wl.kv_head_values(0, 0, 3, 5, 0, 400)[100:300]
    assert torch.equal(a, b)
    c = wl.kv_rows(0, 1, 3, 10, 20)
    assert torch.equal(c[:, 5], wl.kv_head_values(0, 1, 3, 5, 10, 20))
    assert not torch.equal(wl.kv_head_values(0, 0, 3, 5, 0, 50), wl.kv_head_values(0, 1, 3, 5, 0, 50))
    assert torch.equal(wl.q(0, 0), workloads.config(1).q(0, 0))


def test_value_distribution():
    wl = workloads.config(2)
    x = wl.kv_head_values(0, 0, 0, 0, 0, 4096).flatten()
    sig = wl.sigma(0, 0, 0)
    assert 0.5 <= sig <= 2.0
    inl = x[(x.abs() <= 4.9 * sig)]
    frac_out = 1 - inl.numel() / x.numel()
    assert 0.0015 < frac_out < 0.006                       # ~0.5% outliers, most land outside
    assert abs(float(inl.std()) / sig - 1) < 0.05
    q = wl.q().float()
    assert abs(float(q.std()) - 1) < 0.02 and abs(float(q.mean())) < 0.02
    ks, vs = workloads.config(0).scales()
    assert (ks > 0).all() and (vs > 0).all()


def test_sigmas_vary_across_heads():
    wl = workloads.config(2)
    sig = [wl.sigma(0, w, h) for w in (0, 1) for h in range(8)]
    assert min(sig) >= 0.5 and max(sig) <= 2.0 and np.std(sig) > 0.1

"""Helpers for the GPU parity tests: build a workload's cache on the GPU
through kv_append_fp8, and compute expected rows with the CPU oracle from
inputs the generator makes on the host (never from GPU results)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import paged_fp8_kv_03_gb300 as pkv

TOL_MAX_ABS = 2e-3
TOL_REL_L2 = 1e-3


class Filled:
    pass


def step_tokens(wl, layer: int, dev):
    """The decode step's new K/V rows, [B, append, Hkv, D] each (fp32)."""
    A = wl.append
    k = torch.stack([wl.kv_rows(layer, 0, b, L, L + A, device=dev) for b, L in enumerate(wl.prefill_lens)])
    v = torch.stack([wl.kv_rows(layer, 1, b, L, L + A, device=dev) for b, L in enumerate(wl.prefill_lens)])
    return k.contiguous(), v.contiguous()


def fill_gpu(wl, layer: int, dev, chunk_tokens: int = 1 << 15, tail_fill: int = 0x7F,
             step_append: bool = True) -> Filled:
    """Prefill every sequence through kv_append_fp8 (chunked), then (unless
    step_append is False) run the decode step's own append as one batched call."""
    f = Filled()
    f.wl = wl
    f.layer = layer
    f.ks, f.vs = wl.scales(layer, device=dev)
    P, H, D = wl.page_size, wl.hkv, wl.head_dim
    f.kc = torch.full((wl.num_pages, H, P, D), tail_fill, dtype=torch.uint8, device=dev)
    f.vc = torch.full_like(f.kc, tail_fill)
    f.err = torch.zeros(1, dtype=torch.int32, device=dev)
    for b, L in enumerate(wl.prefill_lens):
        for t0 in range(0, L, chunk_tokens):
            t1 = min(L, t0 + chunk_tokens)
            k = wl.kv_rows(layer, 0, b, t0, t1, device=dev)
            v = wl.kv_rows(layer, 1, b, t0, t1, device=dev)
            pkv.kv_append_fp8(k, v, wl.slots(b, t0, t1).to(dev), f.ks, f.vs, f.kc, f.vc, f.err)
    if wl.append and step_append:
        ks, vs, sl = [], [], []
        for b, L in enumerate(wl.prefill_lens):
            ks.append(wl.kv_rows(layer, 0, b, L, L + wl.append, device=dev))
            vs.append(wl.kv_rows(layer, 1, b, L, L + wl.append, device=dev))
            sl.append(wl.slots(b, L, L + wl.append))
        pkv.kv_append_fp8(torch.cat(ks), torch.cat(vs), torch.cat(sl).to(dev), f.ks, f.vs, f.kc, f.vc, f.err)
    f.bt = wl.block_table().to(dev)
    f.lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
    f.q = wl.q(layer, 0, device=dev)
    # per-sequence page sizes (None: the pool page size) and the bound of seq_lens
    f.psz = torch.tensor(wl.page_sizes, dtype=torch.int32, device=dev) if wl.page_sizes is not None else None
    f.max_len = wl.max_len
    torch.cuda.synchronize()
    return f


def oracle_pages(wl, layer: int, b: int, h: int, ks_h: float, vs_h: float):
    """Oracle pools [num_pages, 1, P, D] holding sequence b's tokens of kv head h."""
    P, D = wl.page_size, wl.head_dim
    L = wl.seq_lens[b]
    kc = np.zeros((wl.num_pages, 1, P, D), np.uint8)
    vc = np.zeros_like(kc)
    slots = wl.slots(b, 0, L).numpy()
    k = wl.kv_head_values(layer, 0, b, h, 0, L).numpy()[:, None, :]
    v = wl.kv_head_values(layer, 1, b, h, 0, L).numpy()[:, None, :]
    oracle.kv_append(k, slots, np.array([ks_h], np.float32), kc)
    oracle.kv_append(v, slots, np.array([vs_h], np.float32), vc)
    return kc, vc


def oracle_rows(wl, layer: int, pairs, ks: np.ndarray, vs: np.ndarray, threads: int = 8) -> dict:
    """Expected fp64 output rows {(b, q_head): [D]} for the requested pairs."""
    G = wl.group
    q_bits = wl.q(layer, 0).view(torch.uint16).numpy()
    bt = wl.block_table().numpy()
    by_bh: dict = {}
    for b, i in pairs:
        by_bh.setdefault((b, i // G), []).append(i)
    out = {}
    for (b, h), heads in by_bh.items():
        kc, vc = oracle_pages(wl, layer, b, h, float(ks[h]), float(vs[h]))
        qg = np.ascontiguousarray(q_bits[b:b + 1, h * G:(h + 1) * G])
        sel = np.array([[0, i - h * G] for i in heads], np.int32)
        psz = np.array([wl.page_sizes[b]], np.int32) if wl.page_sizes is not None else None
        rows = oracle.paged_decode(qg, kc, vc, ks[h:h + 1], vs[h:h + 1], bt[b:b + 1],
                                   np.array([wl.seq_lens[b]], np.int32), sel=sel, threads=threads,
                                   seq_page_sizes=psz)
        for i, r in zip(heads, rows):
            out[(b, i)] = r
    return out


def errors(got: np.ndarray, ref: np.ndarray):
    diff = got.astype(np.float64) - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, ref, what=""):
    max_abs, rel = errors(got, ref)
    assert max_abs <= TOL_MAX_ABS and rel <= TOL_REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def sample_pairs(wl, n_bh: int, seed: int = 0):
    """A few (b, q_head) pairs: first, last and seeded random (b, kv head) groups, all their heads."""
    rng = np.random.default_rng(seed)
    bhs = {(0, 0), (wl.batch - 1, wl.hkv - 1)}
    while len(bhs) < min(n_bh, wl.batch * wl.hkv):
        bhs.add((int(rng.integers(wl.batch)), int(rng.integers(wl.hkv))))
    G = wl.group
    return [(b, h * G + g) for (b, h) in sorted(bhs) for g in range(G)]


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def sm_scale(D: int = 128) -> float:
    return 1.0 / math.sqrt(D)

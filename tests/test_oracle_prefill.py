"""Pins for the oracle's chunked-prefill attention (CPU only).

* brute force: dense causal attention in numpy over tokens in logical order,
  quantised with torch's float8 cast (no pages, no block table, no oracle code);
* a chunk of one query is exactly the decode oracle;
* ragged chunks (empty, one token, the whole sequence) and the L < n error.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.dense_ref import dequant_torch, quantize_torch

SM = 1.0 / math.sqrt(128.0)


def _fill(wl):
    ks, vs = wl.scales(0)
    kc = np.full((wl.num_pages, wl.hkv, wl.page_size, 128), 0x7F, np.uint8)   # NaN codes off the sequences
    vc = np.full_like(kc, 0x7F)
    dk, dv = [], []
    for b, L in enumerate(wl.seq_lens):
        sl = wl.slots(b, 0, L).numpy()
        k = wl.kv_rows(0, 0, b, 0, L)
        v = wl.kv_rows(0, 1, b, 0, L)
        oracle.kv_append(k.numpy(), sl, ks.numpy(), kc)
        oracle.kv_append(v.numpy(), sl, vs.numpy(), vc)
        dk.append(dequant_torch(quantize_torch(k, ks), ks))
        dv.append(dequant_torch(quantize_torch(v, vs), vs))
    return kc, vc, ks.numpy(), vs.numpy(), dk, dv


def _dense_causal(q, k, v, first):
    """q [n, Hq, D]; k, v [L, Hkv, D]; query c sits at position first + c and
    sees tokens 0 .. first + c."""
    n, Hq, D = q.shape
    G = Hq // k.shape[1]
    kr = np.repeat(k, G, axis=1)
    vr = np.repeat(v, G, axis=1)
    out = np.zeros((n, Hq, D))
    for c in range(n):
        p = first + c
        s = np.einsum("hd,lhd->hl", q[c], kr[:p + 1]) * SM
        s -= s.max(axis=1, keepdims=True)
        w = np.exp(s)
        w /= w.sum(axis=1, keepdims=True)
        out[c] = np.einsum("hl,lhd->hd", w, vr[:p + 1])
    return out


@pytest.mark.parametrize("chunks,page,sizes", [([5, 0, 3, 1], 16, None), ([40, 7, 3, 70], 32, None),
                                               ([40, 1, 0, 9], 64, None), ([40, 9, 3, 70], 16, [64, 16, 32, 64])])
def test_prefill_matches_dense_causal(chunks, page, sizes):
    wl = workloads.Workload(95, "prefill", [40, 70, 3, 70], 0, 8, 2, page, seed=9, page_sizes=sizes)
    kc, vc, ks, vs, dk, dv = _fill(wl)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = wl.q_rows(0, int(cu[-1]))
    lens = np.array(wl.seq_lens, np.int32)
    out = oracle.paged_prefill(q.view(torch.uint16).numpy(), cu, kc, vc, ks, vs, wl.block_table().numpy(), lens,
                               threads=4, seq_page_sizes=None if sizes is None else np.array(sizes, np.int32))
    for b, L in enumerate(wl.seq_lens):
        n = chunks[b]
        ref = _dense_causal(q[cu[b]:cu[b + 1]].double().numpy(), dk[b], dv[b], L - n)
        got = out[cu[b]:cu[b + 1]]
        assert np.max(np.abs(got - ref), initial=0.0) < 1e-12 * max(1.0, np.abs(ref).max(initial=0.0))
    # the first query of a whole-sequence chunk sees only token 0: its output is V[0] of its kv head
    for b, L in enumerate(wl.seq_lens):
        if chunks[b] == L:
            assert np.allclose(out[cu[b]], np.repeat(dv[b][0], 4, axis=0), rtol=0, atol=1e-12)


def test_single_query_chunk_is_decode():
    wl = workloads.Workload(96, "prefill1", [33, 90], 0, 16, 4, 32, seed=5)
    kc, vc, ks, vs, _, _ = _fill(wl)
    q = wl.q()
    bt = wl.block_table().numpy()
    lens = np.array(wl.seq_lens, np.int32)
    cu = np.arange(wl.batch + 1, dtype=np.int32)
    pre = oracle.paged_prefill(q.view(torch.uint16).numpy(), cu, kc, vc, ks, vs, bt, lens)
    sel = np.array([[b, i] for b in range(wl.batch) for i in range(wl.hq)], np.int32)
    dec = oracle.paged_decode(q.view(torch.uint16).numpy(), kc, vc, ks, vs, bt, lens, sel=sel)
    assert np.array_equal(pre.reshape(-1, 128), dec)


def test_chunk_longer_than_sequence_is_an_error():
    wl = workloads.Workload(97, "prefill2", [4], 0, 8, 1, 16, seed=1)
    kc, vc, ks, vs, _, _ = _fill(wl)
    q = wl.q_rows(0, 5)
    with pytest.raises(ValueError, match="status 3"):
        oracle.paged_prefill(q.view(torch.uint16).numpy(), np.array([0, 5], np.int32), kc, vc, ks, vs,
                             wl.block_table().numpy(), np.array([4], np.int32))

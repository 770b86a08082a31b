"""paged_prefill (chunked-prefill attention, tcgen05) on the GPU against the
fp64 oracle.

The cache is written by kv_append_fp8 on the GPU from the seeded generator;
the oracle builds its own pages from the same host inputs.  Tolerance (fp32
output): max-abs <= 2e-3 and relative L2 <= 1e-3 of the oracle's fp64
attention.  The bf16 output must equal the round-to-nearest-even bf16 of the
fp32 output bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_fill import assert_close, errors, fill_gpu

pytestmark = pytest.mark.gpu


def _cu(chunks):
    return np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)


def _psz_np(wl):
    return np.array(wl.page_sizes, np.int32) if wl.page_sizes is not None else None


def _oracle_pools(wl):
    ks, vs = wl.scales(0)
    shape = (wl.num_pages, wl.hkv, wl.page_size, wl.head_dim)
    kco = np.zeros(shape, np.uint8)
    vco = np.zeros(shape, np.uint8)
    for b, L in enumerate(wl.seq_lens):
        slots = wl.slots(b, 0, L).numpy()
        oracle.kv_append(wl.kv_rows(0, 0, b, 0, L).numpy(), slots, ks.numpy(), kco)
        oracle.kv_append(wl.kv_rows(0, 1, b, 0, L).numpy(), slots, vs.numpy(), vco)
    return kco, vco, ks.numpy(), vs.numpy()


def _prefill(pkv, f, q, cu, max_q_len, out_dtype=torch.float32, err=None, bt=None, lens=None, fill=float("nan"),
             max_total_kv=0):
    out = torch.full(q.shape, fill, dtype=out_dtype, device=q.device)
    pkv.paged_prefill(q, cu, f.kc, f.vc, f.ks, f.vs, f.bt if bt is None else bt, f.lens if lens is None else lens,
                      max_q_len, out=out, device_error=f.err if err is None else err, max_kv_len=f.max_len,
                      max_total_kv=max_total_kv, seq_page_sizes=f.psz)
    torch.cuda.synchronize()
    return out


def _run_case(pkv, dev, lens, chunks, hq, hkv, page, seed=31, sizes=None, max_total_kv=0):
    wl = workloads.Workload(60, "prefill", lens, 0, hq, hkv, page, pool_factor=1.5, seed=seed, page_sizes=sizes)
    f = fill_gpu(wl, 0, dev)
    cu = _cu(chunks)
    T = int(cu[-1])
    q = wl.q_rows(0, T)
    qd = q.to(dev)
    cud = torch.from_numpy(cu).to(dev)
    got = _prefill(pkv, f, qd, cud, max(chunks), max_total_kv=max_total_kv)
    assert int(f.err.item()) == 0
    kco, vco, ks, vs = _oracle_pools(wl)
    ref = oracle.paged_prefill(q.view(torch.uint16).numpy(), cu, kco, vco, ks, vs, wl.block_table().numpy(),
                               np.array(lens, np.int32), threads=8, seq_page_sizes=_psz_np(wl))
    ma, rel = assert_close(got.double().cpu().numpy(), ref, f"prefill {lens} {chunks} G={hq // hkv} P={page}")
    return wl, f, qd, cud, got, ma, rel


@pytest.mark.parametrize("lens,chunks,hq,hkv,page", [
    ([37, 100], [37, 100], 8, 1, 16),                  # whole sequences (first query sees one token)
    ([300, 129, 1000], [17, 129, 256], 64, 8, 16),     # G = 8: 16 tokens per tile, several key tiles
    ([1000, 5, 700], [333, 5, 1], 32, 8, 32),          # G = 4: 32 tokens per tile; one-token chunk
    ([513, 2049], [513, 100], 2, 2, 64),               # G = 1: 128 tokens per tile
    ([400, 257], [200, 0], 16, 8, 16),                 # G = 2, an empty chunk
    ([129, 260], [129, 33], 24, 8, 128),               # G = 3: 42 tokens per tile, 2 padding rows
    ([900, 64], [130, 64], 40, 8, 256),                # G = 5: 25 tokens per tile, 256-token pages
    ([255, 256, 257], [255, 128, 127], 56, 8, 32),     # G = 7: 18 tokens per tile
])
def test_prefill_matches_oracle(pkv, cuda_device, lens, chunks, hq, hkv, page):
    _run_case(pkv, cuda_device, lens, chunks, hq, hkv, page)


@pytest.mark.parametrize("lens,chunks,hq,hkv,sizes", [
    ([300, 129, 1000, 70], [17, 129, 256, 70], 64, 8, [64, 16, 256, 32]),
    ([9000, 700], [500, 700], 32, 8, [64, 16]),          # the notes' 16 / 64 split by length
])
def test_prefill_per_sequence_page_sizes(pkv, cuda_device, lens, chunks, hq, hkv, sizes):
    _run_case(pkv, cuda_device, lens, chunks, hq, hkv, 16, sizes=sizes)


def test_prefill_workspace_sized_by_total_length(pkv, cuda_device):
    """One long prompt chunk beside many short ones, with the workspace sized
    by the lengths' sum (not batch x longest): same rows as the default
    workspace, the oracle's within tolerance; a sum bound that is too small is
    reported and leaves the rows that do not fit unwritten."""
    lens = [4000] + [40 + 7 * i for i in range(15)]
    chunks = [1000] + [40 + 7 * i for i in range(15)]
    wl, f, q, cu, got, _, _ = _run_case(pkv, cuda_device, lens, chunks, 32, 8, 16, max_total_kv=sum(lens))
    small = pkv.pkv_prefill_workspace_size(len(lens), 8, f.max_len, sum(lens))
    big = pkv.pkv_prefill_workspace_size(len(lens), 8, f.max_len)
    assert small * 8 < big
    again = _prefill(pkv, f, q, cu, max(chunks))
    assert torch.equal(again, got)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = _prefill(pkv, f, q, cu, max(chunks), err=err, max_total_kv=1000, fill=5.0)
    assert int(err.item()) & pkv.DEVERR_SEQLEN
    assert torch.all(out == 5.0)                         # the long chunk's region alone exceeds the bound


def test_bf16_output_is_rounded_fp32_and_deterministic(pkv, cuda_device):
    wl, f, q, cu, got32, _, _ = _run_case(pkv, cuda_device, [700, 300], [300, 300], 64, 8, 16)
    again = _prefill(pkv, f, q, cu, 300)
    assert torch.equal(again, got32)
    got16 = _prefill(pkv, f, q, cu, 300, out_dtype=torch.bfloat16)
    assert torch.equal(got16, got32.to(torch.bfloat16))


def test_rows_outside_every_chunk_are_not_written(pkv, cuda_device):
    wl = workloads.Workload(61, "prefill", [90, 40], 0, 16, 2, 16, seed=3)
    f = fill_gpu(wl, 0, cuda_device)
    q = wl.q_rows(0, 80).to(cuda_device)
    cu = torch.tensor([0, 30, 60], dtype=torch.int32, device=cuda_device)      # rows 60..79 belong to nobody
    out = _prefill(pkv, f, q, cu, 30, fill=7.0)
    assert torch.all(out[60:] == 7.0)
    assert torch.isfinite(out[:60]).all()


def test_one_query_chunks_equal_decode(pkv, cuda_device):
    """A chunk of one query per sequence is one decode step: both GPU paths
    agree within the oracle tolerance (their arithmetic differs)."""
    wl = workloads.Workload(62, "prefill", [1, 200, 4097, 33], 0, 64, 8, 16, seed=8)
    f = fill_gpu(wl, 0, cuda_device)
    cu = torch.arange(wl.batch + 1, dtype=torch.int32, device=cuda_device)
    pre = _prefill(pkv, f, f.q, cu, 1)
    dec = pkv.paged_gqa_decode(f.q, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out_dtype=torch.float32)
    torch.cuda.synchronize()
    d = (pre.double() - dec.double()).abs().max().item()
    assert d <= 2e-3, d


def test_explicit_bounds_and_workspace(pkv, cuda_device):
    """max_kv_len as the real bound (a tight workspace) gives the same rows
    as the default bound; a sequence above max_kv_len is reported, not read."""
    wl = workloads.Workload(65, "prefill", [300, 129], 0, 32, 8, 16, seed=6)
    f = fill_gpu(wl, 0, cuda_device)
    q = wl.q_rows(0, 100).to(cuda_device)
    cu = torch.tensor([0, 60, 100], dtype=torch.int32, device=cuda_device)
    ref = _prefill(pkv, f, q, cu, 60)
    ws = torch.full((pkv.pkv_prefill_workspace_size(2, 8, 300),), 0xFF, dtype=torch.uint8, device=cuda_device)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_device)
    pkv.pkv_paged_prefill(q, cu, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out, 60, 300, ws, device_error=f.err)
    torch.cuda.synchronize()
    assert int(f.err.item()) == 0
    assert torch.equal(out, ref)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.pkv_paged_prefill(q, cu, f.kc, f.vc, f.ks, f.vs, f.bt, f.lens, out, 60, 299,
                          torch.empty(pkv.pkv_prefill_workspace_size(2, 8, 299), dtype=torch.uint8,
                                      device=cuda_device), device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_SEQLEN


def test_error_bits(pkv, cuda_device):
    wl = workloads.Workload(63, "prefill", [50, 40], 0, 16, 2, 16, seed=4)
    f = fill_gpu(wl, 0, cuda_device)
    q = wl.q_rows(0, 60).to(cuda_device)
    cu = torch.tensor([0, 20, 60], dtype=torch.int32, device=cuda_device)
    # a chunk longer than its sequence (40 queries, 40 tokens is fine; 41 is not)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    lens = torch.tensor([50, 39], dtype=torch.int32, device=cuda_device)
    out = _prefill(pkv, f, q, cu, 40, err=err, lens=lens, fill=5.0)
    assert int(err.item()) & pkv.DEVERR_SEQLEN
    assert torch.all(out[20:] == 5.0)                 # that sequence's rows are not written
    # chunk longer than max_q_len
    err.zero_()
    _prefill(pkv, f, q, cu, 39, err=err)
    assert int(err.item()) & pkv.DEVERR_SEQLEN
    # a block-table entry outside the pool
    err.zero_()
    bt = f.bt.clone()
    bt[0, 1] = wl.num_pages + 5
    _prefill(pkv, f, q, cu, 40, err=err, bt=bt)
    assert int(err.item()) & pkv.DEVERR_PAGE


def _sampled_rows(wl, q_bits, cu, rows_heads, threads=16):
    """Oracle rows {(row, q_head): [D]} for sampled query rows at full size,
    each through the decode oracle over a pool holding one (sequence, kv head)."""
    G = wl.group
    bt = wl.block_table().numpy()
    out = {}
    groups = {}
    for r, i in rows_heads:
        b = int(np.searchsorted(cu, r, side="right") - 1)
        groups.setdefault((b, i // G), []).append((r, i))
    ks, vs = wl.scales(0)
    ks, vs = ks.numpy(), vs.numpy()
    for (b, h), items in groups.items():
        L = wl.seq_lens[b]
        kc = np.zeros((wl.num_pages, 1, wl.page_size, wl.head_dim), np.uint8)
        vc = np.zeros_like(kc)
        slots = wl.slots(b, 0, L).numpy()
        oracle.kv_append(wl.kv_head_values(0, 0, b, h, 0, L).numpy()[:, None, :], slots, ks[h:h + 1], kc)
        oracle.kv_append(wl.kv_head_values(0, 1, b, h, 0, L).numpy()[:, None, :], slots, vs[h:h + 1], vc)
        n = int(cu[b + 1] - cu[b])
        for r, i in items:
            pos = L - n + (r - int(cu[b]))
            qg = np.ascontiguousarray(q_bits[r:r + 1, h * G:(h + 1) * G])
            row = oracle.paged_decode(qg, kc, vc, ks[h:h + 1], vs[h:h + 1], bt[b:b + 1],
                                      np.array([pos + 1], np.int32), sel=np.array([[0, i - h * G]], np.int32),
                                      threads=threads)
            out[(r, i)] = row[0]
    return out


def test_full_size_last_16k_chunk_of_128k_sampled(pkv, cuda_device):
    """Llama-3-70B attention geometry (64 query heads, 8 kv heads): the last
    16K chunk of a 128K prompt, checked on sampled rows spread over the chunk
    (first, last, and rows near key-tile and query-tile boundaries)."""
    L, n = 131072, 16384
    wl = workloads.Workload(64, "prefill-128k", [L], 0, 64, 8, 16, seed=12)
    f = fill_gpu(wl, 0, cuda_device)
    cu = np.array([0, n], np.int32)
    q = wl.q_rows(0, n)
    out = _prefill(pkv, f, q.to(cuda_device), torch.from_numpy(cu).to(cuda_device), n)
    assert int(f.err.item()) == 0
    rows = [0, 1, 15, 16, 127, 128, 8191, n - 2, n - 1]
    rng = np.random.default_rng(5)
    rows_heads = [(r, int(rng.integers(64))) for r in rows] + [(n - 1, 0), (n - 1, 63), (0, 7)]
    ref = _sampled_rows(wl, q.view(torch.uint16).numpy(), cu, rows_heads)
    got = out.cpu().numpy()
    for (r, i), row in ref.items():
        assert_close(got[r, i][None], row[None], f"row {r} head {i}")
    # The tensor cores' fp32 accumulation rounds toward zero; one accumulator
    # chained over the whole 128K context drifted to max-abs 1.1e-3 on these
    # inputs.  Folding it every 32 key tiles keeps the drift under 1e-4, well
    # inside the bound above: hold the kernel to that.
    max_abs, rel = errors(np.stack([got[r, i] for (r, i) in ref]), np.stack(list(ref.values())))
    print(f"prefill, last 16K chunk of a 128K prompt: max_abs {max_abs:.3e} rel_l2 {rel:.3e}")
    assert max_abs <= 3e-4, max_abs
    assert torch.isfinite(out).all()


def test_maximum_jumps_at_fold_tiles(pkv, cuda_device):
    """The running maximum of every row jumps by more than 2^8 (log2 units) at
    key tiles 16 and 32, where the segment accumulator is also folded into O
    (fold and rescale in one step), and at tile 40, between folds (both
    accumulators rescaled).  Only 8 keys carry each jump, so the earlier keys
    keep a visible share of the softmax and a wrong factor on either
    accumulator would show.  Rows of the chunk sit before, between and after
    the jumps; a second, short sequence makes the batch ragged."""
    Hq, Hkv, D, P = 16, 2, 128, 16
    lens, chunks = [6221, 300], [3200, 40]
    g = torch.Generator().manual_seed(77)
    K = [torch.randn(L, Hkv, D, generator=g) for L in lens]
    V = [torch.randn(L, Hkv, D, generator=g) for L in lens]
    # q . k / sqrt(D) is ~ K[t, h, 0] / sqrt(D): 0 for every key but the jumps
    # (E4M3 codes 144, 288, 448 of the scale absmax/448: about 9.8, 19.7 and
    # 30.6 in log2 units)
    K[0][:, :, 0] = 0.0
    for t0, val in [(2048, 80.0), (4096, 160.0), (5120, 240.0)]:
        K[0][t0:t0 + 8, :, 0] = val
    ks = torch.clamp(torch.stack([k.abs().amax(dim=(0, 2)) for k in K]).amax(0) / 448.0, min=1e-12).float()
    vs = torch.clamp(torch.stack([v.abs().amax(dim=(0, 2)) for v in V]).amax(0) / 448.0, min=1e-12).float()
    pages = [(L + P - 1) // P for L in lens]
    num_pages = sum(pages) + 3
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = torch.zeros(len(lens), max(pages), dtype=torch.int32)
    o = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[o:o + n]
        o += n
    slots = [bt[b].to(torch.int64)[torch.arange(L) // P] * P + torch.arange(L) % P for b, L in enumerate(lens)]
    T = sum(chunks)
    q = torch.zeros(T, Hq, D)
    q[:, :, 0] = 1.0
    q[:, :, 1:] = 0.01 * torch.randn(T, Hq, D - 1, generator=g)
    q = q.to(torch.bfloat16)
    cu = np.array([0, chunks[0], T], np.int32)

    dev = cuda_device
    kc = torch.zeros(num_pages, Hkv, P, D, dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for b in range(len(lens)):
        pkv.kv_append_fp8(K[b].to(dev), V[b].to(dev), slots[b].to(dev), ks.to(dev), vs.to(dev), kc, vc, err)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.float32, device=dev)
    pkv.paged_prefill(q.to(dev), torch.from_numpy(cu).to(dev), kc, vc, ks.to(dev), vs.to(dev), bt.to(dev), lens_d,
                      max(chunks), out=out, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    kco = np.zeros((num_pages, Hkv, P, D), np.uint8)
    vco = np.zeros_like(kco)
    for b in range(len(lens)):
        oracle.kv_append(K[b].numpy(), slots[b].numpy(), ks.numpy(), kco)
        oracle.kv_append(V[b].numpy(), slots[b].numpy(), vs.numpy(), vco)
    assert np.array_equal(kc.cpu().numpy(), kco) and np.array_equal(vc.cpu().numpy(), vco)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    # Sampled rows, each through the decode oracle at its own causal length:
    # the long chunk covers positions 3021 .. 6220, so rows sit before, on
    # and after the jumps at 4096 and 5120; every row of the short sequence.
    q_bits = q.view(torch.uint16).numpy()
    rng = np.random.default_rng(3)
    pos = [3021, 3500, 4095, 4096, 4103, 4104, 4500, 5119, 5120, 5127, 5128, 6000, 6220]
    rows = [(0, p_ - (lens[0] - chunks[0])) for p_ in pos] + [(0, int(r)) for r in rng.integers(0, chunks[0], 8)]
    rows += [(1, chunks[0] + c) for c in range(chunks[1])]
    exp, act = [], []
    for b, r in rows:
        p_ = lens[b] - chunks[b] + (r - int(cu[b]))
        ref = oracle.paged_decode(np.ascontiguousarray(q_bits[r:r + 1]), kco, vco, ks.numpy(), vs.numpy(),
                                  bt[b:b + 1].numpy(), np.array([p_ + 1], np.int32), threads=8)
        exp.append(ref.reshape(Hq, D))         # rows (0, head 0 .. Hq-1)
        act.append(got[r])
    assert_close(np.stack(act), np.stack(exp), "maximum jumps at fold tiles")

"""Seeded synthetic inputs for the paged FP8-KV decode path.

This module is shared by the tests, the benchmark and the oracle side.  It
holds no step of the method itself (no quantisation, no attention): only the
recipe that makes inputs.

Every random value comes from a counter-based integer hash evaluated with
torch integer ops, followed by a fixed sequence of IEEE fp32 operations.  The
same call therefore gives bit-identical tensors on the CPU and on a GPU, so the
GPU side can build a 128K-token cache in milliseconds while the oracle side
regenerates, on the host, exactly the (sequence, kv-head) slices it checks.

Value recipe (shapes and distributions of the Llama-3 workloads):
  * K, V: fp32 ~ N(0, sigma) with sigma ~ U(0.5, 2) drawn per (layer, kv head,
    K or V); each element is multiplied by 8 with probability 0.005
    (outliers).  The normal is approximated by the sum of 8 independent
    uniform bytes (Irwin-Hall, 8 terms), centred and scaled to unit variance:
    bounded at about +-4.9 sigma before the outlier factor.
  * Q: the same unit normal, rounded to bf16 (RNE).
  * scale per (layer, kv head, K or V) = max(absmax / 448, 1e-12) over the
    tokens present before the decode step (absmax/448 as in the Llama-3 FP8
    weight recipe; the 1e-12 floor from the same code).
  * Block tables: physical pages are a seeded random permutation of the pool
    (a fragmented pool of 1.25x the needed pages for the long-context case).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

M32 = 0xFFFFFFFF
_MUL = 0x045D9F3B          # < 2^31, so x * _MUL never leaves int64 for x < 2^32
HEAD_DIM = 128


# --------------------------------------------------------------------------
# counter-based hash
# --------------------------------------------------------------------------
def _mix32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * _MUL) & M32
    x ^= x >> 16
    x = (x * _MUL) & M32
    x ^= x >> 16
    return x


def stream_key(*parts: int) -> int:
    """32-bit key of a named random stream (all parts non-negative ints)."""
    k = 0x9E3779B9
    for p in parts:
        k = _mix32_int(k ^ _mix32_int(int(p) + 0x632BE5AB))
    return k


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """Same finaliser as _mix32_int on an int64 tensor holding 32-bit values."""
    x = x ^ (x >> 16)
    x = (x * _MUL) & M32
    x = x ^ (x >> 16)
    x = (x * _MUL) & M32
    x = x ^ (x >> 16)
    return x


def hash_u32(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Uniform 32-bit values for counters `idx` (int64) in stream `key`."""
    return _mix32((idx ^ key) & M32)


def _byte_sum(h: torch.Tensor) -> torch.Tensor:
    return (h & 255) + ((h >> 8) & 255) + ((h >> 16) & 255) + ((h >> 24) & 255)


# sqrt(8 * (256^2 - 1) / 12): standard deviation of a sum of 8 uniform bytes
_IH_SD = math.sqrt(8.0 * (256.0 * 256.0 - 1.0) / 12.0)


def unit_normal(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Approximately N(0, 1) fp32 values, bit-identical on every device."""
    s = _byte_sum(hash_u32(stream_key(key, 1), idx)) + _byte_sum(hash_u32(stream_key(key, 2), idx))
    centred = (s - 1020).to(torch.float32)          # exact: |s - 1020| <= 1020
    inv_sd = torch.tensor(1.0 / _IH_SD, dtype=torch.float32, device=idx.device)
    return centred * inv_sd


def outlier_mask(key: int, idx: torch.Tensor, prob: float = 0.005) -> torch.Tensor:
    thresh = int(round(prob * 65536.0))
    return (hash_u32(stream_key(key, 3), idx) & 0xFFFF) < thresh


def uniform01(key: int) -> float:
    """One uniform number in (0, 1) for a stream (host-side scalar)."""
    return (_mix32_int(key) + 0.5) / 4294967296.0


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------
@dataclass
class Workload:
    """One decode-step workload.

    prefill_lens[b] tokens are in the cache before the step; the step appends
    `append` tokens per sequence and then attends seq_lens[b] =
    prefill_lens[b] + append tokens with one query per sequence.
    """
    index: int
    name: str
    prefill_lens: list
    append: int
    hq: int
    hkv: int
    page_size: int
    layers: int = 1
    pool_factor: float = 1.0
    seed: int = 0
    head_dim: int = HEAD_DIM
    notes: str = ""
    page_sizes: list | None = None      # tokens per page of each sequence (runs of pool pages); None: page_size
    _bt: torch.Tensor | None = field(default=None, repr=False)

    @property
    def batch(self) -> int:
        return len(self.prefill_lens)

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def seq_lens(self) -> list:
        return [l + self.append for l in self.prefill_lens]

    def seq_page_size(self, b: int) -> int:
        return self.page_sizes[b] if self.page_sizes is not None else self.page_size

    @property
    def pages_per_seq(self) -> list:
        """Block-table entries (logical pages of P_b tokens) of every sequence."""
        return [(l + self.seq_page_size(b) - 1) // self.seq_page_size(b) for b, l in enumerate(self.seq_lens)]

    @property
    def max_pages(self) -> int:
        return max(1, max(self.pages_per_seq))

    @property
    def max_len(self) -> int:
        """Capacity of a table row at the largest page size (a bound of seq_lens)."""
        return self.max_pages * max(self.seq_page_size(b) for b in range(self.batch))

    @property
    def needed_pages(self) -> int:
        """Pool pages the sequences occupy (a P_b-token page is P_b / P pool pages)."""
        P = self.page_size
        return sum(n * (self.seq_page_size(b) // P) for b, n in enumerate(self.pages_per_seq))

    def _groups(self):
        """Variable page sizes: the pool is cut into groups of R = max P_b / P
        consecutive pages; for every ratio r = P_b / P the number of groups its
        runs of r pages need."""
        P = self.page_size
        R = max(self.seq_page_size(b) for b in range(self.batch)) // P
        need = {}
        for b, n in enumerate(self.pages_per_seq):
            r = self.seq_page_size(b) // P
            need[r] = need.get(r, 0) + n
        return R, {r: (n * r + R - 1) // R for r, n in need.items()}

    @property
    def num_pages(self) -> int:
        if self.page_sizes is None:
            return max(1, int(math.ceil(self.needed_pages * self.pool_factor)))
        R, groups = self._groups()
        return R * max(1, int(math.ceil(sum(groups.values()) * self.pool_factor)))

    def _perm(self, n: int, salt: int) -> torch.Tensor:
        h = hash_u32(stream_key(self.seed, self.index, 77, salt) if salt else stream_key(self.seed, self.index, 77),
                     torch.arange(n, dtype=torch.int64))
        return torch.argsort(h * n + torch.arange(n), stable=True)   # ties impossible

    def block_table(self) -> torch.Tensor:
        """int32 [B, max_pages] on the CPU; unused entries are -1.  With
        per-sequence page sizes an entry is the first pool page of a run of
        P_b / P consecutive pool pages."""
        if self._bt is None:
            bt = torch.full((self.batch, self.max_pages), -1, dtype=torch.int32)
            if self.page_sizes is None:
                n = self.num_pages
                perm = self._perm(n, 0)
                pos = 0
                for b, np_b in enumerate(self.pages_per_seq):
                    bt[b, :np_b] = perm[pos:pos + np_b].to(torch.int32)
                    pos += np_b
            else:
                P = self.page_size
                R, groups = self._groups()
                gperm = self._perm(self.num_pages // R, 0)          # groups in random pool order
                gpos = 0
                runs = {}
                for r in sorted(groups, reverse=True):
                    g = gperm[gpos:gpos + groups[r]]
                    gpos += groups[r]
                    starts = (g.view(-1, 1) * R + torch.arange(0, R, r).view(1, -1)).reshape(-1)
                    runs[r] = starts[self._perm(starts.numel(), r)]   # runs of r pages in random order
                used = {r: 0 for r in runs}
                for b, np_b in enumerate(self.pages_per_seq):
                    r = self.seq_page_size(b) // P
                    bt[b, :np_b] = runs[r][used[r]:used[r] + np_b].to(torch.int32)
                    used[r] += np_b
            self._bt = bt
        return self._bt

    def slots(self, b: int, t0: int, t1: int) -> torch.Tensor:
        """int64 cache slots of tokens t0..t1-1 of sequence b (CPU): the table
        entry of the token's logical page times P plus its offset in that page
        (a P_b-token page spans P_b / P consecutive pool pages)."""
        P, Pb = self.page_size, self.seq_page_size(b)
        t = torch.arange(t0, t1, dtype=torch.int64)
        pages = self.block_table()[b].to(torch.int64)[t // Pb]
        return pages * P + t % Pb

    # ---------------- values ----------------
    def _kv_key(self, layer: int, which: int, b: int, h: int) -> int:
        return stream_key(self.seed, self.index, layer, which, b, h)

    def sigma(self, layer: int, which: int, h: int) -> float:
        """Per-(layer, kv head, K/V) spread, U(0.5, 2), as an fp32-exact float."""
        u = uniform01(stream_key(self.seed, self.index, layer, which, h, 991))
        return float(torch.tensor(0.5 + 1.5 * u, dtype=torch.float32))

    def kv_head_values(self, layer: int, which: int, b: int, h: int, t0: int, t1: int,
                       device="cpu") -> torch.Tensor:
        """fp32 [t1 - t0, D] values of K (which=0) or V (which=1), one kv head."""
        D = self.head_dim
        idx = torch.arange(t0 * D, t1 * D, dtype=torch.int64, device=device)
        key = self._kv_key(layer, which, b, h)
        z = unit_normal(key, idx)
        sig = torch.tensor(self.sigma(layer, which, h), dtype=torch.float32, device=device)
        x = z * sig
        eight = torch.tensor(8.0, dtype=torch.float32, device=device)
        x = torch.where(outlier_mask(key, idx), x * eight, x)
        return x.view(t1 - t0, D)

    def kv_rows(self, layer: int, which: int, b: int, t0: int, t1: int, device="cpu") -> torch.Tensor:
        """fp32 [t1 - t0, Hkv, D]: the rows kv_append_fp8 takes for these tokens."""
        return torch.stack([self.kv_head_values(layer, which, b, h, t0, t1, device)
                            for h in range(self.hkv)], dim=1).contiguous()

    def q(self, layer: int = 0, step: int = 0, device="cpu") -> torch.Tensor:
        """bf16 [B, Hq, D] queries of one decode step."""
        B, Hq, D = self.batch, self.hq, self.head_dim
        idx = torch.arange(B * Hq * D, dtype=torch.int64, device=device)
        z = unit_normal(stream_key(self.seed, self.index, layer, 5, step), idx)
        return z.to(torch.bfloat16).view(B, Hq, D)

    def q_rows(self, layer: int, rows: int, step: int = 0, device="cpu") -> torch.Tensor:
        """bf16 [rows, Hq, D] queries of a prefill chunk (the chunks of all
        sequences back to back), drawn like q() from their own stream."""
        Hq, D = self.hq, self.head_dim
        idx = torch.arange(rows * Hq * D, dtype=torch.int64, device=device)
        z = unit_normal(stream_key(self.seed, self.index, layer, 6, step), idx)
        return z.to(torch.bfloat16).view(rows, Hq, D)

    def scales(self, layer: int = 0, device="cpu") -> tuple:
        """(k_scale, v_scale), fp32 [Hkv] each: max(absmax/448, 1e-12) per kv
        head over the prefill tokens of every sequence."""
        out = []
        for which in (0, 1):
            s = torch.zeros(self.hkv, dtype=torch.float32, device=device)
            for h in range(self.hkv):
                m = torch.zeros((), dtype=torch.float32, device=device)
                for b, L in enumerate(self.prefill_lens):
                    step = 1 << 16
                    for t0 in range(0, L, step):
                        v = self.kv_head_values(layer, which, b, h, t0, min(L, t0 + step), device)
                        m = torch.maximum(m, v.abs().max())
                s[h] = m
            d448 = torch.tensor(448.0, dtype=torch.float32, device=device)
            floor = torch.tensor(1e-12, dtype=torch.float32, device=device)
            out.append(torch.maximum(s / d448, floor))
        return tuple(out)

    # ---------------- accounting ----------------
    def kv_bytes(self) -> int:
        """FP8 K+V bytes one decode pass reads per layer: sum_b L_b * Hkv * 2 * D."""
        return sum(self.seq_lens) * self.hkv * 2 * self.head_dim

    def describe(self) -> dict:
        extra = {}
        if self.page_sizes is not None:
            extra = {"seq_page_sizes": {str(p): sum(1 for b in range(self.batch) if self.seq_page_size(b) == p)
                                        for p in sorted(set(self.page_sizes))}}
        return {"workload": self.name, "batch": self.batch, "hq": self.hq, "hkv": self.hkv,
                "head_dim": self.head_dim, "page_size": self.page_size, **extra,
                "seq_len_min": min(self.seq_lens), "seq_len_max": max(self.seq_lens),
                "sum_seq_len": sum(self.seq_lens), "layers": self.layers,
                "append_per_seq": self.append, "pool_pages": self.num_pages}


def _log_uniform_lens(seed: int, n: int, lo: int, hi: int) -> list:
    out = []
    for b in range(n):
        u = uniform01(stream_key(seed, 4, b, 313))
        out.append(int(math.floor(lo * (hi / lo) ** u)))
    return [min(max(l, lo), hi) for l in out]


def dynamic_page_sizes(lens: list, short: int = 16, long: int = 64, long_from: int = 8192) -> list:
    """Per-sequence page sizes by length: `long`-token pages for sequences
    longer than long_from tokens, `short`-token pages otherwise (the Llama 3
    production notes' dynamic page size: 16-token pages below 1024 tokens,
    64-token pages above 8192; between the two they give no size, and the
    default 16 is kept)."""
    return [long if l > long_from else short for l in lens]


def config(i: int, page_size: int | None = None, seed: int = 0, dynamic_pages: bool = False) -> Workload:
    """The five decode workloads (tiny parity case, Llama-3 8B and 70B layer
    shapes, 128K long context, mixed serving batch).  dynamic_pages (mixed
    batch only): 16-token pool pages, 64-token pages for sequences above 8192
    tokens."""
    if dynamic_pages:
        if i != 4:
            raise ValueError("dynamic page sizes are defined for the mixed serving batch")
        lens = _log_uniform_lens(seed, 64, 512, 131072)
        return Workload(4, "mixed_b64_loguniform_512_131072_p16_64dyn", lens, 1, 64, 8, 16, layers=80, seed=seed,
                        page_sizes=dynamic_page_sizes([l + 1 for l in lens]),
                        notes="log-uniform lengths, 80 layers per step, 64-token pages above 8192 tokens")
    if i == 0:
        return Workload(0, "tiny_b2_l37_100_g8", [37, 100], 0, 8, 1, page_size or 16, seed=seed,
                        notes="shuffled block table, no append")
    if i == 1:
        return Workload(1, "llama3_8b_b32_l4096", [4096] * 32, 1, 32, 8, page_size or 16, seed=seed,
                        notes="random physical-page permutation, 1 appended token per sequence")
    if i == 2:
        return Workload(2, "llama3_70b_b16_l16384", [16384] * 16, 1, 64, 8, page_size or 16, seed=seed,
                        notes="1 appended token per sequence")
    if i == 3:
        return Workload(3, "llama3_70b_b4_l127984", [127984] * 4, 0, 64, 8, page_size or 16,
                        pool_factor=1.25, seed=seed,
                        notes="fragmented pool (1.25x pages, random subset and order), no append")
    if i == 4:
        P = page_size or 16
        lens = _log_uniform_lens(seed, 64, 512, 131072)
        return Workload(4, f"mixed_b64_loguniform_512_131072_p{P}", lens, 1, 64, 8, P, layers=80,
                        seed=seed, notes="log-uniform lengths, 80 layers per step")
    raise ValueError(f"no workload {i}")


def prefill_config(page_size: int | None = None, seed: int = 0, prompt: int = 131072, chunk: int = 16384,
                   batch: int = 1):
    """The chunked-prefill workload: `batch` prompts of `prompt` tokens on the
    Llama-3-70B attention geometry (64 query heads, 8 kv heads), prefilled in
    chunks of `chunk` tokens (128K as 8 x 16K by default).  Returns
    (workload, chunk); workload.seq_lens are the full prompt lengths."""
    if prompt % chunk:
        raise ValueError("the prompt must be a whole number of chunks")
    return (Workload(10, f"prefill_llama3_70b_b{batch}_{prompt // 1024}k_as_{prompt // chunk}x{chunk // 1024}k",
                     [prompt] * batch, 0, 64, 8, page_size or 16, seed=seed,
                     notes="chunked prefill: each chunk is appended, then its queries attend causally"),
            chunk)


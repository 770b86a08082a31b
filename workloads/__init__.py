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

    @property
    def pages_per_seq(self) -> list:
        P = self.page_size
        return [(l + P - 1) // P for l in self.seq_lens]

    @property
    def max_pages(self) -> int:
        return max(1, max(self.pages_per_seq))

    @property
    def needed_pages(self) -> int:
        return sum(self.pages_per_seq)

    @property
    def num_pages(self) -> int:
        return max(1, int(math.ceil(self.needed_pages * self.pool_factor)))

    def block_table(self) -> torch.Tensor:
        """int32 [B, max_pages] on the CPU; unused entries are -1."""
        if self._bt is None:
            n = self.num_pages
            h = hash_u32(stream_key(self.seed, self.index, 77), torch.arange(n, dtype=torch.int64))
            perm = torch.argsort(h * n + torch.arange(n), stable=True)   # ties impossible
            bt = torch.full((self.batch, self.max_pages), -1, dtype=torch.int32)
            pos = 0
            for b, np_b in enumerate(self.pages_per_seq):
                bt[b, :np_b] = perm[pos:pos + np_b].to(torch.int32)
                pos += np_b
            self._bt = bt
        return self._bt

    def slots(self, b: int, t0: int, t1: int) -> torch.Tensor:
        """int64 cache slots of tokens t0..t1-1 of sequence b (CPU)."""
        P = self.page_size
        t = torch.arange(t0, t1, dtype=torch.int64)
        pages = self.block_table()[b].to(torch.int64)[t // P]
        return pages * P + t % P

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
        return {"workload": self.name, "batch": self.batch, "hq": self.hq, "hkv": self.hkv,
                "head_dim": self.head_dim, "page_size": self.page_size,
                "seq_len_min": min(self.seq_lens), "seq_len_max": max(self.seq_lens),
                "sum_seq_len": sum(self.seq_lens), "layers": self.layers,
                "append_per_seq": self.append, "pool_pages": self.num_pages}


def _log_uniform_lens(seed: int, n: int, lo: int, hi: int) -> list:
    out = []
    for b in range(n):
        u = uniform01(stream_key(seed, 4, b, 313))
        out.append(int(math.floor(lo * (hi / lo) ** u)))
    return [min(max(l, lo), hi) for l in out]


def config(i: int, page_size: int | None = None, seed: int = 0) -> Workload:
    """The five decode workloads (tiny parity case, Llama-3 8B and 70B layer
    shapes, 128K long context, mixed serving batch)."""
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


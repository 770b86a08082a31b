"""Brute-force dense attention used to pin the paged oracle.

Independent of the oracle: quantisation and dequantisation go through
torch's own float8_e4m3fn cast (a library routine), tokens are taken in
logical order straight from the generator (no pages, no block table), and
the GQA head map is numpy's repeat (query head i -> kv head i // G).
"""
import numpy as np
import torch


def quantize_torch(x: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    """fp32 [..., Hkv, D] -> uint8 codes: torch division by the per-head scale,
    clamp to the E4M3 range, torch's RNE cast."""
    y = x / scale.view(*([1] * (x.dim() - 2)), -1, 1)
    y = torch.clamp(y, -448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def dequant_torch(codes: torch.Tensor, scale: torch.Tensor) -> np.ndarray:
    v = codes.view(torch.float8_e4m3fn).to(torch.float64)
    return (v * scale.to(torch.float64).view(*([1] * (codes.dim() - 2)), -1, 1)).numpy()


def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    """q [Hq, D], k/v [L, Hkv, D] (fp64) -> o [Hq, D]."""
    Hq, D = q.shape
    L, Hkv, _ = k.shape
    G = Hq // Hkv
    if L == 0:
        return np.zeros((Hq, D))
    kr = np.repeat(k, G, axis=1)          # [L, Hq, D]
    vr = np.repeat(v, G, axis=1)
    s = np.einsum("hd,lhd->hl", q, kr) * sm_scale
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return np.einsum("hl,lhd->hd", w, vr)

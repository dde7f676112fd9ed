"""Shared helpers for the GPU-vs-oracle parity tests (test code only).

Tolerances, derived from the arithmetic:
  - routing indices, counts, offsets, row map, receive rows, FP8 bytes and
    scales, source ids: bit-exact (integer / byte work, and the FP8 code is
    decided by one fp32 division on both sides).
  - gate weights: the kernel computes in fp32, the oracle in binary64; u =
    2^-24.  Score-normalised: a sum of k positive terms ((k-1) roundings)
    and one division, within k u relative.  Softmax over the top k: each
    exp(v - max) carries the fp32 subtraction's error (at most d u in the
    exponent, d the distance of v from the maximum) and expf's (<= 2 ulp,
    4 u), in the numerator and, averaged, in the sum; then k - 1 additions
    and one division: 2 (d + 4) u + k u.  Renormalised full softmax: the
    normaliser cancels in the ratio, leaving one more division per selected
    term, k u more.  Bound used (w_rtol): max(32, 2k + 2 (d + 4) + 2) u, d
    the largest distance between a token's best score and its selected
    scores -- 32 u (~1.9e-6) for the workloads (k <= 8, d <= 4).
  - combine: the kernel accumulates k fp32 fused multiply-adds and rounds once
    to bf16; the oracle sums exactly-representable products in binary64 and
    rounds once.  The fp32 error (< k * 2^-24 relative) can move the result
    across at most one bf16 rounding boundary: <= 1 bf16 ulp.
"""
from __future__ import annotations

import numpy as np
import torch

from combine_layout_gb300 import synth

W_RTOL = 32 * 2.0 ** -24


def w_rtol(k: int, scores: np.ndarray | None = None, idx: np.ndarray | None = None) -> float:
    """Relative tolerance of the gate weights (module docstring); d is taken
    from the fp32 scores and the selected expert ids when given."""
    d = 0.0
    if scores is not None and idx is not None and scores.size and idx.size:
        sel = np.take_along_axis(scores.astype(np.float64), np.maximum(idx, 0).astype(np.int64), 1)
        d = float((scores.max(1).astype(np.float64) - sel.min(1)).max())
    return max(32.0, 2 * k + 2 * (d + 4) + 2) * 2.0 ** -24


def to_dev_bf16(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def defined_rows(w_mode: int, cnt: np.ndarray, S: int, total: int) -> np.ndarray:
    """Receive rows the layout defines: HT [0, total); LL e*S + [0, cnt[e])."""
    if w_mode == synth.MODE_HT:
        return np.arange(total)
    return np.concatenate([e * S + np.arange(c) for e, c in enumerate(cnt)]) if len(cnt) else \
        np.zeros(0, np.int64)


def dequant_on_device(q: torch.Tensor, scale: torch.Tensor, chunk: int = 8192) -> torch.Tensor:
    """Identity expert for FP8 payloads (test harness, torch ops):
    y = bf16(float(q) * scale) in the receive layout.  Any deterministic bf16 y
    serves: the same y feeds the kernel and the oracle."""
    rows, H = q.shape
    y = torch.empty((rows, H), dtype=torch.bfloat16, device=q.device)
    for a in range(0, rows, chunk):
        b = min(rows, a + chunk)
        f = q[a:b].view(torch.float8_e4m3fn).float().view(b - a, H // 128, 128)
        f = torch.nan_to_num(f * scale[a:b, :, None], nan=0.0, posinf=0.0, neginf=0.0)
        y[a:b] = f.view(b - a, H).to(torch.bfloat16)
    return y


def identity_rows(x_bits: np.ndarray, tokens, fp8: bool) -> np.ndarray:
    """The oracle's expert input for each listed token under identity experts:
    the token's bf16 row, or (FP8) bf16_rn(float(q) * scale) of the oracle's
    own quantisation of it.  [len(tokens)][H] bf16 bits, oracle values only."""
    import oracle
    rows = []
    for t in np.asarray(tokens).reshape(-1):
        if fp8:
            q, s = oracle.quant_row(x_bits[t])
            rows.append(oracle.dequant_rows(q[None], s[None], [0])[0])
        else:
            rows.append(x_bits[t])
    return np.stack(rows) if rows else np.zeros((0, x_bits.shape[1]), np.uint16)

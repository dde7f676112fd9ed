"""Shared helpers for the GPU-vs-oracle parity tests (test code only).

Tolerances, derived from the arithmetic:
  - routing indices, counts, offsets, row map, receive rows, FP8 bytes and
    scales, source ids: bit-exact (integer / byte work, and the FP8 code is
    decided by one fp32 division on both sides).
  - gate weights, score-normalised: bit-exact.  Both sides take the same fp32
    definition (the sum of the selected scores in j order, one rounding per
    addition, then one division per weight), which has one answer; NaN
    weights (infinite or NaN scores) compare equal to NaN.
  - gate weights, softmax rules: the kernel computes in fp32 (expf), the
    oracle in binary64; u = 2^-24.  Softmax over the top k: each
    exp(v - max) carries the fp32 subtraction's error (at most d u in the
    exponent, d the distance of v from the maximum) and expf's (<= 2 ulp,
    4 u), in the numerator and, averaged, in the sum; then k - 1 additions
    and one division: 2 (d + 4) u + k u.  Renormalised full softmax: the
    normaliser cancels in the ratio, leaving one more division per selected
    term, k u more.  Bound used (w_rtol): max(32, 2k + 2 (d + 4) + 2) u, d
    the largest distance between a token's best score and its selected
    scores -- 32 u (~1.9e-6) for the softmax workloads (k <= 8, d <= 4).
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


def assert_weights_match(got: np.ndarray, want: np.ndarray, weight_mode: int, k: int,
                         scores: np.ndarray | None = None, idx: np.ndarray | None = None):
    """Gate weights against the oracle's: bit for bit for the score-normalised
    rule (NaN equals NaN), within w_rtol for the softmax rules."""
    got = np.asarray(got, np.float32)
    if weight_mode == synth.W_SCORE_NORM:
        want32 = np.asarray(want).astype(np.float32)
        same = (got.view(np.uint32) == want32.view(np.uint32)) | (np.isnan(got) & np.isnan(want32))
        bad = np.argwhere(~same)
        assert bad.size == 0, f"weights differ at {bad[:4].tolist()}: {got[tuple(bad[0])]!r} vs {want32[tuple(bad[0])]!r}"
    else:
        np.testing.assert_allclose(got, want, rtol=w_rtol(k, scores, idx), atol=0)


def assert_rows_equal(got: np.ndarray, want: np.ndarray, what: str):
    """Element-by-element equality of two row arrays, naming the first bad row."""
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if not np.array_equal(got, want):
        diff = (got != want).reshape(got.shape[0], -1).any(1)
        r = int(np.argmax(diff))
        raise AssertionError(f"{what}: {int(diff.sum())} rows differ, first at row {r}")


def oracle_token_payload(x_bits: np.ndarray, fp8: bool):
    """The oracle's payload of every token, one row per token (orc_dispatch
    with the row map t -> t): bf16 bits, or e4m3 codes [T][H] with their
    scales [T][H/128]."""
    import oracle
    T = x_bits.shape[0]
    row = np.arange(T, dtype=np.int32).reshape(T, 1)
    q, s, _ = oracle.dispatch(x_bits, row, T, fp8)
    return q, (s if fp8 else None)


def oracle_identity_tokens(x_bits: np.ndarray, fp8: bool) -> np.ndarray:
    """Each token's expert input under identity experts, oracle values only:
    the bf16 token, or (FP8) bf16_rn(float(q) * scale) of the oracle's own
    quantisation of it (orc_dequant_rows).  [T][H] bf16 bits."""
    import oracle
    q, s = oracle_token_payload(x_bits, fp8)
    if not fp8:
        return q
    return oracle.dequant_rows(q, s, np.arange(x_bits.shape[0]))


def take_rows(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    """rows of a device tensor: a slice when they are 0..n-1, else a gather."""
    if rows.size and rows[0] == 0 and rows[-1] == rows.size - 1:
        return t[: rows.size]
    return t.index_select(0, torch.from_numpy(np.ascontiguousarray(rows, np.int64)).to(t.device))


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

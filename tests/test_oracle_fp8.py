"""Pins for the oracle's FP8 e4m3 encoder and per-128 quantisation.

The pages fix FP8 dispatch with one fp32 scale per 128 elements
("NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式").  The element format is
OCP e4m3fn; these tests pin the oracle's encoder to hand-worked cases, to the
format's own decode table, and to torch's (non-saturating) cast where the two
agree by definition.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden


def _parse(v: str) -> float:
    return float.fromhex(v) if "p" in v else float(v)


def test_hand_worked_cases(orc):
    rows = read_golden("fp8_e4m3_cases.txt")
    assert len(rows) >= 20
    for r in rows:
        v, code = _parse(r[0]), int(r[1], 16)
        assert orc.e4m3_from_float(v) == code, (r[0], hex(orc.e4m3_from_float(v)), hex(code))


def test_decode_table_closed_form(orc):
    vals = [orc.e4m3_to_double(c) for c in range(256)]
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    finite = [v for v in vals if not math.isnan(v)]
    assert len(finite) == 254
    assert max(finite) == 448.0 and min(finite) == -448.0
    assert vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    # codes 0..0x7E strictly increasing; negatives mirror positives
    pos = vals[: 0x7F]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    for c in range(0x7F):
        assert vals[c | 0x80] == -vals[c] or (c == 0 and vals[0x80] == 0.0)
    # 8 values per binade for normals: 2^(e-7) * (1 + m/8)
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            assert vals[(e << 3) | m] == (1 + m / 8) * 2.0 ** (e - 7)


def test_roundtrip_every_finite_code(orc):
    for c in range(256):
        v = orc.e4m3_to_double(c)
        if math.isnan(v):
            continue
        assert orc.e4m3_from_float(v) == c


def test_nearest_even_brute_force(orc):
    """Every fp32 value between consecutive codes goes to the nearer code; exact
    midpoints go to the even code (checked by distance, not by formula)."""
    codes = [c for c in range(0x7F)]
    vals = np.array([orc.e4m3_to_double(c) for c in codes])
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.uniform(0, 448, 20000), rng.uniform(0, 2 ** -5, 20000),
        (vals[:-1] + vals[1:]) / 2,                      # exact midpoints
        np.nextafter((vals[:-1] + vals[1:]) / 2, 0),
        np.nextafter((vals[:-1] + vals[1:]) / 2, 1000),
    ]).astype(np.float32)
    got = orc.e4m3_from_float_array(xs)
    for x, g in zip(xs.astype(np.float64), got):
        d = np.abs(vals - x)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert g == want, (x, g, want)


def test_agrees_with_torch_cast_below_overflow(orc):
    """torch's float8_e4m3fn cast rounds to nearest even but does not saturate;
    below the overflow midpoint (464) both must agree bit for bit."""
    rng = np.random.default_rng(2)
    bf = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    xs = (bf.astype(np.uint32) << 16).view(np.float32)
    xs = xs[np.isfinite(xs) & (np.abs(xs) < 464)]
    xs = np.concatenate([xs, rng.normal(0, 100, 50000).astype(np.float32)])
    xs = xs[np.abs(xs) < 464]
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_from_float_array(xs)
    assert np.array_equal(got, want)


def test_quant_row_properties(orc):
    """scale = amax/448; the block maximum lands on +-448; dequantisation error
    within half a unit of the last place (2^-4 relative for normals, 2^-10
    * scale absolute for subnormals)."""
    from combine_layout_gb300 import synth
    rng = np.random.default_rng(3)
    x = synth.tokens_bf16(rng, 4, 7168)
    x[1, :128] = 0                      # all-zero block -> scale 1
    x[2, 128:256] = synth.f32_to_bf16_bits(np.full(128, -3.0, np.float32))
    for t in range(x.shape[0]):
        q, s = orc.quant_row(x[t])
        xf = synth.bf16_bits_to_f32(x[t]).reshape(-1, 128)
        amax = np.abs(xf).max(1)
        want_s = np.where(amax == 0, np.float32(1), (amax / np.float32(448)).astype(np.float32))
        assert np.array_equal(s, want_s.astype(np.float32))
        deq = np.array([orc.e4m3_to_double(c) for c in q]).reshape(-1, 128) * s[:, None]
        for b in range(xf.shape[0]):
            if amax[b] == 0:
                assert np.all(q.reshape(-1, 128)[b] & 0x7F == 0)
                continue
            i = int(np.argmax(np.abs(xf[b])))
            assert q.reshape(-1, 128)[b, i] in (0x7E, 0xFE)
            err = np.abs(deq[b] - xf[b])
            bound = np.maximum(np.abs(xf[b]) * 2.0 ** -4, 2.0 ** -10 * s[b]) * (1 + 1e-6)
            assert np.all(err <= bound)
    assert np.all(orc.quant_row(x[2])[0][128:256] == 0xFE)


def test_quant_row_rejects_ragged_hidden(orc):
    with pytest.raises(ValueError):
        orc.quant_row(np.zeros(100, np.uint16))

"""Pins for the oracle's combine (weighted un-permute to token order) and its
bf16 rounding.

Combine gathers the expert outputs back to token order using the routing state
of the handle and reduces them ("NCCL EP 论文解读", "核心功能函数"); the result is
the BF16 weighted sum of the expert outputs ("NVSHMEM 与 DeepEP：GPU 发起的通信",
section "高吞吐模式").  Pins: hand-worked bf16 roundings, torch's fp32 -> bf16
cast (a library routine) on values fp32 holds exactly, and closed forms of the
round trip.
"""
import numpy as np
import torch

from combine_layout_gb300 import synth
from conftest import read_golden


def test_bf16_hand_cases(orc):
    for r in read_golden("bf16_rounding_cases.txt"):
        v = float.fromhex(r[0])
        assert orc.bf16_from_double(v) == int(r[1], 16), r


def test_bf16_matches_torch_on_fp32_values(orc):
    rng = np.random.default_rng(9)
    xs = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-38, 2000),
                         rng.normal(0, 1e37, 2000)]).astype(np.float32)
    # exact midpoints between bf16 neighbours
    b = synth.f32_to_bf16_bits(rng.normal(0, 1, 2000).astype(np.float32)).astype(np.uint32)
    mids = ((b << 16) | 0x8000).view(np.float32)
    xs = np.concatenate([xs, mids])
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_from_double(float(v)) for v in xs], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_to_double_exact(orc):
    for bits in (0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049):
        f = np.array([bits << 16], np.uint32).view(np.float32)[0]
        assert orc.bf16_to_double(bits) == float(f)


def _ht(orc, T, E, R, k, seed):
    rng = np.random.default_rng(seed)
    s = synth.uniform_bias_scores(rng, T, E)
    idx, w = orc.route(s, k, weight_mode=orc.W_SCORE_NORM)
    L, _ = orc.layout(idx, E, R, orc.MODE_HT)
    x = synth.tokens_bf16(rng, T, 128)
    return x, idx, w.astype(np.float32), L["row"]


def test_single_expert_unit_weight_is_identity(orc):
    x, idx, _, row = _ht(orc, 50, 8, 4, 1, 0)
    y, _, _ = orc.dispatch(x, row, 50, fp8=False)
    out = orc.combine(y, row, np.ones((50, 1), np.float32))
    assert np.array_equal(out, x)


def test_one_hot_weights_select_one_row(orc):
    x, idx, _, row = _ht(orc, 60, 16, 4, 4, 1)
    rng = np.random.default_rng(2)
    y = synth.tokens_bf16(rng, 60 * 4, 128)          # arbitrary expert outputs
    for jsel in range(4):
        w = np.zeros((60, 4), np.float32)
        w[:, jsel] = 1
        out = orc.combine(y, row, w)
        assert np.array_equal(out, y[row[:, jsel]])


def test_identity_round_trip_weights_sum_to_one(orc):
    """Identity experts and weights summing to 1 reproduce the input to within
    one bf16 unit in the last place."""
    x, idx, w, row = _ht(orc, 80, 32, 8, 4, 3)
    y, _, _ = orc.dispatch(x, row, 80 * 4, fp8=False)
    out = orc.combine(y, row, w)
    a = synth.bf16_bits_to_f32(out).astype(np.float64)
    b = synth.bf16_bits_to_f32(x).astype(np.float64)
    ulp = np.abs(b) * 2.0 ** -7
    assert np.all(np.abs(a - b) <= ulp)


def test_linear_in_weights_and_masking(orc):
    x, idx, w, row = _ht(orc, 30, 8, 2, 2, 4)
    y, _, _ = orc.dispatch(x, row, 60, fp8=False)
    # masking a pair drops its term: same as a zero weight
    row_m = row.copy()
    row_m[:, 1] = -1
    w0 = w.copy()
    w0[:, 1] = 0
    assert np.array_equal(orc.combine(y, row_m, w), orc.combine(y, row, w0))
    # powers of two scale exactly
    assert np.array_equal(orc.combine(y, row, w * 2),
                          synth.f32_to_bf16_bits(2 * synth.bf16_bits_to_f32(orc.combine(y, row, w))))


def test_token_subset_matches_full(orc):
    x, idx, w, row = _ht(orc, 64, 16, 4, 4, 5)
    y, _, _ = orc.dispatch(x, row, 256, fp8=False)
    full = orc.combine(y, row, w)
    sub = orc.combine(y, row, w, tokens=[63, 0, 17])
    assert np.array_equal(sub, full[[63, 0, 17]])

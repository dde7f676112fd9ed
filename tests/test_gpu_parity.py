"""GPU parity: libmoeep (through the C ABI) against the CPU oracle on the same
seeded inputs, for the five workloads.

Every case compares every output element: routing, gate weights, layout,
every receive row the layout defines (bf16 payload, or FP8 bytes and scales,
and the source token), and every combined token.  Reduced token counts
(several 32-token tiles plus a ragged tail) and the full-size workloads run
the same comparison; the full sizes in the launch configuration the
benchmark times (including its moe_ep_set_x_before_route declaration, in
test_parity_with_x_before_route).  Tolerances: see tests/parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_layout_gb300 import synth
from parity import (assert_rows_equal, assert_weights_match, bf16_bits, bf16_ulp_diff,
                    defined_rows, oracle_identity_tokens, take_rows, to_dev_bf16)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _pipeline(w, x_early=False):
    from combine_layout_gb300.pipeline import EpPipeline
    return EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k, fp8=w.fp8, device=DEV,
                      x_before_route=x_early)


def _check_route_layout(w, p, inp):
    idx = p.topk_idx[: w.T].cpu().numpy()
    wg = p.topk_w[: w.T].cpu().numpy()
    idx_o, w_o = oracle.route(inp["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    assert np.array_equal(idx, idx_o), "topk_idx differs"
    assert_weights_match(wg, w_o, w.weight_mode, w.k, inp["scores"], idx_o)
    L = {k: v.cpu().numpy() for k, v in p.layout().items()}
    L_o, st = oracle.layout(idx_o, w.E, w.R, w.mode, w.slots)
    assert st == oracle.OK
    for key in ("cnt", "off", "rcnt", "roff", "row"):
        assert np.array_equal(L[key], L_o[key]), key
    return idx_o, w_o, L_o


def _run(w, seed=None, x_early=False):
    p = _pipeline(w, x_early)
    d = _check_pass(p, w, synth.make_inputs(w, seed))
    p.close()
    return d


def _check_pass(p, w, inp):
    """One forward of w.T tokens on pipeline p (whose group may hold more),
    every output element against the oracle; returns the combine's ulp
    differences."""
    scores = torch.from_numpy(inp["scores"]).to(DEV)
    x = to_dev_bf16(inp["x"], DEV)
    p.route(scores, w.T, w.G, w.kg, 0, w.weight_mode)
    total, per_rank, per_expert = p.num_recv_tokens()
    p.dispatch(x)
    torch.cuda.synchronize()
    idx_o, w_o, L_o = _check_route_layout(w, p, inp)

    if w.mode == synth.MODE_HT:
        assert total == w.T * w.k
        assert per_rank == L_o["rcnt"].tolist() and per_expert == L_o["cnt"].tolist()
    else:
        assert total == w.E * w.slots
    assert np.array_equal(p.recv_cnt.cpu().numpy(), L_o["cnt"])

    # the oracle's dispatch of every pair into the receive layout; every
    # defined row is compared
    rx_o, rs_o, src_o = oracle.dispatch(inp["x"], L_o["row"], p.rows, w.fp8)
    rows = defined_rows(w.mode, L_o["cnt"], w.slots, int(L_o["off"][-1]))
    assert np.array_equal(take_rows(p.recv_src, rows).cpu().numpy(), src_o[rows]), "recv_src"
    if w.fp8:
        assert_rows_equal(take_rows(p.recv_x, rows).cpu().numpy(), rx_o[rows], "FP8 bytes")
        assert_rows_equal(take_rows(p.recv_scale, rows).cpu().numpy().view(np.uint32),
                          rs_o[rows].view(np.uint32), "FP8 scales")
        # expert input: each row's token dequantised by the oracle (identity
        # experts); the same y feeds the kernel and the oracle
        y_o = np.zeros((p.rows, w.H), np.uint16)
        y_o[rows] = oracle_identity_tokens(inp["x"], True)[src_o[rows]]
        y = to_dev_bf16(y_o, DEV)
    else:
        assert_rows_equal(bf16_bits(take_rows(p.recv_x, rows)), rx_o[rows], "bf16 payload")
        y_o, y = rx_o, p.recv_x

    # both sides combine with the oracle's gate weights (fp32), every token
    w32 = np.ascontiguousarray(w_o, dtype=np.float32)
    out = p.combine(y, topk_w=torch.from_numpy(w32).to(DEV))
    torch.cuda.synchronize()
    want = oracle.combine(y_o, L_o["row"], w32)
    got = bf16_bits(out)
    d = bf16_ulp_diff(got, want)
    assert d.max() <= 1, f"combine differs by {d.max()} bf16 ulp"
    # round trip: identity experts, weights summing to 1, bf16 payload -> x within 1 ulp
    if not w.fp8:
        rt = bf16_ulp_diff(got, inp["x"])
        assert rt.max() <= 1, f"round trip off by {rt.max()} ulp"
    return d


@pytest.mark.parametrize("name,T", [("tiny_ll", 128), ("tiny_ll", 77), ("ll_decode", 128),
                                    ("ll_decode", 45), ("ht_prefill", 300), ("ht_prefill_fp8", 300),
                                    ("mixtral", 1000), ("skewed", 333)])
def test_parity_elementwise(name, T):
    w = synth.WORKLOADS[name].with_tokens(T, slots=synth.WORKLOADS[name].slots or None)
    _run(w)


@pytest.mark.parametrize("name", ["tiny_ll", "ll_decode", "ht_prefill", "ht_prefill_fp8",
                                  "mixtral", "skewed"])
def test_parity_full_size(name):
    _run(synth.WORKLOADS[name])


@pytest.mark.parametrize("name,T,H", [("tiny_ll", 77, None), ("ll_decode", 128, None),
                                      ("ht_prefill", 300, None), ("ht_prefill_fp8", 300, None),
                                      ("ht_prefill_fp8", 300, 640), ("mixtral", 1000, None),
                                      ("ht_prefill", 4096, None), ("ht_prefill_fp8", 4096, None),
                                      ("mixtral", 8192, None)])
def test_parity_with_x_before_route(name, T, H):
    """moe_ep_set_x_before_route: each bf16 dispatch CTA reads its token
    before waiting for the router; the results are the same (the FP8 cases,
    general kernel at H = 640 and exact-fit at 7168, read after the wait)."""
    base = synth.WORKLOADS[name]
    w = base.with_tokens(T, slots=base.slots or None)
    if H is not None:
        d = dict(w.__dict__)
        d.pop("extra")
        d["H"] = H
        w = synth.Workload(**d)
    _run(w, x_early=True)


def test_fp8_conversion_sweep_all_bf16_values():
    """Blocks whose maximum is 448 have scale exactly 1, so the payload is the
    plain e4m3 conversion of every finite bf16 value of magnitude <= 448."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(bits)
    vals = bits[np.isfinite(f) & (np.abs(f) <= 448)]
    per_block = 127
    nblk = -(-vals.size // per_block)
    H = 7168
    T = -(-nblk // (H // 128)) + 1          # last token: the tiny-magnitude block
    blocks = np.zeros((T * (H // 128), 128), np.uint16)
    blocks[:, 0] = synth.f32_to_bf16_bits(np.array([448.0], np.float32))[0]
    flat = np.zeros(T * (H // 128) * per_block, np.uint16)
    flat[: vals.size] = vals
    blocks[:, 1:] = flat.reshape(-1, per_block)
    x = blocks.reshape(T, H)
    # tiny-magnitude blocks: subnormal bf16 inputs, scales in fp32's subnormal range
    x[-1, :128] = np.arange(128, dtype=np.uint16)
    from combine_layout_gb300.pipeline import EpPipeline
    p = EpPipeline(synth.MODE_HT, 8, 2, T, H, 1, fp8=True, device=DEV)
    idx = torch.zeros((T, 1), dtype=torch.int32, device=DEV)
    p.route_given(idx)
    p.dispatch(to_dev_bf16(x, DEV))
    torch.cuda.synchronize()
    q = p.recv_x[:T].cpu().numpy()
    s = p.recv_scale[:T].cpu().numpy()
    for t in range(T):
        qo, so = oracle.quant_row(x[t])
        assert np.array_equal(s[t], so)
        assert np.array_equal(q[t], qo), t
    assert np.all(s[:-1] == 1.0)
    p.close()


def _e4m3_values_and_midpoints():
    vals = sorted({abs(oracle.e4m3_to_double(c)) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    return np.array(vals + mids)


def test_fp8_quotients_on_ties_with_odd_scales():
    """Blocks with amax = 448 * S * 2^j (S = 1..36) have the exact scale S * 2^j,
    and elements x = m * S * 2^j put x / scale exactly on e4m3 values and
    rounding midpoints (ties to even) for non-power-of-two scales; neighbours
    one bf16 step away sit just off the ties.  Every byte must equal the
    oracle's (IEEE fp32 division)."""
    rng = np.random.default_rng(21)
    targets = _e4m3_values_and_midpoints()
    H = 7168
    nblk = H // 128
    T = 64
    x = np.zeros((T, H), np.float32)
    for t in range(T):
        for b in range(nblk):
            S = int(rng.integers(1, 37))
            j = int(rng.integers(-60, 60))
            scale = np.float32(S * 2.0 ** j)
            blk = np.empty(128, np.float32)
            blk[0] = np.float32(448.0 * S * 2.0 ** j)
            m = rng.choice(targets, 127) * rng.choice([-1.0, 1.0], 127)
            blk[1:] = (m * float(scale)).astype(np.float32)
            x[t, b * 128:(b + 1) * 128] = blk
    xb = synth.f32_to_bf16_bits(x)
    # half the tokens: nudge every element one bf16 step up or down (off the ties)
    nudge = rng.integers(-1, 2, xb.shape).astype(np.int32)
    nudge[: T // 2] = 0
    nudge[:, ::128] = 0                       # keep each block's amax element
    xb = np.where(xb & 0x7FFF, (xb.astype(np.int32) + nudge).astype(np.uint16), xb)
    _fp8_bytes_match_oracle(xb)


def test_fp8_quotients_random_scales_both_paths():
    """Random blocks whose amax spans 2^-130 .. 2^120 (both the reciprocal path
    and the direct-division path), random signs and magnitudes inside blocks."""
    rng = np.random.default_rng(22)
    T, H = 256, 7168
    e = rng.integers(-130, 121, (T, H // 128)).astype(np.float64)
    mag = 2.0 ** (e[:, :, None] - rng.integers(0, 40, (T, H // 128, 128)))
    x = (rng.uniform(0.5, 1.0, (T, H // 128, 128)) * mag * rng.choice([-1, 1], (T, H // 128, 128)))
    x = np.clip(x, -3e38, 3e38).astype(np.float32).reshape(T, H)
    x[::7, ::5] = -0.0
    _fp8_bytes_match_oracle(synth.f32_to_bf16_bits(x))


def _fp8_bytes_match_oracle(xb):
    from combine_layout_gb300.pipeline import EpPipeline
    T, H = xb.shape
    p = EpPipeline(synth.MODE_HT, 8, 2, T, H, 1, fp8=True, device=DEV)
    p.route_given(torch.zeros((T, 1), dtype=torch.int32, device=DEV))
    p.dispatch(to_dev_bf16(xb, DEV))
    torch.cuda.synchronize()
    q = p.recv_x[:T].cpu().numpy()
    s = p.recv_scale[:T].cpu().numpy()
    for t in range(T):
        qo, so = oracle.quant_row(xb[t])
        assert np.array_equal(s[t], so), t
        bad = np.nonzero(q[t] != qo)[0]
        assert bad.size == 0, (t, bad[:4], q[t][bad[:4]], qo[bad[:4]])
    p.close()


def test_fp8_scale_for_every_bf16_block_maximum():
    """The block maximum is always a bf16 value: every positive finite one
    (0x0001 .. 0x7f7f) is some block's maximum here, so the scale amax / 448
    (Markstein's method inside 2^-80 .. 2^100, IEEE division outside) is
    compared with the oracle's fp32 division for every value it can take, and
    the bytes of the block's other elements with it."""
    rng = np.random.default_rng(23)
    amax_bits = np.arange(1, 0x7F80, dtype=np.uint16)
    H = 7168
    nblk = H // 128
    T = -(-amax_bits.size // nblk)
    amax = np.ones(T * nblk, np.uint16) * 0x3F80          # padding blocks: amax 1.0
    amax[: amax_bits.size] = amax_bits
    af = synth.bf16_bits_to_f32(amax).astype(np.float64)
    blocks = rng.uniform(-1.0, 1.0, (T * nblk, 128)) * af[:, None]
    xb = synth.f32_to_bf16_bits(blocks.astype(np.float32))
    big = np.abs(synth.bf16_bits_to_f32(xb)) > synth.bf16_bits_to_f32(amax)[:, None]
    xb = np.where(big, amax[:, None], xb)                 # rounding must not exceed amax
    pos = rng.integers(0, 128, T * nblk)
    xb[np.arange(T * nblk), pos] = amax                   # the maximum itself
    _fp8_bytes_match_oracle(xb.reshape(T, H).astype(np.uint16))


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("name,per_sm,extra,H", [
    ("ht_prefill", 4, -1, None), ("ht_prefill", 4, 0, None), ("ht_prefill", 16, -1, None),
    ("ht_prefill", 16, 0, None), ("ht_prefill", 16, 37, None), ("mixtral", 16, 5, None),
    ("ht_prefill", 16, 3, 7296)])
def test_parity_around_the_sliced_tail(name, per_sm, extra, H):
    """Large batches put their last tokens in column slices (the bf16
    dispatch from 16 tokens per SM, the combine from 4): token counts on both
    sides of each threshold, a row width whose 16-vector units split only
    into odd slices (H = 7296: 57 units), and the 4096-wide rows that take
    the 64-thread dispatch CTAs -- every element against the oracle."""
    base = synth.WORKLOADS[name]
    w = base.with_tokens(per_sm * _sms() + extra)
    if H is not None:
        d = dict(w.__dict__)
        d.pop("extra")
        d["H"] = H
        w = synth.Workload(**d)
    _run(w, x_early=True)


@pytest.mark.parametrize("name,max_tokens,sizes", [
    ("ht_prefill", 4096, (4096, 1, 3000, 257, 2500, 33, 4096)),
    ("ht_prefill_fp8", 3000, (3000, 77, 2600, 5)),
    ("ll_decode", 300, (300, 100, 1, 300, 256, 257))])
def test_one_handle_through_batches_of_changing_size(name, max_tokens, sizes):
    """One group and handle, forwards of changing size in a row (small and
    large batches, LL layouts deferred to the dispatch and finished by the
    router's last CTA, sliced and unsliced tails): the workspace left by one
    forward must not leak into the next.  Every forward against the oracle."""
    base = synth.WORKLOADS[name]
    p = _pipeline(base.with_tokens(max_tokens, slots=max_tokens if base.slots else None))
    for i, T in enumerate(sizes):
        w = base.with_tokens(T, slots=max_tokens if base.slots else None)
        _check_pass(p, w, synth.make_inputs(w, 1000 + i))
    p.close()

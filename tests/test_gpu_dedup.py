"""GPU parity of the per-rank dedup path (moe_ep_dispatch_dedup,
moe_ep_expand, moe_ep_combine_dedup) against the CPU oracle.

Tolerances (from the arithmetic):
  - rank counts, offsets, dedup row tokens and masks, the payload bytes and
    FP8 scales of every dedup row, and the expanded HT rows: bit-exact.
  - partial rows: the kernel's fp32 fma chain over a rank's pairs is rounded
    once to bf16, the oracle's exact sum too; the fp32 error can cross at most
    one bf16 rounding boundary: <= 1 ulp.
  - out: each kernel partial is within 1 ulp of the oracle's, and the source
    adds them in fp32 and rounds once: |out - out_oracle| <= sum of the
    token's partials' ulps + ulp(out); where every partial of a token agrees,
    <= 1 ulp.
Both sides combine with the oracle's gate weights and expert inputs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_layout_gb300 import synth
from parity import (assert_rows_equal, bf16_bits, bf16_ulp_diff, oracle_token_payload,
                    to_dev_bf16)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _ulp(bits):
    f = np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(f, 2.0 ** -126))) - 7)


def _run(w, x_early=False):
    """The whole dedup path against the oracle, every element compared."""
    from combine_layout_gb300.pipeline import EpPipeline
    p = EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k, fp8=w.fp8, device=DEV,
                   x_before_route=x_early)
    r = _check_pass(p, w, synth.make_inputs(w))
    p.close()
    return r


def _check_pass(p, w, inp):
    """One dedup forward of w.T tokens on pipeline p (whose group may hold
    more tokens), every element against the oracle."""
    x_d = to_dev_bf16(inp["x"], DEV)
    p.route(torch.from_numpy(inp["scores"]).to(DEV), w.T, w.G, w.kg, 0, w.weight_mode)
    p.dispatch_dedup(x_d)
    p.recv_x.zero_()
    p.expand()
    torch.cuda.synchronize()

    idx_o, w_o = oracle.route(inp["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    assert np.array_equal(p.topk_idx[: w.T].cpu().numpy(), idx_o)
    RL, st = oracle.rank_layout(idx_o, w.E, w.R)
    assert st == oracle.OK
    nd = int(RL["off"][-1])
    assert np.array_equal(p.rank_cnt.cpu().numpy(), RL["cnt"])
    assert np.array_equal(p.rank_off.cpu().numpy(), RL["off"])
    assert np.array_equal(p.drecv_src[:nd].cpu().numpy(), RL["src"])
    assert np.array_equal(p.drecv_mask[:nd].cpu().numpy().view(np.uint32), RL["mask"])

    # payload of every dedup row: its token's oracle payload
    q_tok, s_tok = oracle_token_payload(inp["x"], w.fp8)
    if w.fp8:
        assert_rows_equal(p.drecv_x[:nd].cpu().numpy(), q_tok[RL["src"]], "dedup FP8 bytes")
        assert_rows_equal(p.drecv_scale[:nd].cpu().numpy().view(np.uint32),
                          s_tok[RL["src"]].view(np.uint32), "dedup FP8 scales")
    else:
        assert_rows_equal(bf16_bits(p.drecv_x[:nd]), q_tok[RL["src"]], "dedup bf16 payload")

    # expansion = the oracle's direct dispatch, every row
    D, _ = oracle.layout(idx_o, w.E, w.R, oracle.MODE_HT)
    nrows = int(D["off"][-1])
    rx_o, rs_o, src_o = oracle.dispatch(inp["x"], D["row"], nrows, w.fp8)
    assert np.array_equal(p.recv_src[:nrows].cpu().numpy(), src_o)
    if w.fp8:
        assert_rows_equal(p.recv_x[:nrows].cpu().numpy(), rx_o, "expanded FP8 bytes")
        assert_rows_equal(p.recv_scale[:nrows].cpu().numpy().view(np.uint32),
                          rs_o.view(np.uint32), "expanded FP8 scales")
    else:
        assert_rows_equal(bf16_bits(p.recv_x[:nrows]), rx_o, "expanded bf16 payload")

    # two-stage combine on the oracle's expert inputs and weights, every token
    w32 = np.ascontiguousarray(w_o, dtype=np.float32)
    y_tok = oracle.dequant_rows(q_tok, s_tok, np.arange(w.T)) if w.fp8 else q_tok
    y_rows = y_tok[src_o]                                     # [nrows][H], oracle values
    y_d = torch.zeros((p.rows, w.H), dtype=torch.bfloat16, device=DEV)
    y_d[:nrows] = to_dev_bf16(y_rows, DEV)
    out = p.combine_dedup(y_d, topk_w=torch.from_numpy(w32).to(DEV))
    torch.cuda.synchronize()
    want, part = oracle.combine_dedup(y_rows, idx_o, D["row"], w32, w.E, w.R, RL["drow"], nd,
                                      want_partial=True)
    got = bf16_bits(out)
    got_part = bf16_bits(p.partial[:nd])
    dp = bf16_ulp_diff(got_part, part)
    assert dp.max() <= 1, f"partial rows differ by {dp.max()} ulp"
    # the out bound, every token: the sum of its partials' ulps plus the
    # result's; where all its partials agree, 1 ulp
    qs = RL["drow"]
    pu = _ulp(part)
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    o = synth.bf16_bits_to_f32(want).astype(np.float64)
    bound = np.maximum(_ulp(got), _ulp(want))
    agree = np.ones(w.T, bool)
    for j in range(w.k):
        has = qs[:, j] >= 0
        bound[has] += pu[qs[has, j]]
        agree[has] &= dp[qs[has, j]].max(1) == 0
    assert np.all(np.abs(g - o) <= bound * (1 + 1e-6)), "out outside the two-rounding bound"
    assert bf16_ulp_diff(got[agree], want[agree]).max(initial=0) <= 1
    return nd, nrows


@pytest.mark.parametrize("name,T", [("ht_prefill", 300), ("ht_prefill_fp8", 300),
                                    ("mixtral", 1000), ("skewed", 333), ("ht_prefill", 45)])
def test_dedup_elementwise(name, T):
    w = synth.WORKLOADS[name].with_tokens(T)
    nd, nrows = _run(w)
    if w.E // w.R > 1:
        assert nd < nrows
    else:
        assert nd == nrows                    # one expert per rank: nothing to dedup


@pytest.mark.parametrize("name", ["ht_prefill", "ht_prefill_fp8", "skewed", "mixtral"])
def test_dedup_full_size(name):
    w = synth.WORKLOADS[name]
    nd, nrows = _run(w)
    assert nd < nrows if w.E // w.R > 1 else nd == nrows


@pytest.mark.parametrize("name", ["ht_prefill", "ht_prefill_fp8"])
def test_dedup_with_x_before_route(name):
    _run(synth.WORKLOADS[name].with_tokens(300), x_early=True)


def test_dedup_small_ranks_wide_masks():
    """E/R = 32 local experts (a full 32-bit mask), k = 8."""
    w = synth.Workload("wide", T=200, H=256, E=64, R=2, k=8, mode=synth.MODE_HT, fp8=False,
                       scores="uniform_bias", weight_mode=synth.W_SCORE_NORM, seed=5)
    _run(w)


def test_dedup_argument_errors():
    import combine_layout_gb300.moe_ep as ep
    from combine_layout_gb300.pipeline import EpPipeline
    w = synth.WORKLOADS["ht_prefill"].with_tokens(64)
    inp = synth.make_inputs(w)
    p = EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k, device=DEV)
    p._dedup_buffers()
    y = p.recv_x
    with pytest.raises(ep.MoeEpError):           # no route yet
        p.dispatch_dedup(to_dev_bf16(inp["x"], DEV))
    p.route(torch.from_numpy(inp["scores"]).to(DEV), w.T, w.G, w.kg, 0, w.weight_mode)
    with pytest.raises(ep.MoeEpError):           # no dedup dispatch for this route
        p.expand()
    with pytest.raises(ep.MoeEpError):
        p.combine_dedup(y)
    p.dispatch_dedup(to_dev_bf16(inp["x"], DEV))
    with pytest.raises(ep.MoeEpError):           # capacity below T * min(k, R)
        ep.moe_ep_dispatch_dedup(p.handle, to_dev_bf16(inp["x"], DEV), False, p.drecv_x,
                                 drecv_rows=w.T * w.k - 1)
    with pytest.raises(ep.MoeEpError):           # partial overlapping out
        ep.moe_ep_combine_dedup(p.handle, y, p.topk_w, p.drecv_src, p.partial, p.partial)
    p.route(torch.from_numpy(inp["scores"]).to(DEV), w.T, w.G, w.kg, 0, w.weight_mode)
    with pytest.raises(ep.MoeEpError):           # the new route cleared the dedup layout
        p.expand()
    p.close()
    q = EpPipeline(synth.MODE_LL, 16, 4, 32, 256, 2, device=DEV)
    q.route(torch.zeros((32, 16), device=DEV), 32)
    with pytest.raises(ep.MoeEpError):           # HT only
        q.dispatch_dedup(torch.zeros((32, 256), dtype=torch.bfloat16, device=DEV))
    q.close()


def test_dedup_with_caller_routing_masked_and_invalid_ids():
    """Caller-made routing with padding (-1), out-of-range and repeated ids:
    the dedup rows skip them exactly as the oracle does, the expansion still
    equals the direct dispatch, and the device error word latches the ids."""
    import combine_layout_gb300.moe_ep as ep
    from combine_layout_gb300.pipeline import EpPipeline
    rng = np.random.default_rng(31)
    T, E, R, H, k = 90, 32, 8, 256, 6
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    idx[::5, 2] = -1
    idx[7, :] = -1
    idx[11, 0] = E          # out of range
    idx[13, 3] = idx[13, 1]  # repeated expert
    x = synth.tokens_bf16(rng, T, H)
    p = EpPipeline(synth.MODE_HT, E, R, T, H, k, device=DEV)
    p.route_given(torch.from_numpy(idx).to(DEV))
    torch.cuda.synchronize()
    assert p.device_errors() & ep.MOE_EP_DEVERR_EXPERT_RANGE
    p.clear_device_errors()
    p.dispatch_dedup(to_dev_bf16(x, DEV))
    p.recv_x.zero_()
    p.expand()
    torch.cuda.synchronize()
    RL, st = oracle.rank_layout(idx, E, R)
    assert st == oracle.ERR_INVALID
    nd = int(RL["off"][-1])
    assert np.array_equal(p.rank_off.cpu().numpy(), RL["off"])
    assert np.array_equal(p.drecv_src[:nd].cpu().numpy(), RL["src"])
    assert np.array_equal(p.drecv_mask[:nd].cpu().numpy().view(np.uint32), RL["mask"])
    assert np.array_equal(bf16_bits(p.drecv_x[:nd]), x[RL["src"]])
    D, _ = oracle.layout(idx, E, R, oracle.MODE_HT)
    nrows = int(D["off"][-1])
    want, _, want_src = oracle.dispatch(x, D["row"], nrows, fp8=False)
    assert np.array_equal(bf16_bits(p.recv_x[:nrows]), want)
    assert np.array_equal(p.recv_src[:nrows].cpu().numpy(), want_src)
    w32 = rng.random((T, k)).astype(np.float32)
    out = p.combine_dedup(p.recv_x, topk_w=torch.from_numpy(w32).to(DEV))
    torch.cuda.synchronize()
    want_out, part = oracle.combine_dedup(want, idx, D["row"], w32, E, R, RL["drow"], nd,
                                          want_partial=True)
    assert bf16_ulp_diff(bf16_bits(p.partial[:nd]), part).max() <= 1
    assert np.all(bf16_bits(out)[7] == 0)                 # no pair: zero row
    got = synth.bf16_bits_to_f32(bf16_bits(out)).astype(np.float64)
    o = synth.bf16_bits_to_f32(want_out).astype(np.float64)
    pu = _ulp(part)
    for t in range(T):
        qs = RL["drow"][t][RL["drow"][t] >= 0]
        bound = pu[qs].sum(0) + np.maximum(_ulp(bf16_bits(out)[t]), _ulp(want_out[t]))
        assert np.all(np.abs(got[t] - o[t]) <= bound * (1 + 1e-6)), t
    assert p.device_errors() == 0
    p.close()


def test_dedup_empty_batch():
    from combine_layout_gb300.pipeline import EpPipeline
    p = EpPipeline(synth.MODE_HT, 16, 4, 64, 256, 4, device=DEV)
    p.route(torch.zeros((0, 16), device=DEV), 0)
    p.dispatch_dedup(torch.zeros((1, 256), dtype=torch.bfloat16, device=DEV))
    p.expand()
    p.combine_dedup(p.recv_x)
    torch.cuda.synchronize()
    assert p.rank_cnt.cpu().tolist() == [0] * 4 and p.rank_off.cpu().tolist() == [0] * 5
    p.close()


@pytest.mark.parametrize("name", ["ht_prefill", "ht_prefill_fp8"])
def test_dedup_through_batches_of_changing_size(name):
    """One group and handle, dedup forwards of changing size in a row: the
    rank layout and the dedup row map of one forward must not leak into the
    next.  Every forward against the oracle."""
    from combine_layout_gb300.pipeline import EpPipeline
    base = synth.WORKLOADS[name]
    big = base.with_tokens(3000)
    p = EpPipeline(big.mode, big.E, big.R, big.max_tokens, big.H, big.k, fp8=big.fp8,
                   device=DEV)
    for i, T in enumerate((3000, 40, 2500, 1, 700)):
        w = base.with_tokens(T)
        _check_pass(p, w, synth.make_inputs(w, 2000 + i))
    p.close()

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
from parity import bf16_bits, bf16_ulp_diff, identity_rows, to_dev_bf16

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _ulp(bits):
    f = np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(f, 2.0 ** -126))) - 7)


def _run(w, sample=None, x_early=False):
    from combine_layout_gb300.pipeline import EpPipeline
    inp = synth.make_inputs(w)
    p = EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k, fp8=w.fp8, device=DEV,
                   x_before_route=x_early)
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

    # payload of the dedup rows (sampled at full size)
    rows = np.arange(nd)
    if sample is not None and nd > sample:
        rng = np.random.default_rng(11)
        rows = np.unique(np.concatenate([rows[:64], rows[-64:], rng.choice(nd, sample)]))
    rt = torch.from_numpy(rows).to(DEV)
    src = RL["src"][rows]
    if w.fp8:
        q = p.drecv_x.index_select(0, rt).cpu().numpy()
        sc = p.drecv_scale.index_select(0, rt).cpu().numpy()
        for i, t in enumerate(src):
            qo, so = oracle.quant_row(inp["x"][t])
            assert np.array_equal(q[i], qo) and np.array_equal(sc[i], so), rows[i]
    else:
        assert np.array_equal(bf16_bits(p.drecv_x.index_select(0, rt)), inp["x"][src])

    # expansion = the direct dispatch's rows (oracle layout)
    D, _ = oracle.layout(idx_o, w.E, w.R, oracle.MODE_HT)
    nrows = int(D["off"][-1])
    erows = np.arange(nrows)
    if sample is not None and nrows > sample:
        rng = np.random.default_rng(12)
        erows = np.unique(np.concatenate([erows[:64], erows[-64:], rng.choice(nrows, sample)]))
    want_src = np.empty(nrows, np.int64)
    flat = D["row"].ravel()
    want_src[flat[flat >= 0]] = np.nonzero(flat >= 0)[0] // w.k
    et = torch.from_numpy(erows).to(DEV)
    assert np.array_equal(p.recv_src.index_select(0, et).cpu().numpy(), want_src[erows])
    if w.fp8:
        q = p.recv_x.index_select(0, et).cpu().numpy()
        sc = p.recv_scale.index_select(0, et).cpu().numpy()
        for i, t in enumerate(want_src[erows]):
            qo, so = oracle.quant_row(inp["x"][t])
            assert np.array_equal(q[i], qo) and np.array_equal(sc[i], so), erows[i]
    else:
        assert np.array_equal(bf16_bits(p.recv_x.index_select(0, et)), inp["x"][want_src[erows]])

    # two-stage combine on the oracle's expert inputs and weights
    w32 = np.ascontiguousarray(w_o, dtype=np.float32)
    y_rows = identity_rows(inp["x"], np.arange(w.T), w.fp8)[want_src]   # [nrows][H], oracle values
    y_d = torch.zeros((p.rows, w.H), dtype=torch.bfloat16, device=DEV)
    y_d[:nrows] = to_dev_bf16(y_rows, DEV)
    out = p.combine_dedup(y_d, topk_w=torch.from_numpy(w32).to(DEV))
    torch.cuda.synchronize()
    tokens = np.arange(w.T)
    if sample is not None and w.T > sample:
        rng = np.random.default_rng(13)
        tokens = np.unique(np.concatenate([tokens[:32], tokens[-32:], rng.choice(w.T, sample)]))
    want, part = oracle.combine_dedup(y_rows, idx_o, D["row"], w32, w.E, w.R, RL["drow"], nd,
                                      tokens=tokens, want_partial=True)
    got = bf16_bits(out[torch.from_numpy(tokens).to(DEV)])
    qs = RL["drow"][tokens]
    qrows = np.unique(qs[qs >= 0])
    got_part = bf16_bits(p.partial.index_select(0, torch.from_numpy(qrows).to(DEV)))
    dp = bf16_ulp_diff(got_part, part[qrows])
    assert dp.max() <= 1, f"partial rows differ by {dp.max()} ulp"
    # the out bound, token by token
    pos = {q: i for i, q in enumerate(qrows)}
    pu = _ulp(part[qrows])
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    o = synth.bf16_bits_to_f32(want).astype(np.float64)
    for i, t in enumerate(tokens):
        mine = [pos[q] for q in qs[i] if q >= 0]
        bound = pu[mine].sum(0) + np.maximum(_ulp(got[i]), _ulp(want[i]))
        assert np.all(np.abs(g[i] - o[i]) <= bound * (1 + 1e-6)), t
        if np.all(dp[mine] == 0):
            assert bf16_ulp_diff(got[i], want[i]).max() <= 1, t
    p.close()
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


@pytest.mark.parametrize("name", ["ht_prefill", "ht_prefill_fp8"])
def test_dedup_full_size(name):
    nd, nrows = _run(synth.WORKLOADS[name], sample=1024)
    assert nd < nrows


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

"""GPU edge cases and error behaviour of the C ABI: empty and single-token
batches, the maximum token count, masked and invalid expert ids (device-error
word, no out-of-bounds writes), host-side argument checks, hot experts."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_layout_gb300 import synth
from parity import assert_weights_match, bf16_bits, bf16_ulp_diff, to_dev_bf16

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _ep():
    import combine_layout_gb300.moe_ep as ep
    return ep


def _pipe(mode, E, R, S, H, k, fp8=False):
    from combine_layout_gb300.pipeline import EpPipeline
    return EpPipeline(mode, E, R, S, H, k, fp8=fp8, device=DEV)


def test_empty_batch():
    p = _pipe(synth.MODE_HT, 16, 4, 64, 256, 2)
    scores = torch.zeros((0, 16), device=DEV)
    p.route(scores, 0)
    total, pr, pe = p.num_recv_tokens()
    assert total == 0 and sum(pr) == 0 and sum(pe) == 0
    p.dispatch(torch.zeros((1, 256), dtype=torch.bfloat16, device=DEV))
    p.combine(p.recv_x)
    torch.cuda.synchronize()
    assert p.layout()["off"].cpu().tolist() == [0] * 17
    p.close()


@pytest.mark.parametrize("mode", [synth.MODE_LL, synth.MODE_HT])
def test_single_token_and_max_tokens(mode):
    E, R, S, H, k = 64, 8, 96, 512, 6
    rng = np.random.default_rng(0)
    for T in (1, S):
        s = rng.random((T, E)).astype(np.float32)
        x = synth.tokens_bf16(rng, T, H)
        p = _pipe(mode, E, R, S, H, k)
        p.route(torch.from_numpy(s).to(DEV), T, 8, 3)
        p.dispatch(to_dev_bf16(x, DEV))
        out = p.combine(p.recv_x)
        torch.cuda.synchronize()
        idx_o, _ = oracle.route(s, k, 8, 3)
        assert np.array_equal(p.topk_idx[:T].cpu().numpy(), idx_o)
        L_o, _ = oracle.layout(idx_o, E, R, mode, S)
        assert np.array_equal(p.layout()["row"].cpu().numpy(), L_o["row"])
        assert bf16_ulp_diff(bf16_bits(out), x).max() <= 1
        p.close()


def test_too_many_tokens_is_overflow():
    ep = _ep()
    p = _pipe(synth.MODE_LL, 16, 4, 32, 256, 2)
    with pytest.raises(ep.MoeEpError) as e:
        p.route(torch.zeros((33, 16), device=DEV), 33)
    assert e.value.status == ep.MOE_EP_ERR_OVERFLOW
    p.close()


def test_masked_pairs_get_no_row_and_no_term():
    T, E, R, H, k = 70, 8, 4, 256, 3
    rng = np.random.default_rng(1)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    idx[::5, 1] = -1
    idx[7, :] = -1
    x = synth.tokens_bf16(rng, T, H)
    p = _pipe(synth.MODE_HT, E, R, T, H, k)
    p.route_given(torch.from_numpy(idx).to(DEV))
    total, _, _ = p.num_recv_tokens()
    L_o, st = oracle.layout(idx, E, R, oracle.MODE_HT)
    assert st == oracle.OK and total == int((idx >= 0).sum())
    assert np.array_equal(p.layout()["row"].cpu().numpy(), L_o["row"])
    p.dispatch(to_dev_bf16(x, DEV))
    w_h = rng.random((T, k)).astype(np.float32)
    out = p.combine(p.recv_x, torch.from_numpy(w_h).to(DEV))
    torch.cuda.synchronize()
    y_o, _, _ = oracle.dispatch(x, L_o["row"], total, fp8=False)
    want = oracle.combine(y_o, L_o["row"], w_h)
    assert bf16_ulp_diff(bf16_bits(out), want).max() <= 1
    assert np.all(bf16_bits(out)[7] == 0)
    assert p.device_errors() == 0
    p.close()


def test_receive_buffer_sized_by_query():
    """HT buffers sized exactly by the receive-count query are accepted."""
    ep = _ep()
    T, E, R, H, k = 64, 8, 4, 128, 2
    idx = np.tile(np.array([[0, -1]], np.int32), (T, 1))
    p = _pipe(synth.MODE_HT, E, R, T, H, k)
    p.route_given(torch.from_numpy(idx).to(DEV))
    x = torch.ones((T, H), dtype=torch.bfloat16, device=DEV)
    small = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ep.MoeEpError):          # T*k rows required before the query
        ep.moe_ep_dispatch(p.handle, x, False, small)
    total, _, _ = p.num_recv_tokens()
    assert total == T
    ep.moe_ep_dispatch(p.handle, x, False, small)
    torch.cuda.synchronize()
    assert torch.equal(small, x)
    p.close()


def test_invalid_expert_ids_latch_device_error_without_stray_writes():
    ep = _ep()
    T, E, R, H, k = 40, 8, 4, 128, 2
    idx = np.array([[t % E, (t + 1) % E] for t in range(T)], np.int32)
    idx[3, 0] = 8          # out of range
    idx[9, 1] = -7         # out of range
    idx[12, 1] = idx[12, 0]  # repeated expert
    p = _pipe(synth.MODE_HT, E, R, T, H, k)
    guard = torch.full((p.rows + 64, H), 7, dtype=torch.bfloat16, device=DEV)
    p.recv_x = guard[: p.rows]
    p.route_given(torch.from_numpy(idx).to(DEV))
    torch.cuda.synchronize()
    bits = p.device_errors()
    assert bits & ep.MOE_EP_DEVERR_EXPERT_RANGE and bits & ep.MOE_EP_DEVERR_DUPLICATE
    with pytest.raises(ep.MoeEpError) as e:
        p.num_recv_tokens()
    assert e.value.status == ep.MOE_EP_ERR_DEVICE
    p.clear_device_errors()
    L_o, st = oracle.layout(idx, E, R, oracle.MODE_HT)
    assert st == oracle.ERR_INVALID
    assert np.array_equal(p.layout()["row"].cpu().numpy(), L_o["row"])
    total, _, _ = p.num_recv_tokens()
    assert total == T * k - 3
    p.dispatch(torch.ones((T, H), dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(guard[p.rows:] == 7)
    assert torch.all(guard[total:p.rows] == 7)
    p.close()


def test_host_argument_errors():
    ep = _ep()
    p = _pipe(synth.MODE_HT, 16, 4, 64, 256, 2, fp8=False)
    s = torch.rand((10, 16), device=DEV)
    bad = [dict(num_groups=3), dict(num_groups=4, topk_groups=5), dict(num_groups=64),
           dict(weight_mode=9), dict(num_groups=8, topk_groups=1, group_topk=5)]
    for kw in bad:
        with pytest.raises(ep.MoeEpError) as e:
            p.route(s, 10, **kw)
        assert e.value.status == ep.MOE_EP_ERR_INVALID, kw
    p.route(s, 10)
    x = torch.zeros((10, 256), dtype=torch.bfloat16, device=DEV)
    buf = torch.zeros(10 * 256 + 8, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ep.MoeEpError):       # misaligned x
        ep.moe_ep_dispatch(p.handle, buf[1:].data_ptr(), False, p.recv_x, None, None, None, p.rows)
    with pytest.raises(ep.MoeEpError):       # FP8 needs H % 128 == 0 and scales
        ep.moe_ep_dispatch(p.handle, x, True, p.recv_x, None, None, None, p.rows)
    with pytest.raises(ep.MoeEpError):       # too few receive rows
        ep.moe_ep_dispatch(p.handle, x, False, p.recv_x, None, None, None, 19)
    with pytest.raises(ep.MoeEpError):       # out overlapping y
        ep.moe_ep_combine(p.handle, p.recv_x, p.topk_w, p.recv_x, p.rows)
    h2 = ep.moe_ep_create_handle(p.group, 2)
    with pytest.raises(ep.MoeEpError):       # dispatch before any route
        ep.moe_ep_dispatch(h2, x, False, p.recv_x, None, None, None, p.rows)
    with pytest.raises(ep.MoeEpError):       # group with live handles
        ep.moe_ep_destroy_group(p.group)
    ep.moe_ep_destroy_handle(h2)
    p.close()


def test_hot_expert_every_token():
    """All tokens pick the same experts: one expert receives T rows."""
    T, E, R, H, k = 1000, 32, 8, 256, 4
    s = np.zeros((T, E), np.float32)
    s[:, [3, 17, 30, 5]] = [4, 3, 2, 1]
    rng = np.random.default_rng(2)
    x = synth.tokens_bf16(rng, T, H)
    for mode, S in ((synth.MODE_HT, T), (synth.MODE_LL, T)):
        p = _pipe(mode, E, R, S, H, k)
        p.route(torch.from_numpy(s).to(DEV), T, weight_mode=synth.W_SOFTMAX_TOPK)
        p.dispatch(to_dev_bf16(x, DEV))
        out = p.combine(p.recv_x)
        torch.cuda.synchronize()
        L = p.layout()
        assert L["cnt"].cpu().numpy()[[3, 5, 17, 30]].tolist() == [T] * 4
        assert bf16_ulp_diff(bf16_bits(out), x).max() <= 1
        assert np.array_equal(p.topk_idx[:T].cpu().numpy()[0], [3, 17, 30, 5])
        p.close()


def test_two_calls_in_a_row_reuse_the_handle():
    w = synth.WORKLOADS["ht_prefill"].with_tokens(200)
    p = _pipe(w.mode, w.E, w.R, w.T, w.H, w.k)
    rng = np.random.default_rng(5)
    for T in (200, 57):
        s = synth.uniform_bias_scores(rng, T, w.E)
        x = synth.tokens_bf16(rng, T, w.H)
        p.route(torch.from_numpy(s).to(DEV), T, w.G, w.kg)
        p.num_recv_tokens()
        p.dispatch(to_dev_bf16(x, DEV))
        out = p.combine(p.recv_x)
        torch.cuda.synchronize()
        idx_o, _ = oracle.route(s, w.k, w.G, w.kg)
        assert np.array_equal(p.topk_idx[:T].cpu().numpy(), idx_o)
        assert bf16_ulp_diff(bf16_bits(out), x).max() <= 1
    p.close()


@pytest.mark.parametrize("E,G,kg,k,m", [(256, 8, 4, 8, 2), (64, 8, 3, 6, 2), (16, 1, 1, 2, 1),
                                        (32, 4, 2, 4, 1), (128, 8, 2, 8, 3), (8, 1, 1, 2, 1)])
def test_router_adversarial_scores(E, G, kg, k, m):
    """Exact ties, wide exponent spreads (sums binary64 cannot hold), NaN, +-0
    and +-inf: the kernel's picks equal the oracle's."""
    rng = np.random.default_rng(E + G + k)
    T = 333
    s = (rng.random((T, E)) * 2.0 ** rng.integers(-80, 3, (T, E))).astype(np.float32)
    s[::7] = np.round(s[::7] * 4) / 4                     # many exact ties
    s[1::11, : E // 2] = 1.0                              # tied groups
    s[2::13, 0] = np.nan
    s[3::17, 1] = -0.0
    s[4::19, 2] = np.inf
    s[5::23, 3] = -np.inf
    s[6::29] *= -1.0                                      # negative scores
    from combine_layout_gb300.pipeline import EpPipeline
    p = EpPipeline(synth.MODE_HT, E, E // 8 if E >= 8 else 1, T, 128, k, device=DEV)
    p.route(torch.from_numpy(s).to(DEV), T, G, kg, m, synth.W_SCORE_NORM)
    torch.cuda.synchronize()
    idx_o, w_o = oracle.route(s, k, G, kg, group_topk=m, weight_mode=oracle.W_SCORE_NORM)
    got = p.topk_idx[:T].cpu().numpy()
    bad = np.nonzero((got != idx_o).any(1))[0]
    assert bad.size == 0, (bad[:5], got[bad[:2]], idx_o[bad[:2]])
    # score-normalised weights, bit for bit (infinite and NaN sums included)
    assert_weights_match(p.topk_w[:T].cpu().numpy(), w_o, synth.W_SCORE_NORM, k)
    p.close()


@pytest.mark.parametrize("T", [1, 31, 33, 128, 255, 256, 257])
def test_ll_small_batch_layout_without_dispatch(T):
    """Small LL batches leave the counts and offsets to the first consumer:
    the layout copy, a combine and a dequantisation that come before any
    dispatch, and a second dispatch of the same route, all see the oracle's
    layout (256 tokens and fewer; 257 takes the router's own tail)."""
    E, R, S, H, k, G, kg = 64, 8, 300, 256, 6, 8, 3
    rng = np.random.default_rng(T)
    s = synth.uniform_bias_scores(rng, T, E)
    x = synth.tokens_bf16(rng, T, H)
    idx_o, w_o = oracle.route(s, k, G, kg)
    L_o, st = oracle.layout(idx_o, E, R, synth.MODE_LL, S)
    assert st == oracle.OK
    sc = torch.from_numpy(s).to(DEV)

    # layout copy straight after the route
    p = _pipe(synth.MODE_LL, E, R, S, H, k)
    p.route(sc, T, G, kg)
    L = {key: v.cpu().numpy() for key, v in p.layout().items()}
    for key in ("cnt", "off", "rcnt", "roff", "row"):
        assert np.array_equal(L[key], L_o[key]), key
    # combine before any dispatch: rows from the words; y holds each pair's token
    y = np.zeros((E * S, H), np.uint16)
    flat = L_o["row"].ravel()
    y[flat] = x[np.arange(T * k) // k]
    w32 = np.ascontiguousarray(w_o, dtype=np.float32)
    p2 = _pipe(synth.MODE_LL, E, R, S, H, k)
    p2.route(sc, T, G, kg)
    out = p2.combine(to_dev_bf16(y, DEV), topk_w=torch.from_numpy(w32).to(DEV))
    torch.cuda.synchronize()
    want = oracle.combine(y, L_o["row"], w32)
    assert bf16_ulp_diff(bf16_bits(out[:T]), want).max() <= 1
    # two dispatches of one route: the counts are right both times
    for _ in range(2):
        p2.recv_cnt.fill_(-1)
        p2.dispatch(to_dev_bf16(x, DEV))
        torch.cuda.synchronize()
        assert np.array_equal(p2.recv_cnt.cpu().numpy(), L_o["cnt"])
        got = bf16_bits(p2.recv_x[torch.from_numpy(flat.astype(np.int64)).to(DEV)])
        assert np.array_equal(got, x[np.arange(T * k) // k])
    p.close()
    p2.close()

    # dequantisation before any dispatch writes exactly the defined slots
    p3 = _pipe(synth.MODE_LL, E, R, S, H, k, fp8=True)
    p3.route(sc, T, G, kg)
    p3.recv_x.zero_()
    p3.recv_scale.fill_(1.0)
    yq = torch.full((E * S, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    p3.dequant(yq)
    torch.cuda.synchronize()
    defined = np.zeros(E * S, bool)
    defined[flat] = True
    got = yq.float().cpu().numpy()
    assert np.all(got[defined] == 0.0) and np.all(np.isnan(got[~defined]))
    p3.close()


@pytest.mark.parametrize("T", [70, 300])
def test_ll_caller_routing_masked_repeated_and_invalid(T):
    """Caller routing in LL mode (70 tokens: the deferred layout; 300: the
    router's tail): masked pairs get no slot and no combine term, invalid and
    repeated ids latch the device-error word and get no slot, and nothing is
    written outside the defined slots."""
    ep = _ep()
    E, R, H, k = 16, 4, 128, 3
    S = T
    rng = np.random.default_rng(T)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    idx[::5, 1] = -1
    idx[7, :] = -1
    idx[3, 0] = E           # out of range
    idx[9, 2] = -4          # out of range
    idx[12, 2] = idx[12, 0]  # repeated expert
    x = synth.tokens_bf16(rng, T, H)
    p = _pipe(synth.MODE_LL, E, R, S, H, k)
    guard = torch.full((p.rows + 64, H), 7, dtype=torch.bfloat16, device=DEV)
    p.recv_x = guard[: p.rows]
    p.route_given(torch.from_numpy(idx).to(DEV))
    torch.cuda.synchronize()
    bits = p.device_errors()
    assert bits & ep.MOE_EP_DEVERR_EXPERT_RANGE and bits & ep.MOE_EP_DEVERR_DUPLICATE
    p.clear_device_errors()
    L_o, st = oracle.layout(idx, E, R, oracle.MODE_LL, S)
    assert st == oracle.ERR_INVALID
    p.dispatch(to_dev_bf16(x, DEV))
    w_h = rng.random((T, k)).astype(np.float32)
    out = p.combine(p.recv_x, torch.from_numpy(w_h).to(DEV))
    torch.cuda.synchronize()
    L = {key: v.cpu().numpy() for key, v in p.layout().items()}
    for key in ("cnt", "off", "rcnt", "roff", "row"):
        assert np.array_equal(L[key], L_o[key]), key
    assert np.array_equal(p.recv_cnt.cpu().numpy(), L_o["cnt"])
    # defined slots hold their tokens; every other row keeps the guard
    defined = np.zeros(p.rows + 64, bool)
    rows = L_o["row"][L_o["row"] >= 0]
    defined[rows] = True
    g = bf16_bits(guard)
    assert np.all(g[~defined] == bf16_bits(torch.full((1,), 7, dtype=torch.bfloat16))[0])
    tok = np.nonzero(L_o["row"] >= 0)[0]
    assert np.array_equal(g[L_o["row"][L_o["row"] >= 0]], x[tok])
    # combine: no term for pairs without a slot
    y = np.zeros((p.rows, H), np.uint16)
    y[rows] = x[tok]
    want = oracle.combine(y, L_o["row"], w_h)
    assert bf16_ulp_diff(bf16_bits(out[:T]), want).max() <= 1
    assert np.all(bf16_bits(out)[7] == 0)
    assert p.device_errors() == 0
    p.close()


def test_ht_forward_replayed_from_a_cuda_graph():
    """An HT route + dispatch + combine recorded into a CUDA graph and replayed
    on new inputs (written into the captured buffers): every replay's routing,
    counts and combined tokens against the oracle.  Each replay publishes its
    counts under the sequence number of the capture, so the receive-count
    query after a replay waits for the replay's stream and returns that
    replay's counts, not the previous one's; during the capture the query is
    refused (a host wait cannot be recorded)."""
    ep = _ep()
    w = synth.WORKLOADS["ht_prefill"].with_tokens(300)
    p = _pipe(w.mode, w.E, w.R, w.T, w.H, w.k)
    s = torch.cuda.Stream(DEV)
    first = synth.make_inputs(w, 700)
    scores = torch.from_numpy(first["scores"]).to(DEV)
    x = to_dev_bf16(first["x"], DEV)
    out = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device=DEV)

    def forward():
        p.route(scores, w.T, w.G, w.kg, 0, w.weight_mode, stream=s)
        p.dispatch(x, stream=s)
        p.combine(p.recv_x, out=out, stream=s)

    with torch.cuda.stream(s):
        forward()                               # eager, outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        forward()
        with pytest.raises(ep.MoeEpError) as e:
            p.num_recv_tokens(stream=s)
        assert e.value.status == ep.MOE_EP_ERR_INVALID
    torch.cuda.synchronize()
    for i in range(3):
        inp = synth.make_inputs(w, 710 + i)
        scores.copy_(torch.from_numpy(inp["scores"]))
        x.copy_(to_dev_bf16(inp["x"], DEV))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        total, per_rank, per_expert = p.num_recv_tokens(stream=s)
        idx_o, _ = oracle.route(inp["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
        L_o, st = oracle.layout(idx_o, w.E, w.R, w.mode, w.slots)
        assert st == oracle.OK
        assert total == w.T * w.k
        assert per_rank == L_o["rcnt"].tolist() and per_expert == L_o["cnt"].tolist(), i
        torch.cuda.synchronize()
        assert np.array_equal(p.topk_idx[: w.T].cpu().numpy(), idx_o), i
        assert bf16_ulp_diff(bf16_bits(out), inp["x"]).max() <= 1, i
    p.close()

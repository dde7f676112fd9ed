"""Staged LL execution ("NCCL EP 论文解读", item "send_only与双buffer"): send-only
dispatch / combine and complete on two handles (double buffers, two
micro-batches), overlapped on two streams, and the same sequence captured in a
CUDA graph and replayed on new inputs -- LL mode has no host synchronisation
("低延迟模式": all shapes fixed, CUDA-Graph capturable).

Every micro-batch is compared with the oracle element by element: routing and
gate weights (orc_route), the layout (orc_layout), the FP8 bytes and scales of
every defined slot (orc_dispatch), the dequantised expert inputs
(orc_dequant_rows) and every combined token (orc_combine, <= 1 bf16 ulp); and
with the single-stream path bit for bit.  The receive-side signal checks of
moe_ep_complete must never time out; the signal primitives under them are
tested on their own, including a wait that runs out on a word nothing sets.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_layout_gb300 import synth
from parity import (assert_rows_equal, assert_weights_match, bf16_bits, bf16_ulp_diff,
                    defined_rows, to_dev_bf16)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
W = synth.WORKLOADS["ll_decode"]


def _make():
    from combine_layout_gb300.pipeline import EpPipeline
    ps = [EpPipeline(W.mode, W.E, W.R, W.slots, W.H, W.k, fp8=True, device=DEV) for _ in range(2)]
    ys = [torch.zeros((p.rows, W.H), dtype=torch.bfloat16, device=DEV) for p in ps]
    outs = [torch.zeros((W.T, W.H), dtype=torch.bfloat16, device=DEV) for _ in ps]
    return ps, ys, outs


def _inputs(seed):
    inp = [synth.make_inputs(W, seed + b) for b in range(2)]
    return (inp, [torch.from_numpy(i["scores"]).to(DEV) for i in inp],
            [to_dev_bf16(i["x"], DEV) for i in inp])


def _serial(ps, ys, outs, scores, xs):
    import combine_layout_gb300.moe_ep as ep
    s = torch.cuda.current_stream()
    for b, p in enumerate(ps):
        p.route(scores[b], W.T, W.G, W.kg, 0, W.weight_mode, stream=s)
        p.dispatch(xs[b], stream=s)
        p.dequant(ys[b], stream=s)
        ep.moe_ep_combine(p.handle, ys[b], p.topk_w, outs[b], ys[b].shape[0], s)


def _staged(ps, ys, outs, scores, xs, s_comm):
    import combine_layout_gb300.moe_ep as ep
    s_main = torch.cuda.current_stream()
    for b, p in enumerate(ps):
        p.route(scores[b], W.T, W.G, W.kg, 0, W.weight_mode, stream=s_main)
    routed = torch.cuda.Event()
    routed.record(s_main)
    s_comm.wait_event(routed)
    for b, p in enumerate(ps):                  # both micro-batches' dispatches in flight
        ep.moe_ep_dispatch_send(p.handle, xs[b], True, p.recv_x, p.recv_scale, p.recv_src,
                                p.recv_cnt, p.rows, s_comm)
    for b, p in enumerate(ps):
        ep.moe_ep_complete(p.handle, s_main)    # micro-batch b's tokens have arrived
        p.dequant(ys[b], stream=s_main)         # the experts (identity on the bf16 rows)
        done = torch.cuda.Event()
        done.record(s_main)
        s_comm.wait_event(done)
        ep.moe_ep_combine_send(p.handle, ys[b], p.topk_w, outs[b], ys[b].shape[0], s_comm)
    for p in ps:
        ep.moe_ep_complete(p.handle, s_main)    # join the communication stream back


def _check_oracle(p, y, out, inp):
    """One micro-batch of the staged path against the oracle, every element."""
    idx_o, w_o = oracle.route(inp["scores"], W.k, W.G, W.kg, weight_mode=W.weight_mode)
    assert np.array_equal(p.topk_idx[: W.T].cpu().numpy(), idx_o), "topk_idx"
    assert_weights_match(p.topk_w[: W.T].cpu().numpy(), w_o, W.weight_mode, W.k)
    L_o, st = oracle.layout(idx_o, W.E, W.R, W.mode, W.slots)
    assert st == oracle.OK
    L = {k: v.cpu().numpy() for k, v in p.layout().items()}
    for key in ("cnt", "off", "rcnt", "roff", "row"):
        assert np.array_equal(L[key], L_o[key]), key
    assert np.array_equal(p.recv_cnt.cpu().numpy(), L_o["cnt"])
    rows = defined_rows(W.mode, L_o["cnt"], W.slots, 0)
    rt = torch.from_numpy(rows).to(DEV)
    q_o, s_o, src_o = oracle.dispatch(inp["x"], L_o["row"], p.rows, True)
    assert np.array_equal(p.recv_src.index_select(0, rt).cpu().numpy(), src_o[rows])
    assert_rows_equal(p.recv_x.index_select(0, rt).cpu().numpy(), q_o[rows], "FP8 bytes")
    assert_rows_equal(p.recv_scale.index_select(0, rt).cpu().numpy().view(np.uint32),
                      s_o[rows].view(np.uint32), "FP8 scales")
    y_o = oracle.dequant_rows(q_o, s_o, rows)
    assert_rows_equal(bf16_bits(y.index_select(0, rt)), y_o[rows], "dequantised rows")
    want = oracle.combine(y_o, L_o["row"], np.ascontiguousarray(w_o, np.float32))
    d = bf16_ulp_diff(bf16_bits(out), want)
    assert d.max() <= 1, f"combine differs by {d.max()} bf16 ulp"
    assert p.device_errors() == 0


def test_staged_two_microbatches_match_oracle_and_serial():
    ps, ys, outs = _make()
    inp, scores, xs = _inputs(100)
    _serial(ps, ys, outs, scores, xs)
    torch.cuda.synchronize()
    want = [bf16_bits(o) for o in outs]
    for o in outs:
        o.zero_()
    for y in ys:
        y.zero_()
    s_comm = torch.cuda.Stream(DEV)
    _staged(ps, ys, outs, scores, xs, s_comm)
    torch.cuda.synchronize()
    for b in range(2):
        _check_oracle(ps[b], ys[b], outs[b], inp[b])
        assert np.array_equal(bf16_bits(outs[b]), want[b])
    for p in ps:
        p.close()


def test_staged_sequence_captured_in_a_cuda_graph():
    ps, ys, outs = _make()
    inp, scores, xs = _inputs(200)
    s_comm = torch.cuda.Stream(DEV)
    _staged(ps, ys, outs, scores, xs, s_comm)     # warm up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _staged(ps, ys, outs, scores, xs, s_comm)
    torch.cuda.synchronize()
    for seed in (300, 400, 500):                  # replay on new inputs, same buffers
        new_inp, new_scores, new_xs = _inputs(seed)
        for b in range(2):
            scores[b].copy_(new_scores[b])
            xs[b].copy_(new_xs[b])
            outs[b].zero_()
            ys[b].zero_()
        g.replay()
        torch.cuda.synchronize()
        for b in range(2):
            _check_oracle(ps[b], ys[b], outs[b], new_inp[b])
        got = [bf16_bits(o) for o in outs]
        _serial(ps, ys, outs, new_scores, new_xs)
        torch.cuda.synchronize()
        for b in range(2):
            assert np.array_equal(got[b], bf16_bits(outs[b])), (seed, b)
    for p in ps:
        p.close()


def test_complete_without_send_is_a_no_op():
    import combine_layout_gb300.moe_ep as ep
    ps, _, _ = _make()
    ep.moe_ep_complete(ps[0].handle, torch.cuda.current_stream())
    ep.moe_ep_complete(ps[0].handle, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert ps[0].device_errors() == 0
    for p in ps:
        p.close()


def test_sends_of_an_empty_batch_still_signal():
    """A route of 0 tokens: the sends launch one CTA each, which signals; the
    completes find both signals (no timeout)."""
    import combine_layout_gb300.moe_ep as ep
    ps, ys, outs = _make()
    p = ps[0]
    s = torch.cuda.current_stream()
    p.route(torch.zeros((0, W.E), device=DEV), 0, W.G, W.kg, 0, W.weight_mode, stream=s)
    ep.moe_ep_dispatch_send(p.handle, torch.zeros((1, W.H), dtype=torch.bfloat16, device=DEV),
                            True, p.recv_x, p.recv_scale, p.recv_src, p.recv_cnt, p.rows, s)
    ep.moe_ep_combine_send(p.handle, ys[0], p.topk_w, outs[0], p.rows, s)
    ep.moe_ep_complete(p.handle, s)
    torch.cuda.synchronize()
    assert p.device_errors() == 0
    assert np.all(p.recv_cnt.cpu().numpy() == 0)
    for q in ps:
        q.close()


def test_signal_add_then_wait_consumes():
    import combine_layout_gb300.moe_ep as ep
    ps, _, _ = _make()
    g = ps[0].group
    sig = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream()
    ep.moe_ep_signal_add(g, sig, 3, s)
    ep.moe_ep_wait_signal(g, sig, 2, 10 ** 9, s)
    torch.cuda.synchronize()
    assert sig.item() == 1 and ps[0].device_errors() == 0
    ep.moe_ep_wait_signal(g, sig, 1, 10 ** 9, s)
    torch.cuda.synchronize()
    assert sig.item() == 0 and ps[0].device_errors() == 0
    for p in ps:
        p.close()


def test_wait_on_a_signal_nothing_sets_times_out():
    """The bounded wait runs out (2 ms) on a word that no one adds to: the
    kernel latches the timeout bit and returns, the word is untouched, the
    group's next call reports MOE_EP_ERR_TIMEOUT, and clearing the error word
    makes the group usable again."""
    import combine_layout_gb300.moe_ep as ep
    ps, _, _ = _make()
    g = ps[0].group
    sig = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream()
    ep.moe_ep_wait_signal(g, sig, 1, 2 * 10 ** 6, s)
    torch.cuda.synchronize()
    assert ps[0].device_errors() == ep.MOE_EP_DEVERR_TIMEOUT
    assert sig.item() == 0
    with pytest.raises(ep.MoeEpError) as e:
        ep.moe_ep_signal_add(g, sig, 1, s)
    assert e.value.status == ep.MOE_EP_ERR_TIMEOUT
    ps[0].clear_device_errors()
    ep.moe_ep_signal_add(g, sig, 1, s)
    ep.moe_ep_wait_signal(g, sig, 1, 10 ** 9, s)
    torch.cuda.synchronize()
    assert sig.item() == 0 and ps[0].device_errors() == 0
    with pytest.raises(ep.MoeEpError) as e:
        ep.moe_ep_wait_signal(g, sig, 1, 0, s)            # limit out of range
    assert e.value.status == ep.MOE_EP_ERR_INVALID
    for p in ps:
        p.close()

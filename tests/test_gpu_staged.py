"""Staged LL execution: send-only dispatch / combine and complete on two
handles (double buffers, two micro-batches), overlapped on two streams, and the
same sequence captured in a CUDA graph -- LL mode has no host synchronisation
("低延迟模式": all shapes fixed, CUDA-Graph capturable).  Results must equal the
single-stream path bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from combine_layout_gb300 import synth
from parity import bf16_bits, to_dev_bf16

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
    return ([torch.from_numpy(i["scores"]).to(DEV) for i in inp],
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


def test_staged_two_microbatches_equal_serial():
    ps, ys, outs = _make()
    scores, xs = _inputs(100)
    _serial(ps, ys, outs, scores, xs)
    torch.cuda.synchronize()
    want = [bf16_bits(o) for o in outs]
    for o in outs:
        o.zero_()
    s_comm = torch.cuda.Stream(DEV)
    _staged(ps, ys, outs, scores, xs, s_comm)
    torch.cuda.synchronize()
    for b in range(2):
        assert np.array_equal(bf16_bits(outs[b]), want[b])
    for p in ps:
        p.close()


def test_staged_sequence_captured_in_a_cuda_graph():
    ps, ys, outs = _make()
    scores, xs = _inputs(200)
    s_comm = torch.cuda.Stream(DEV)
    _staged(ps, ys, outs, scores, xs, s_comm)     # warm up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _staged(ps, ys, outs, scores, xs, s_comm)
    torch.cuda.synchronize()
    for seed in (300, 400):                       # replay on new inputs, same buffers
        new_scores, new_xs = _inputs(seed)
        for b in range(2):
            scores[b].copy_(new_scores[b])
            xs[b].copy_(new_xs[b])
            outs[b].zero_()
        g.replay()
        torch.cuda.synchronize()
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
    torch.cuda.synchronize()
    for p in ps:
        p.close()

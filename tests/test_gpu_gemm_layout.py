"""GEMM-ready receive layouts: HT expert blocks padded to a row multiple
(moe_ep_set_row_align) and receive-side FP8 -> bf16 dequantisation
(moe_ep_dequant), against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_layout_gb300 import synth
from parity import bf16_bits, bf16_ulp_diff, to_dev_bf16

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SENT = 0x7BAD  # bf16 sentinel bits in rows that must stay untouched


def _pipe(w, align, fp8=None):
    from combine_layout_gb300.pipeline import EpPipeline
    return EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k,
                      fp8=w.fp8 if fp8 is None else fp8, device=DEV, align=align)


def _defined_rows(w, L):
    if w.mode == synth.MODE_HT:
        return np.concatenate([L["off"][e] + np.arange(c) for e, c in enumerate(L["cnt"])])
    return np.concatenate([e * w.slots + np.arange(c) for e, c in enumerate(L["cnt"])])


@pytest.mark.parametrize("name,T,align", [("ht_prefill", 300, 8), ("ht_prefill", 300, 128),
                                          ("skewed", 2000, 64), ("mixtral", 1000, 256),
                                          ("ht_prefill", 4096, 1)])
def test_aligned_layout_and_round_trip(name, T, align):
    w = synth.WORKLOADS[name].with_tokens(T)
    inp = synth.make_inputs(w)
    p = _pipe(w, align, fp8=False)
    p.recv_x.view(torch.int16).fill_(SENT)
    p.route(torch.from_numpy(inp["scores"]).to(DEV), T, w.G, w.kg, 0, w.weight_mode)
    total, per_rank, per_expert = p.num_recv_tokens()
    p.dispatch(to_dev_bf16(inp["x"], DEV))
    out = p.combine(p.recv_x)
    torch.cuda.synchronize()
    idx_o, _ = oracle.route(inp["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    assert np.array_equal(p.topk_idx[:T].cpu().numpy(), idx_o)
    L_o, st = oracle.layout(idx_o, w.E, w.R, oracle.MODE_HT, align=align)
    assert st == oracle.OK
    L = {k_: v.cpu().numpy() for k_, v in p.layout().items()}
    for key in ("cnt", "off", "rcnt", "roff", "row"):
        assert np.array_equal(L[key], L_o[key]), key
    assert total == int(L_o["off"][-1]) and per_expert == L_o["cnt"].tolist()
    assert per_rank == L_o["rcnt"].tolist()
    assert bf16_ulp_diff(bf16_bits(out), inp["x"]).max() <= 1
    rx = bf16_bits(p.recv_x)
    used = np.zeros(p.rows, bool)
    used[_defined_rows(w, L_o)] = True
    assert np.all(rx[~used] == SENT)          # padding and spare rows untouched
    p.close()


@pytest.mark.parametrize("name,T,align", [("ht_prefill_fp8", 300, 128), ("skewed", 1000, 1),
                                          ("ll_decode", 128, 1), ("ll_decode", 45, 1),
                                          ("ht_prefill_fp8", 4096, 1)])
def test_dequant_matches_oracle(name, T, align):
    _dequant_check(synth.WORKLOADS[name].with_tokens(T, slots=synth.WORKLOADS[name].slots or None),
                   align)


@pytest.mark.parametrize("H,T,align", [(640, 300, 1), (640, 800, 16), (512, 300, 1),
                                       (512, 800, 1), (1536, 800, 8)])
def test_dequant_hidden_sizes(H, T, align):
    """H % 512 == 0 with at least 8 rows per CTA of two per SM (T*k >= 2432
    here) takes the TMA-staged kernel (rows staged in shared memory by bulk
    copies); other widths and small batches the register-path kernel.  Both
    against the oracle."""
    w = synth.Workload("narrow", T=T, H=H, E=32, R=8, k=4, mode=synth.MODE_HT, fp8=True,
                       scores="uniform_bias", weight_mode=synth.W_SCORE_NORM, seed=3)
    _dequant_check(w, align)


def _dequant_check(w, align):
    T = w.T
    inp = synth.make_inputs(w)
    p = _pipe(w, align, fp8=True)
    p.route(torch.from_numpy(inp["scores"]).to(DEV), T, w.G, w.kg, 0, w.weight_mode)
    p.dispatch(to_dev_bf16(inp["x"], DEV))
    y = torch.full((p.rows, w.H), 0, dtype=torch.bfloat16, device=DEV)
    y.view(torch.int16).fill_(SENT)
    p.dequant(y)
    torch.cuda.synchronize()
    idx_o, _ = oracle.route(inp["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    assert np.array_equal(p.topk_idx[:T].cpu().numpy(), idx_o)
    L_o, _ = oracle.layout(idx_o, w.E, w.R, w.mode, w.slots, align=align)
    rows = _defined_rows(w, L_o)
    # the oracle dequantises its own FP8 dispatch of the same tokens
    q, sc, _ = oracle.dispatch(inp["x"], L_o["row"], p.rows, fp8=True)
    want = oracle.dequant_rows(q, sc, rows)
    got = bf16_bits(y)
    assert np.array_equal(got[rows], want[rows])
    used = np.zeros(p.rows, bool)
    used[rows] = True
    assert np.all(got[~used] == SENT)
    p.close()


def test_row_align_arguments():
    import combine_layout_gb300.moe_ep as ep
    w = synth.WORKLOADS["ht_prefill"].with_tokens(64)
    p = _pipe(w, 1, fp8=False)
    for bad in (0, 3, 2048):
        with pytest.raises(ep.MoeEpError):
            ep.moe_ep_set_row_align(p.handle, bad)
    p.close()
    wl = synth.WORKLOADS["ll_decode"]
    from combine_layout_gb300.pipeline import EpPipeline
    q = EpPipeline(wl.mode, wl.E, wl.R, wl.max_tokens, wl.H, wl.k, fp8=True, device=DEV)
    with pytest.raises(ep.MoeEpError):
        ep.moe_ep_set_row_align(q.handle, 64)     # LL layouts are slot-aligned already
    q.close()


def test_fp8_dispatch_and_dequant_in_a_cuda_graph():
    """Route, FP8 dispatch and the TMA-staged dequantisation (4096 tokens)
    captured in a CUDA graph give, replayed on new scores, what eager calls give."""
    w = synth.WORKLOADS["ht_prefill_fp8"]
    inp = synth.make_inputs(w)
    inp2 = synth.make_inputs(w, seed=w.seed + 1)
    p = _pipe(w, 1, fp8=True)
    scores = torch.from_numpy(inp["scores"]).to(DEV)
    x = to_dev_bf16(inp["x"], DEV)
    y = torch.zeros((p.rows, w.H), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()

    def step():
        p.route(scores, w.T, w.G, w.kg, 0, w.weight_mode, stream=s)
        p.dispatch(x, stream=s)
        p.dequant(y, stream=s)

    with torch.cuda.stream(s):
        step()                          # eager: sets up what the launches need
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    scores.copy_(torch.from_numpy(inp2["scores"]))
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = bf16_bits(y).copy()
    got_idx = p.topk_idx[: w.T].cpu().numpy()
    y.zero_()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    assert np.array_equal(got_idx, p.topk_idx[: w.T].cpu().numpy())
    assert np.array_equal(got, bf16_bits(y))
    idx_o, _ = oracle.route(inp2["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    assert np.array_equal(got_idx, idx_o)
    assert p.device_errors() == 0
    p.close()

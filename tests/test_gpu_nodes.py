"""GPU parity of the node-level (two-hop) layout and routing statistics
(moe_ep_node_layout) against the oracle, including the page's own routing
simulation, whose printed copy counts the device statistics must reproduce."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_layout_gb300 import synth
from conftest import read_golden

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _node_layout(p, N, src):
    import combine_layout_gb300.moe_ep as ep
    T, k = p.T, p.k
    rows = max(1, T * min(k, N))
    i32 = dict(dtype=torch.int32, device=DEV)
    cnt = torch.full((N,), -7, **i32)
    off = torch.full((N + 1,), -7, **i32)
    srcs = torch.full((rows,), -7, **i32)
    mask = torch.zeros((rows,), dtype=torch.int32, device=DEV)
    stats = torch.full((4,), -7, dtype=torch.int64, device=DEV)
    ep.moe_ep_node_layout(p.handle, N, src, cnt, off, srcs, mask, stats, rows)
    torch.cuda.synchronize()
    n = int(off[-1].item())
    return dict(cnt=cnt.cpu().numpy(), off=off.cpu().numpy(), src=srcs[:n].cpu().numpy(),
                mask=mask[:n].cpu().numpy().view(np.uint32), stats=stats.cpu().numpy())


def _check(got, want):
    for key in ("cnt", "off", "src", "mask", "stats"):
        assert np.array_equal(got[key], want[key]), key


def test_page_simulation_statistics_on_device():
    from combine_layout_gb300.pipeline import EpPipeline
    golden = {r[0]: [float(v) for v in r[1:]] for r in read_golden("page_routing_stats.txt")}
    rng = np.random.default_rng(0)
    s = synth.uniform_bias_scores(rng, 4096, 256)
    for name, G, kg in (("unlimited", 1, 1), ("limited", 8, 4)):
        p = EpPipeline(synth.MODE_HT, 256, 64, 4096, 128, 8, device=DEV)
        p.route(torch.from_numpy(s).to(DEV), 4096, G, kg, 2)
        got = _node_layout(p, 8, 0)
        idx_o, _ = oracle.route(s, 8, G, kg, group_topk=2)
        assert np.array_equal(p.topk_idx[:4096].cpu().numpy(), idx_o)
        _check(got, oracle.node_layout(idx_o, 256, 64, 8, 0))
        per_tok = (got["stats"] / 4096.0).tolist()
        assert [f"{v:.2f}" for v in per_tok] == [f"{v:.2f}" for v in golden[name][:4]], name
        p.close()


@pytest.mark.parametrize("name,T,N,src", [("ht_prefill", 300, 8, 3), ("skewed", 16384, 8, 0),
                                          ("tiny_ll", 77, 2, 1), ("mixtral", 1000, 4, 2),
                                          ("ll_decode", 128, 64, 5), ("ht_prefill", 4096, 2, 1)])
def test_node_layout_matches_oracle(name, T, N, src):
    from combine_layout_gb300.pipeline import EpPipeline
    w = synth.WORKLOADS[name].with_tokens(T, slots=synth.WORKLOADS[name].slots or None)
    inp = synth.make_inputs(w)
    p = EpPipeline(w.mode, w.E, w.R, w.max_tokens, 128, w.k, device=DEV)
    p.route(torch.from_numpy(inp["scores"]).to(DEV), T, w.G, w.kg, 0, w.weight_mode)
    got = _node_layout(p, N, src)
    idx_o, _ = oracle.route(inp["scores"], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    assert np.array_equal(p.topk_idx[:T].cpu().numpy(), idx_o)
    _check(got, oracle.node_layout(idx_o, w.E, w.R, N, src))
    p.close()


def test_node_layout_with_masked_and_repeated_ids():
    from combine_layout_gb300.pipeline import EpPipeline
    rng = np.random.default_rng(4)
    T, E, R, k = 200, 32, 8, 4
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    idx[::3, 1] = -1
    idx[::7, 2] = idx[::7, 0]           # repeated expert: counted once (error latched)
    p = EpPipeline(synth.MODE_HT, E, R, T, 128, k, device=DEV)
    p.route_given(torch.from_numpy(idx).to(DEV))
    torch.cuda.synchronize()
    p.clear_device_errors()
    got = _node_layout(p, 4, 1)
    _check(got, oracle.node_layout(idx, E, R, 4, 1))
    p.close()

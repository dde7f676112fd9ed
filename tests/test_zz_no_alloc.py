"""The allocation-free routing + layout entry point (moe_ep_route_layout_static).

Some callers cannot allocate device memory at all -- their memory pool or fixed
memory plan owns every device byte -- so they cannot create a handle, whose
workspace is allocated.  This entry point keeps its scratch in a static device
array instead.  The test calls it through the C ABI twice in a row and checks
each result against the handle-based entry points (moe_ep_route followed by
moe_ep_copy_layout) on the same inputs: routing, counts, offsets and the row
map and gate weights bit for bit (both run the same router).  It lives in a
file of its own that pytest collects last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from combine_layout_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _both(w, seed):
    import combine_layout_gb300.moe_ep as ep
    from combine_layout_gb300.pipeline import EpPipeline
    inp = synth.make_inputs(w, seed)
    scores = torch.from_numpy(inp["scores"]).to(DEV)
    T, E, R, k = w.T, w.E, w.R, w.k

    p = EpPipeline(w.mode, E, R, w.max_tokens, w.H, k, device=DEV)
    p.route(scores, T, w.G, w.kg, 0, w.weight_mode)
    ref = {k_: v.cpu().numpy() for k_, v in p.layout().items()}
    ref["idx"] = p.topk_idx[:T].cpu().numpy()
    ref["w"] = p.topk_w[:T].cpu().numpy()
    p.close()

    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(idx=torch.full((T, k), -9, **i32), w=torch.zeros((T, k), device=DEV),
               row=torch.full((T, k), -9, **i32), cnt=torch.full((E,), -9, **i32),
               off=torch.full((E + 1,), -9, **i32), rcnt=torch.full((R,), -9, **i32),
               roff=torch.full((R + 1,), -9, **i32))
    ep.moe_ep_route_layout_static(scores, T, E, R, w.mode, w.slots, k, out["idx"], out["w"],
                                  out["row"], out["cnt"], out["off"], out["rcnt"], out["roff"],
                                  w.G, w.kg, 0, w.weight_mode)
    torch.cuda.synchronize()
    got = {k_: v.cpu().numpy() for k_, v in out.items()}
    for key in ("idx", "row", "cnt", "off", "rcnt", "roff"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.array_equal(got["w"].view(np.uint32), ref["w"].view(np.uint32)), "w"


def test_static_entry_point_matches_handle_path_twice_in_a_row():
    # two calls in a row, different shapes and modes, sharing the static scratch
    _both(synth.WORKLOADS["ht_prefill"], seed=11)
    _both(synth.WORKLOADS["ll_decode"], seed=12)
    _both(synth.WORKLOADS["tiny_ll"].with_tokens(77, slots=128), seed=13)


def test_static_entry_point_at_its_capacity():
    # ceil(8192 / 32) * 256 = 65536 cells: exactly the scratch's capacity,
    # where the last group of byte counts is padded the most
    _both(synth.WORKLOADS["ht_prefill"].with_tokens(8192), seed=14)


@pytest.mark.parametrize("T", [8193, 16384])
def test_static_entry_point_rejects_sizes_beyond_its_scratch(T):
    import combine_layout_gb300.moe_ep as ep
    E = 256                      # 257 or 512 tiles x 256 experts > 65536 cells
    z = torch.zeros((T, E), device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    with pytest.raises(ep.MoeEpError) as e:
        ep.moe_ep_route_layout_static(z, T, E, 64, ep.MOE_EP_HT, 0, 8,
                                      torch.empty((T, 8), **i32), None, torch.empty((T, 8), **i32),
                                      torch.empty(E, **i32), torch.empty(E + 1, **i32),
                                      torch.empty(64, **i32), torch.empty(65, **i32), 8, 4)
    assert e.value.status == ep.MOE_EP_ERR_OVERFLOW

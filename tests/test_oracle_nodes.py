"""Pins for the oracle's node-level (two-hop) layout and routing statistics.

"NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": in high-throughput mode a
token is sent once per remote node (to the GPU in the same position) and
forwarded inside the node to the GPUs holding its experts; the page's routing
simulation prints, for 4096 tokens of a GPU on node 0, the nodes touched per
token and the cross-node copies per expert / per GPU / per node.  The oracle's
statistics reproduce every printed digit; the rows are pinned by invariants
and brute force.
"""
import numpy as np
import pytest

from combine_layout_gb300 import synth
from conftest import read_golden


def test_page_statistics_from_node_layout(orc):
    golden = {r[0]: [float(v) for v in r[1:]] for r in read_golden("page_routing_stats.txt")}
    rng = np.random.default_rng(0)
    s = synth.uniform_bias_scores(rng, 4096, 256)
    token_bytes = 7168 + 7168 // 128 * 4
    for name, G, kg in (("unlimited", 1, 1), ("limited", 8, 4)):
        idx, _ = orc.route(s, 8, num_groups=G, topk_groups=kg, group_topk=2)
        N = orc.node_layout(idx, 256, 64, 8, src_node=0)
        nodes, pe, pg, pn = (N["stats"] / 4096.0).tolist()
        got = [nodes, pe, pg, pn] + [4096 * c * token_bytes / 50e9 * 1e3 for c in (pe, pg, pn)]
        assert [f"{v:.2f}" for v in got] == [f"{v:.2f}" for v in golden[name]], (name, got)


def test_rows_and_masks_brute_force(orc):
    rng = np.random.default_rng(1)
    T, E, R, N, k = 75, 32, 8, 4, 5
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    idx[::9, 2] = -1
    L, GPN = E // R, R // N
    for src in range(N):
        out = orc.node_layout(idx, E, R, N, src_node=src)
        rows = []
        stats = np.zeros(4, np.int64)
        for n in range(N):
            for t in range(T):
                m = 0
                for e in idx[t]:
                    if e >= 0 and (e // L) // GPN == n:
                        m |= 1 << ((e // L) % GPN)
                if m:
                    rows.append((t, m))
        assert out["src"].tolist() == [r[0] for r in rows]
        assert out["mask"].tolist() == [r[1] for r in rows]
        for t in range(T):
            ex = [e for e in idx[t] if e >= 0]
            gpus = {e // L for e in ex}
            nodes = {g // GPN for g in gpus}
            stats += [len(nodes), sum(1 for e in ex if (e // L) // GPN != src),
                      len({g for g in gpus if g // GPN != src}), len(nodes - {src})]
        assert out["stats"].tolist() == stats.tolist()
        assert np.array_equal(np.diff(out["off"]), out["cnt"]) and out["off"][-1] == out["stats"][0]


def test_one_node_and_one_gpu_per_node(orc):
    idx = np.array([[0, 1, 2], [3, 2, 1]], np.int32)
    out = orc.node_layout(idx, 4, 1, 1)
    assert out["cnt"].tolist() == [2] and out["mask"].tolist() == [1, 1]
    assert out["stats"].tolist() == [2, 0, 0, 0]
    out = orc.node_layout(idx, 4, 4, 4, src_node=2)     # one GPU per node
    assert out["stats"].tolist() == [6, 4, 4, 4]


def test_node_layout_rejects_bad_shapes(orc):
    with pytest.raises(ValueError):
        orc.node_layout(np.zeros((2, 2), np.int32), 8, 4, 3)
    with pytest.raises(ValueError):
        orc.node_layout(np.zeros((2, 2), np.int32), 8, 4, 2, src_node=2)

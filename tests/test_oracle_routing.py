"""Pins for the oracle's node-limited top-k router and gate weights.

Routing follows "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": score each
node by the sum of its two best expert scores, keep the best 4 nodes, then
take the best 8 experts among them.  Pins: the page's own printed statistics
(worked example), brute-force enumeration on tiny inputs, numpy's stable
argsort for the no-limit case, and closed forms for the weights.
"""
import itertools
import math

import numpy as np
import pytest

from combine_layout_gb300 import synth
from conftest import read_golden


def _page_stats(idx, per_gpu=4, gpn=8):
    gpu = idx // per_gpu
    node = gpu // gpn
    nodes = np.mean([len(set(r)) for r in node])
    by_expert = (node != 0).sum(1).mean()
    by_gpu = np.mean([len({g for g in r if g // gpn != 0}) for r in gpu])
    by_node = np.mean([len(set(r) - {0}) for r in node])
    return nodes, by_expert, by_gpu, by_node


def test_page_printed_statistics(orc):
    """Worked example: the oracle, on the page's inputs (cast to fp32), gives every
    digit the page prints for nodes per token and cross-node copies."""
    golden = {r[0]: [float(v) for v in r[1:]] for r in read_golden("page_routing_stats.txt")}
    rng = np.random.default_rng(0)
    s = synth.uniform_bias_scores(rng, 4096, 256)
    token_bytes = 7168 + 7168 // 128 * 4
    for name, G, kg in (("unlimited", 1, 1), ("limited", 8, 4)):
        idx, _ = orc.route(s, 8, num_groups=G, topk_groups=kg, group_topk=2)
        nodes, pe, pg, pn = _page_stats(idx)
        got = [nodes, pe, pg, pn] + [4096 * c * token_bytes / 50e9 * 1e3 for c in (pe, pg, pn)]
        for g, want in zip(got, golden[name]):
            assert f"{g:.2f}" == f"{want:.2f}", (name, got, golden[name])
        if G > 1:
            assert max(len(set(r)) for r in idx // 32) <= 4


def _brute_route(s, k, G, kg, m):
    """Enumerate: group score = best m-subset sum (binary64); kept groups = the
    kg-subset with the largest total; experts = the k-subset of allowed experts
    with the largest total, listed best first.  Inputs are tie-free."""
    E = s.size
    gs = E // G
    allowed = list(range(E))
    if 1 < G and kg < G:
        gscore = []
        for n in range(G):
            vals = [float(v) for v in s[n * gs:(n + 1) * gs]]
            gscore.append(max(sum(sorted(c)) for c in itertools.combinations(vals, m)))
        best = max(itertools.combinations(range(G), kg), key=lambda c: sum(gscore[n] for n in c))
        allowed = [e for e in range(E) if e // gs in best]
    sel = max(itertools.combinations(allowed, k), key=lambda c: sum(float(s[e]) for e in c))
    return sorted(sel, key=lambda e: -float(s[e]))


@pytest.mark.parametrize("E,G,kg,k,m", [(8, 4, 2, 2, 1), (12, 4, 2, 3, 2), (16, 8, 4, 4, 2),
                                        (16, 4, 1, 3, 2), (16, 2, 1, 4, 3), (16, 1, 1, 4, 1),
                                        (9, 3, 2, 5, 2)])
def test_brute_force_tiny(orc, E, G, kg, k, m):
    rng = np.random.default_rng(E * 100 + G * 10 + k)
    for trial in range(40):
        s = rng.permutation(np.linspace(0.01, 1.0, E)).astype(np.float32) \
            + rng.random(E).astype(np.float32) * np.float32(1e-3)
        assert len(set(s.tolist())) == E
        idx, _ = orc.route(s[None, :], k, num_groups=G, topk_groups=kg, group_topk=m)
        assert idx[0].tolist() == _brute_route(s, k, G, kg, m), (trial, s)


def test_no_limit_equals_stable_argsort(orc):
    """Library special case: without a node limit the selection is numpy's stable
    argsort of the negated scores (ties: lower index first)."""
    rng = np.random.default_rng(5)
    s = rng.integers(0, 6, (500, 24)).astype(np.float32) / 4   # many exact ties
    idx, _ = orc.route(s, 5)
    want = np.argsort(-s, axis=1, kind="stable")[:, :5]
    assert np.array_equal(idx, want)


def test_tie_breaks_by_lower_index(orc):
    # two nodes tie on their group score: the lower node index is kept
    s = np.zeros((1, 8), np.float32)
    s[0, 0:2] = [0.5, 0.25]      # node 0: 0.75
    s[0, 2:4] = [0.25, 0.5]      # node 1: 0.75
    s[0, 4:6] = [0.1, 0.1]       # node 2: 0.2
    s[0, 6:8] = [0.7, 0.0]       # node 3: 0.7
    idx, _ = orc.route(s, 2, num_groups=4, topk_groups=1, group_topk=2)
    assert idx[0].tolist() == [0, 1]
    idx, _ = orc.route(s, 3, num_groups=4, topk_groups=2, group_topk=2)
    assert idx[0].tolist() == [0, 3, 1]     # 0.5 (e0), 0.5 (e3), then e1 beats e2 at 0.25
    # expert ties inside kept nodes go to the lower index
    idx, _ = orc.route(np.array([[1, 3, 3, 2, 3]], np.float32), 3)
    assert idx[0].tolist() == [1, 2, 4]


def test_ban_lowest_scoring_nodes_only(orc):
    # node 1 holds the single best expert but its second best is poor
    s = np.array([[0.6, 0.6, 0.99, 0.0, 0.55, 0.55]], np.float32)
    idx, _ = orc.route(s, 2, num_groups=3, topk_groups=2, group_topk=2)
    assert idx[0].tolist() == [0, 1]
    idx, _ = orc.route(s, 2, num_groups=3, topk_groups=2, group_topk=1)
    assert idx[0].tolist() == [2, 0]


def test_weights_closed_forms(orc):
    rng = np.random.default_rng(6)
    s = rng.random((64, 16)).astype(np.float32)
    idx, w = orc.route(s, 4, weight_mode=orc.W_SCORE_NORM)
    sel = np.take_along_axis(s.astype(np.float64), idx, 1)
    # fp32 rule: k - 1 roundings in the sum, one per quotient
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=8 * 2.0 ** -24)
    assert np.allclose(w * sel.sum(1, keepdims=True), sel, rtol=8 * 2.0 ** -24, atol=0)
    # k = 2 softmax is the logistic function of the score gap
    idx, w = orc.route(s, 2, weight_mode=orc.W_SOFTMAX_TOPK)
    sel = np.take_along_axis(s.astype(np.float64), idx, 1)
    assert np.allclose(w[:, 0], 1 / (1 + np.exp(sel[:, 1] - sel[:, 0])), rtol=1e-14, atol=0)
    # renormalising the full softmax over the selected experts cancels the full
    # denominator: same weights as the softmax over the selected scores
    idx2, w2 = orc.route(s, 2, weight_mode=orc.W_SOFTMAX_RENORM)
    assert np.array_equal(idx, idx2)
    assert np.allclose(w, w2, rtol=1e-14, atol=0)
    # k = 1: a single weight of exactly 1
    _, w1 = orc.route(s, 1, weight_mode=orc.W_SOFTMAX_TOPK)
    assert np.all(w1 == 1.0)
    _, w1 = orc.route(s, 1, weight_mode=orc.W_SCORE_NORM)
    assert np.all(w1 == 1.0)


def test_rejects_bad_parameters(orc):
    s = np.zeros((2, 8), np.float32)
    for kw in (dict(k=9), dict(k=3, num_groups=3), dict(k=5, num_groups=4, topk_groups=2),
               dict(k=2, num_groups=4, topk_groups=5)):
        with pytest.raises(ValueError):
            orc.route(s, **kw)


def test_no_limit_nodes_formula_matches_when_groups_all_kept(orc):
    rng = np.random.default_rng(7)
    s = rng.random((200, 32)).astype(np.float32)
    a, wa = orc.route(s, 4, num_groups=4, topk_groups=4)
    b, wb = orc.route(s, 4)
    assert np.array_equal(a, b) and np.array_equal(wa, wb)
    assert math.isclose(float(wa.sum()), 200.0, rel_tol=8 * 2.0 ** -24)   # fp32 weights


def test_node_scores_compare_exact_sums(orc):
    """Node scores are exact sums: (1 + 2^-60) beats (1 + 2^-61) although both
    round to 1.0 in binary64; exact rational arithmetic (fractions) decides."""
    from fractions import Fraction
    s = np.zeros((1, 8), np.float32)
    s[0, 0:2] = [1.0, 2.0 ** -61]     # node 0
    s[0, 2:4] = [0.5, 0.25]           # node 1: 0.75
    s[0, 4:6] = [1.0, 2.0 ** -60]     # node 2
    s[0, 6:8] = [0.25, 0.25]          # node 3: 0.5
    exact = [Fraction(float(s[0, 2 * n])) + Fraction(float(s[0, 2 * n + 1])) for n in range(4)]
    assert float(exact[0]) == float(exact[2]) and exact[2] > exact[0]
    idx, _ = orc.route(s, 1, num_groups=4, topk_groups=1, group_topk=2)
    assert idx[0].tolist() == [4]                       # node 2's best expert
    idx, _ = orc.route(s, 2, num_groups=4, topk_groups=2, group_topk=2)
    assert sorted(idx[0].tolist()) == [0, 4]            # nodes 2 and 0 (exact order)
    # brute force with exact rationals on random tiny scores with wide exponents
    rng = np.random.default_rng(8)
    for trial in range(200):
        v = (rng.random(12) * 2.0 ** rng.integers(-70, 2, 12)).astype(np.float32)
        idx, _ = orc.route(v[None, :], 2, num_groups=6, topk_groups=2, group_topk=2)
        gs = [sum(sorted((Fraction(float(a)) for a in v[2 * n:2 * n + 2]), reverse=True)[:2])
              for n in range(6)]
        kept = sorted(range(6), key=lambda n: (-gs[n], n))[:2]
        allowed = [e for e in range(12) if e // 2 in kept]
        want = sorted(allowed, key=lambda e: (-Fraction(float(v[e])), e))[:2]
        assert idx[0].tolist() == want, (trial, v)


def test_score_norm_weights_hand_worked(orc):
    """Score-normalised weights on hand-worked cases (tests/golden/score_norm_weights.txt):
    fp32 sum in j order (best first), one fp32 division per weight."""
    from conftest import read_golden
    rows = read_golden("score_norm_weights.txt")
    assert len(rows) == 7
    for r in rows:
        s = np.array([float.fromhex(v) for v in r[0].split(",")], np.float32)[None, :]
        want_idx = [int(v) for v in r[1].split(",")]
        want_bits = [int(v, 16) for v in r[2].split(",")]
        idx, w = orc.route(s, s.shape[1], weight_mode=orc.W_SCORE_NORM)
        assert idx[0].tolist() == want_idx, r
        got = w[0].astype(np.float32)
        assert np.array_equal(got.astype(np.float64), w[0]), "weights are fp32 values"
        assert got.view(np.uint32).tolist() == want_bits, (r, [hex(b) for b in got.view(np.uint32)])


def test_score_norm_weights_sum_and_ratio(orc):
    """Closed forms of the fp32 rule on random scores: the weights sum to 1
    within the k-term rounding bound, w_i / w_j = s_i / s_j within two
    roundings, and a -0 score gives the weight +0."""
    rng = np.random.default_rng(31)
    for k in (1, 2, 8, 16):
        s = (rng.random((300, 32)) * 2.0 ** rng.integers(-20, 20, (300, 1))).astype(np.float32)
        idx, w = orc.route(s, k, weight_mode=orc.W_SCORE_NORM)
        sel = np.take_along_axis(s.astype(np.float64), idx, 1)
        u = 2.0 ** -24
        # sum: (k - 1) roundings in the denominator, one per quotient
        assert np.all(np.abs(w.sum(1) - 1.0) <= 2 * k * u)
        assert np.allclose(w / w[:, :1], sel / sel[:, :1], rtol=4 * u, atol=0)
    s = np.array([[-0.0, -0.0, 1.0]], np.float32)
    _, w = orc.route(s, 3, weight_mode=orc.W_SCORE_NORM)
    assert w[0].tolist() == [1.0, 0.0, 0.0] and not np.signbit(w[0, 1:]).any()

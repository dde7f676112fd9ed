"""Pins for the oracle's per-rank dedup layout, receiver-side expansion and
two-stage combine.

"NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": the routing simulation
counts the copies a token needs when it is sent once per destination GPU
("按目标卡去重"), and combine sends back BF16 weighted sums of the expert
outputs.  Pins: brute-force set counting on tiny inputs, the node-layout
routine at rank granularity, expansion against the direct dispatch (byte for
byte, bf16 and FP8), closed forms where both roundings are exact, reductions
to the direct combine (one rank; one expert per rank with unit weights), and
the error bound of two roundings.
"""
import numpy as np
import pytest

from combine_layout_gb300 import synth


def _routing(rng, T, E, k, bad=True):
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    if bad:
        idx[::7, -1] = -1                      # padding
        idx[3::11, 1] = idx[3::11, 0]          # repeated expert (skipped)
    return idx


def _valid_pairs(idx, E):
    """(t, j) pairs the layout counts: id in range, first occurrence."""
    out = []
    for t in range(idx.shape[0]):
        seen = set()
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            if 0 <= e < E and e not in seen:
                out.append((t, j, e))
            if e >= 0:
                seen.add(e)
    return out


def test_brute_force_rank_layout(orc):
    rng = np.random.default_rng(0)
    T, E, R, k = 37, 24, 6, 5
    L_ = E // R
    idx = _routing(rng, T, E, k)
    L, st = orc.rank_layout(idx, E, R)
    assert st == orc.ERR_INVALID            # the repeats are reported
    need = [dict() for _ in range(T)]       # token -> {rank: mask}
    first = {}
    for t, j, e in _valid_pairs(idx, E):
        r = e // L_
        need[t][r] = need[t].get(r, 0) | (1 << (e % L_))
        first.setdefault((t, r), j)
    for r in range(R):
        toks = [t for t in range(T) if r in need[t]]
        assert L["cnt"][r] == len(toks)
        for i, t in enumerate(toks):
            q = L["off"][r] + i
            assert L["src"][q] == t and L["mask"][q] == need[t][r]
            assert L["drow"][t, first[(t, r)]] == q
    assert (L["drow"] >= 0).sum() == sum(len(n) for n in need) == L["off"][-1]


def test_rank_layout_is_node_layout_at_rank_granularity(orc):
    """One "GPU" per expert and one "node" per rank: the node routine's rows
    and GPU masks are the dedup rows and local-expert masks."""
    rng = np.random.default_rng(1)
    for T, E, R, k in ((200, 256, 64, 8), (64, 16, 4, 3), (50, 64, 2, 6)):
        idx = _routing(rng, T, E, k, bad=False)
        L, st = orc.rank_layout(idx, E, R)
        assert st == orc.OK
        N = orc.node_layout(idx, E, E, R)
        for a, b in (("cnt", "cnt"), ("off", "off"), ("src", "src"), ("mask", "mask")):
            assert np.array_equal(L[a], N[b]), a


def test_copies_per_token_match_distinct_ranks(orc):
    rng = np.random.default_rng(2)
    w = synth.WORKLOADS["ht_prefill"]
    s = synth.uniform_bias_scores(rng, 512, w.E)
    idx, _ = orc.route(s, w.k, w.G, w.kg)
    L, st = orc.rank_layout(idx, w.E, w.R)
    assert st == orc.OK
    distinct = sum(len(np.unique(r // (w.E // w.R))) for r in idx)
    assert L["off"][-1] == distinct
    assert distinct < idx.size                # some token has two experts on one rank


@pytest.mark.parametrize("fp8", [False, True])
def test_expand_of_dedup_dispatch_is_direct_dispatch(orc, fp8):
    rng = np.random.default_rng(3)
    T, H, E, R, k = 60, 256, 32, 8, 6
    x = synth.tokens_bf16(rng, T, H)
    idx = _routing(rng, T, E, k)
    D, _ = orc.layout(idx, E, R, orc.MODE_HT)
    nrows = int(D["off"][-1])
    rx, rs, rsrc = orc.dispatch(x, D["row"], nrows, fp8=fp8)
    RL, _ = orc.rank_layout(idx, E, R)
    nd = int(RL["off"][-1])
    dx, ds, dsrc = orc.dispatch(x, RL["drow"], nd, fp8=fp8)
    assert np.array_equal(dsrc, RL["src"])
    ex, es, esrc = orc.expand(dx, ds if fp8 else None, RL["src"], RL["mask"], RL["off"], E, idx,
                              D["row"], nrows)
    assert np.array_equal(ex, rx) and np.array_equal(esrc, rsrc)
    if fp8:
        assert np.array_equal(es, rs)
    assert nd < nrows                          # fewer copies cross the "network"


def _direct(orc, idx, E, R, H, y_rows_from, w, rng):
    D, _ = orc.layout(idx, E, R, orc.MODE_HT)
    nrows = int(D["off"][-1])
    y = y_rows_from(nrows)
    return D, y, orc.combine(y, D["row"], w)


def test_combine_dedup_one_rank_is_direct_combine(orc):
    """R = 1: stage 1 already rounds the full weighted sum once; stage 2
    rounds a bf16 value again, which changes nothing."""
    rng = np.random.default_rng(4)
    T, H, E, k = 40, 128, 16, 4
    idx = _routing(rng, T, E, k)
    w = rng.random((T, k)).astype(np.float32)
    D, y, want = _direct(orc, idx, E, 1, H, lambda n: synth.tokens_bf16(rng, n, H), w, rng)
    RL, _ = orc.rank_layout(idx, E, 1)
    got = orc.combine_dedup(y, idx, D["row"], w, E, 1, RL["drow"], int(RL["off"][-1]))
    assert np.array_equal(got, want)


def test_combine_dedup_one_expert_per_rank_unit_weights(orc):
    """L = 1 with unit weights: every partial is one bf16 row, exactly; the
    source's single rounding of their exact sum is the direct combine."""
    rng = np.random.default_rng(5)
    T, H, E, k = 40, 128, 16, 5
    idx = _routing(rng, T, E, k)
    w = np.ones((T, k), np.float32)
    D, y, want = _direct(orc, idx, E, E, H, lambda n: synth.tokens_bf16(rng, n, H), w, rng)
    RL, _ = orc.rank_layout(idx, E, E)
    got = orc.combine_dedup(y, idx, D["row"], w, E, E, RL["drow"], int(RL["off"][-1]))
    assert np.array_equal(got, want)


def test_combine_dedup_exact_arithmetic_closed_form(orc):
    """Small integers times halves: every partial and every sum is a bf16
    value, so both stages are exact and out = sum_j w_j y_j (numpy, float64)."""
    rng = np.random.default_rng(6)
    T, H, E, R, k = 50, 128, 32, 8, 8
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    w = rng.choice([0.5, 1.0], (T, k)).astype(np.float32)
    D, _ = orc.layout(idx, E, R, orc.MODE_HT)
    nrows = int(D["off"][-1])
    yv = rng.integers(-2, 3, (nrows, H)).astype(np.float32)
    y = synth.f32_to_bf16_bits(yv)
    RL, _ = orc.rank_layout(idx, E, R)
    got = orc.combine_dedup(y, idx, D["row"], w, E, R, RL["drow"], int(RL["off"][-1]))
    exact = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            exact[t] += float(w[t, j]) * yv[D["row"][t, j]]
    assert np.array_equal(got, synth.f32_to_bf16_bits(exact.astype(np.float32)))
    assert np.array_equal(got, orc.combine(y, D["row"], w))


def _ulp(bits):
    """bf16 unit in the last place of each value (normal range)."""
    f = np.abs(synth.bf16_bits_to_f32(bits).astype(np.float64))
    e = np.floor(np.log2(np.maximum(f, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def test_combine_dedup_within_two_rounding_bound(orc):
    """|dedup - direct| <= sum_r ulp(p_r) / 2 + ulp(out): each partial is one
    rounding of its exact sum, the source adds them exactly and rounds once."""
    rng = np.random.default_rng(7)
    T, H, E, R, k = 64, 256, 64, 16, 8
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    D, _ = orc.layout(idx, E, R, orc.MODE_HT)
    nrows = int(D["off"][-1])
    y = synth.tokens_bf16(rng, nrows, H)
    RL, _ = orc.rank_layout(idx, E, R)
    nd = int(RL["off"][-1])
    got, part = orc.combine_dedup(y, idx, D["row"], w, E, R, RL["drow"], nd, want_partial=True)
    want = orc.combine(y, D["row"], w)
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    d = synth.bf16_bits_to_f32(want).astype(np.float64)
    pu = _ulp(part)
    bound = np.zeros((T, H))
    for t in range(T):
        qs = RL["drow"][t][RL["drow"][t] >= 0]
        bound[t] = pu[qs].sum(0) / 2
    bound += np.maximum(_ulp(got), _ulp(want))
    assert np.all(np.abs(g - d) <= bound * (1 + 1e-9))
    assert np.any(got != want)                 # the two roundings do show
    # token subsets give the same rows
    sub = np.array([0, 5, 63])
    assert np.array_equal(orc.combine_dedup(y, idx, D["row"], w, E, R, RL["drow"], nd,
                                            tokens=sub), got[sub])


def test_page_copies_by_destination_gpu(orc):
    """The page's routing simulation (4096 tokens on a GPU of node 0, 8 nodes x
    8 GPUs, 4 experts per GPU): dedup rows on GPUs of other nodes, per token,
    are its printed "按目标卡去重" copies, 6.50 (no node limit) and 6.26 (4
    nodes), and their network time at 50 GB/s, 3.93 / 3.79 ms."""
    from conftest import read_golden
    golden = {r[0]: [float(v) for v in r[1:]] for r in read_golden("page_routing_stats.txt")}
    rng = np.random.default_rng(0)
    s = synth.uniform_bias_scores(rng, 4096, 256)
    token_bytes = 7168 + 7168 // 128 * 4
    for name, G, kg in (("unlimited", 1, 1), ("limited", 8, 4)):
        idx, _ = orc.route(s, 8, num_groups=G, topk_groups=kg, group_topk=2)
        L, st = orc.rank_layout(idx, 256, 64)
        assert st == orc.OK
        remote = int(L["off"][-1] - L["off"][8])          # ranks 8..63: nodes 1..7
        per_tok = remote / 4096.0
        ms = 4096 * per_tok * token_bytes / 50e9 * 1e3
        assert (f"{per_tok:.2f}", f"{ms:.2f}") == (f"{golden[name][2]:.2f}", f"{golden[name][5]:.2f}")

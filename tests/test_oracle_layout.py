"""Pins for the oracle's counting / prefix layout and dispatch packing.

Layout: count tokens per expert and rank ("NVSHMEM 与 DeepEP：GPU 发起的通信",
section "高吞吐模式"); HT output is 2D, all experts concatenated in deterministic
order with per-expert counts marking the boundaries; LL output is expert-major
with fixed slots ("NCCL EP 论文解读", "算法模式", "Tensor Layouts"; "低延迟模式" on
the DeepEP page).  Pins: invariants, brute-force counting on tiny inputs, and
numpy's stable argsort (the stable (expert, token) order is a library sort).
"""
import numpy as np
import pytest

from combine_layout_gb300 import synth
from conftest import read_golden


def _routed(orc, T=300, E=32, k=4, G=4, kg=2, seed=0):
    rng = np.random.default_rng(seed)
    s = synth.uniform_bias_scores(rng, T, E)
    idx, _ = orc.route(s, k, num_groups=G, topk_groups=kg)
    return idx


def test_ht_invariants(orc):
    T, E, R, k = 300, 32, 8, 4
    idx = _routed(orc, T, E, k)
    L, st = orc.layout(idx, E, R, orc.MODE_HT)
    assert st == orc.OK
    cnt, off, rcnt, roff, row = L["cnt"], L["off"], L["rcnt"], L["roff"], L["row"]
    assert cnt.sum() == T * k
    assert off[0] == 0 and np.array_equal(np.diff(off), cnt)
    assert np.array_equal(rcnt, cnt.reshape(R, -1).sum(1))
    assert np.array_equal(np.diff(roff), rcnt) and roff[-1] == T * k
    # bijection onto [0, T*k)
    assert np.array_equal(np.sort(row.ravel()), np.arange(T * k))
    # expert e's rows are [off[e], off[e+1]) with tokens ascending
    for e in range(E):
        t, j = np.nonzero(idx == e)
        rows = row[t, j]
        order = np.argsort(t)
        assert np.array_equal(rows[order], np.arange(off[e], off[e + 1]))


def test_ht_rows_equal_stable_argsort(orc):
    """Library special case: the HT row of the pair at flat position p is the
    position of p in numpy's stable argsort of the flattened expert ids."""
    for seed in range(3):
        idx = _routed(orc, 257, 64, 6, G=8, kg=3, seed=seed)
        L, st = orc.layout(idx, 64, 16, orc.MODE_HT)
        order = np.argsort(idx.ravel(), kind="stable")
        want = np.empty(order.size, np.int64)
        want[order] = np.arange(order.size)
        assert np.array_equal(L["row"].ravel(), want)


def test_brute_force_counting(orc):
    rng = np.random.default_rng(11)
    T, E, R, k, S = 23, 6, 3, 3, 40
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    for mode in (orc.MODE_HT, orc.MODE_LL):
        L, st = orc.layout(idx, E, R, mode, S)
        assert st == orc.OK
        for t in range(T):
            for j in range(k):
                e = idx[t, j]
                rank = sum(1 for tt in range(t) for jj in range(k) if idx[tt, jj] == e)
                cnt_before = sum(1 for tt in range(T) for jj in range(k) if idx[tt, jj] < e)
                want = cnt_before + rank if mode == orc.MODE_HT else e * S + rank
                assert L["row"][t, j] == want


def test_ll_slots_and_overflow(orc):
    T, E, R, k = 100, 16, 4, 2
    idx = _routed(orc, T, E, k, G=1, kg=1)
    L, st = orc.layout(idx, E, R, orc.MODE_LL, 128)
    assert st == orc.OK
    slot = L["row"] - idx * 128
    assert np.all((slot >= 0) & (slot < L["cnt"][idx]))
    # every (expert, slot < cnt) maps back to exactly one pair
    used = set(zip(idx.ravel().tolist(), slot.ravel().tolist()))
    assert len(used) == T * k
    # too few slots: overflow reported
    every = np.tile(np.arange(2, dtype=np.int32), (T, 1))
    L, st = orc.layout(every, E, R, orc.MODE_LL, 50)
    assert st == orc.ERR_OVERFLOW
    assert np.all(L["row"][50:] == -1) and np.all(L["row"][:50] >= 0)


def test_masked_and_invalid_pairs(orc):
    idx = np.array([[0, -1], [1, 1], [7, 2], [-5, 0]], np.int32)
    L, st = orc.layout(idx, 4, 2, orc.MODE_HT)
    assert st == orc.ERR_INVALID
    assert L["row"].tolist() == [[0, -1], [2, -1], [-1, 3], [-1, 1]]
    assert L["cnt"].tolist() == [2, 1, 1, 0]
    L, st = orc.layout(np.array([[0, -1], [-1, -1]], np.int32), 4, 2, orc.MODE_HT)
    assert st == orc.OK and L["cnt"].sum() == 1


def test_empty_batch(orc):
    L, st = orc.layout(np.zeros((0, 8), np.int32), 256, 64, orc.MODE_HT)
    assert st == orc.OK and L["cnt"].sum() == 0 and L["off"][-1] == 0


def test_dispatch_places_every_token(orc):
    T, H, E, R, k = 40, 256, 8, 4, 3
    rng = np.random.default_rng(4)
    x = synth.tokens_bf16(rng, T, H)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    L, _ = orc.layout(idx, E, R, orc.MODE_HT)
    rx, _, src = orc.dispatch(x, L["row"], T * k, fp8=False)
    assert np.array_equal(np.sort(src), np.repeat(np.arange(T), k))
    for r in range(T * k):
        assert np.array_equal(rx[r], x[src[r]])
    rq, sc, src8 = orc.dispatch(x, L["row"], T * k, fp8=True)
    assert np.array_equal(src8, src)
    for r in range(0, T * k, 7):
        q, s = orc.quant_row(x[src[r]])
        assert np.array_equal(rq[r], q) and np.array_equal(sc[r], s)


def test_page_ll_buffer_arithmetic():
    """The page's LL receive-buffer figures follow from slots x (hidden FP8 +
    hidden/128 fp32 scales + 16 B header) per (local expert, source rank)."""
    rows = [r for r in read_golden("ll_buffer_sizes.txt")]
    for r in rows:
        ranks, experts, slots, hidden, msg, total = map(int, r[:6])
        assert hidden + hidden // 128 * 4 + 16 == msg
        assert (experts // ranks) * ranks * slots * msg == total
    r0 = rows[0]
    assert f"{int(r0[5]) / 2 ** 20:.0f}" == r0[6]
    used = 128 * 64 * 8 / 256 * 4 * int(r0[4]) / 2 ** 20     # 8 of 256 experts per token
    assert f"{used:.1f}" == r0[7]
    assert round(int(rows[1][5]) / 1e6) == 121 and round(int(rows[2][5]) / 1e6) == 485


@pytest.mark.parametrize("mode", [0, 1])
def test_layout_rejects_bad_shapes(orc, mode):
    L, st = orc.layout(np.zeros((4, 2), np.int32), 10, 3, mode, 8)
    assert st == orc.ERR_INVALID


def test_aligned_layout_pads_expert_blocks(orc):
    T, E, R, k = 300, 32, 8, 4
    idx = _routed(orc, T, E, k)
    base, _ = orc.layout(idx, E, R, orc.MODE_HT)
    for align in (1, 2, 8, 128):
        L, st = orc.layout(idx, E, R, orc.MODE_HT, align=align)
        assert st == orc.OK
        pad = (base["cnt"] + align - 1) // align * align
        assert np.array_equal(L["cnt"], base["cnt"]) and np.array_equal(L["rcnt"], base["rcnt"])
        assert np.array_equal(np.diff(L["off"]), pad) and np.all(L["off"] % align == 0)
        assert np.array_equal(L["roff"], L["off"][:: E // R])
        # same in-expert ranks, shifted to the padded block starts
        e = idx
        assert np.array_equal(L["row"] - L["off"][e], base["row"] - base["off"][e])
    L1, _ = orc.layout(idx, E, R, orc.MODE_HT, align=1)
    assert all(np.array_equal(L1[k_], base[k_]) for k_ in base)


def test_dequant_closed_forms_and_torch(orc):
    import torch
    rng = np.random.default_rng(9)
    q = rng.integers(0, 256, (6, 256)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x12                   # no NaN codes
    sc = np.ones((6, 2), np.float32)
    y = orc.dequant_rows(q, sc, [0, 2])
    # scale 1: every e4m3 value is a bf16 value, exactly
    want = synth.f32_to_bf16_bits(np.array([orc.e4m3_to_double(c) for c in q[0]], np.float32))
    assert np.array_equal(y[0], want) and np.all(y[1] == 0)
    # library routine: torch's fp8 decode, fp32 product, bf16 round to nearest even
    sc = (rng.random((6, 2)) * 2.0 ** rng.integers(-20, 20, (6, 2))).astype(np.float32)
    y = orc.dequant_rows(q, sc, range(6))
    tq = torch.from_numpy(q).view(torch.float8_e4m3fn).float()
    ts = torch.from_numpy(np.repeat(sc, 128, axis=1))
    want = (tq * ts).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, want)
    # round trip: dequant(quant(x)) within half an e4m3 ulp of x
    x = synth.tokens_bf16(rng, 1, 256)[0]
    qq, ss = orc.quant_row(x)
    yy = synth.bf16_bits_to_f32(orc.dequant_rows(qq[None], ss[None], [0])[0]).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    amax = np.repeat(np.abs(xf).reshape(2, 128).max(1), 128)
    assert np.all(np.abs(yy - xf) <= np.maximum(np.abs(xf) * 2 ** -4, amax / 448 * 2 ** -10) * 1.01
                  + np.abs(xf) * 2 ** -8)

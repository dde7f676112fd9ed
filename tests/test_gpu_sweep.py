"""GPU parity over a seeded sweep of shapes the five workloads do not reach.

Each case draws experts E, ranks R, routing groups G (powers of two and
not), groups kept kg, top-k, hidden size, token count, LL or HT, bf16 or FP8,
score distribution and gate-weight rule, and runs the whole path (route,
layout, receive-count query, dispatch, combine) against the oracle element
by element, as the workload parity tests do.  Routing constraints follow the
router's: groups of E/G experts, k <= kg * E/G, m = ceil(k / kg) <= 4 scores
per group when the node limit is on, at most 16 experts per lane.  The
per-rank dedup path (HT, at most 32 local experts per rank) is swept the
same way through its own parity check.
"""
from __future__ import annotations

import numpy as np
import pytest

from combine_layout_gb300 import synth
from test_gpu_dedup import _run as _run_dedup
from test_gpu_parity import _run

pytestmark = pytest.mark.gpu


def _lanes_per_group(G: int) -> int:
    lpg = 1
    while lpg * 2 * G <= 32:
        lpg *= 2
    return lpg


def _cases(n: int = 24, seed: int = 2024, dedup: bool = False):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        E = int(rng.choice([8, 12, 16, 24, 32, 48, 64, 96, 128, 160, 256, 384, 512]))
        divs = [d for d in range(1, 33) if E % d == 0]
        G = int(rng.choice(divs))
        gs = E // G
        if -(-gs // _lanes_per_group(G)) > 16:
            continue
        kg = int(rng.integers(1, G + 1))
        kmax = min(32, kg * gs, E)
        k = int(rng.integers(1, kmax + 1))
        limit = G > 1 and kg < G
        if limit and -(-k // kg) > min(4, gs):
            continue
        R = int(rng.choice([d for d in range(1, E + 1)
                            if E % d == 0 and (not dedup or E // d <= 32)]))
        fp8 = bool(rng.random() < 0.5)
        H = int(rng.choice([128, 256, 384, 640, 1024, 2048])) if fp8 else \
            int(rng.choice([8, 24, 136, 256, 712, 1024, 4104]))
        mode = synth.MODE_HT if dedup or rng.random() < 0.5 else synth.MODE_LL
        T = int(rng.integers(1, 700))
        scores = str(rng.choice(["uniform_bias", "uniform_raw", "zipf_bias", "normal_logits"]))
        # score-normalised weights need positive scores
        wm = int(rng.choice([synth.W_SOFTMAX_TOPK, synth.W_SOFTMAX_RENORM] +
                            ([synth.W_SCORE_NORM] if scores != "normal_logits" else [])))
        out.append(synth.Workload(
            f"{'dedup' if dedup else 'sweep'}{len(out)}", T=T, H=H, E=E, R=R, k=k, mode=mode,
            fp8=fp8, scores=scores, weight_mode=wm, G=G, kg=kg,
            slots=T if mode == synth.MODE_LL else 0,
            seed=int(rng.integers(1 << 30))))
    return out


def _ids(cases):
    return [f"{c.name}-E{c.E}R{c.R}G{c.G}kg{c.kg}k{c.k}H{c.H}T{c.T}"
            f"{'LL' if c.mode == synth.MODE_LL else 'HT'}{'fp8' if c.fp8 else ''}w{c.weight_mode}"
            for c in cases]


CASES = _cases()
DEDUP_CASES = _cases(12, seed=77, dedup=True)


@pytest.mark.parametrize("w", CASES, ids=_ids(CASES))
def test_parity_sweep(w):
    _run(w)


@pytest.mark.parametrize("w", DEDUP_CASES, ids=_ids(DEDUP_CASES))
def test_dedup_parity_sweep(w):
    _run_dedup(w)


def _large_cases(n: int = 6, seed: int = 4242):
    """HT batches of 2 500 - 6 000 tokens with rows of 2 048 - 7 168 elements:
    the regime where the bf16 dispatch and the combine slice their last tokens
    (unit counts 16 - 56, so the tail slices come in 2 to 7 per row)."""
    rng = np.random.default_rng(seed)
    out = []
    for c in _cases(4 * n, seed=seed):
        if len(out) == n:
            break
        if c.mode != synth.MODE_HT:
            continue
        d = dict(c.__dict__)
        d.pop("extra")
        d["name"] = f"large{len(out)}"
        d["T"] = int(rng.integers(2500, 6001))
        d["H"] = int(rng.choice([2048, 3072, 5120, 6144, 7168]))
        out.append(synth.Workload(**d))
    return out


LARGE_CASES = _large_cases()


@pytest.mark.parametrize("w", LARGE_CASES, ids=_ids(LARGE_CASES))
def test_parity_sweep_large_batches(w):
    _run(w)

"""Seeded synthetic inputs for MoE dispatch / combine workloads.

This module only draws random numbers and lays them out: it holds none of the
routing, layout, quantisation or combine arithmetic.  It is the one piece the
tests, the benchmark and the CPU oracle's callers share.

Draw order (numpy ``default_rng(seed)``), following the routing simulation of
"NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": scores
``rng.random((T, E))`` first, then the per-expert bias ``rng.random(E) * 0.5``,
summed in binary64 and then cast to fp32 (the router's input type).  Tokens
are drawn afterwards from the same generator, ``standard_normal((T, H),
float32)``, and rounded to bf16 (nearest, ties to even).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MODE_LL, MODE_HT = 0, 1
W_SOFTMAX_TOPK, W_SOFTMAX_RENORM, W_SCORE_NORM = 0, 1, 2


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 bit patterns (nearest, ties to even)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def uniform_bias_scores(rng: np.random.Generator, T: int, E: int, bias: float = 0.5) -> np.ndarray:
    """U[0,1) scores plus a per-expert U[0, bias) offset (binary64 sum, then fp32)."""
    u = rng.random((T, E))
    b = rng.random(E) * bias
    return (u + b).astype(np.float32)


def zipf_bias_scores(rng: np.random.Generator, T: int, E: int, s: float = 1.2,
                     amp: float = 0.5) -> np.ndarray:
    """U[0,1) scores plus a Zipf(s) per-expert bias amp*(pi(e)+1)^-s, pi a random
    permutation drawn after the scores: a few hot experts."""
    u = rng.random((T, E))
    perm = rng.permutation(E)
    b = amp * (perm.astype(np.float64) + 1.0) ** (-s)
    return (u + b).astype(np.float32)


def normal_logits(rng: np.random.Generator, T: int, E: int) -> np.ndarray:
    return rng.standard_normal((T, E)).astype(np.float32)


def tokens_bf16(rng: np.random.Generator, T: int, H: int) -> np.ndarray:
    """N(0,1) token activations as bf16 bit patterns [T][H] (uint16)."""
    return f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


@dataclass(frozen=True)
class Workload:
    """One synthetic MoE dispatch/combine configuration."""
    name: str
    T: int                 # tokens on this GPU
    H: int                 # hidden size
    E: int                 # experts
    R: int                 # logical ranks (E/R local experts each)
    k: int                 # experts per token
    mode: int              # MODE_LL or MODE_HT
    fp8: bool              # FP8 e4m3 dispatch payload
    scores: str            # "uniform_bias" | "zipf_bias" | "normal_logits"
    weight_mode: int
    G: int = 1             # routing groups (nodes); 1 = no node limit
    kg: int = 1            # groups kept per token
    slots: int = 0         # LL slots per (rank, local expert) = max tokens
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def max_tokens(self) -> int:
        return self.slots if self.mode == MODE_LL else self.T

    def recv_rows(self) -> int:
        return self.E * self.slots if self.mode == MODE_LL else self.T * self.k

    def with_tokens(self, T: int, slots: int | None = None) -> "Workload":
        d = dict(self.__dict__)
        d["T"] = T
        if self.mode == MODE_LL:
            d["slots"] = max(T, 1) if slots is None else slots
        d.pop("extra")
        return Workload(**d)


WORKLOADS: dict[str, Workload] = {
    # Tiny LL round trip: 16 experts over 4 ranks, top-2, no node limit.
    "tiny_ll": Workload("tiny_ll", T=128, H=256, E=16, R=4, k=2, mode=MODE_LL, fp8=False,
                        scores="uniform_raw", weight_mode=W_SOFTMAX_TOPK, slots=128),
    # LL decode: 256 experts / 64 ranks / 8 nodes, top-8 over <= 4 nodes, FP8.
    "ll_decode": Workload("ll_decode", T=128, H=7168, E=256, R=64, k=8, mode=MODE_LL, fp8=True,
                          scores="uniform_bias", weight_mode=W_SCORE_NORM, G=8, kg=4, slots=128),
    # HT prefill (the headline workload): bf16 payload; ht_prefill_fp8 is the FP8 variant.
    "ht_prefill": Workload("ht_prefill", T=4096, H=7168, E=256, R=64, k=8, mode=MODE_HT, fp8=False,
                           scores="uniform_bias", weight_mode=W_SCORE_NORM, G=8, kg=4),
    "ht_prefill_fp8": Workload("ht_prefill_fp8", T=4096, H=7168, E=256, R=64, k=8, mode=MODE_HT,
                               fp8=True, scores="uniform_bias", weight_mode=W_SCORE_NORM, G=8, kg=4),
    # Mixtral-style: 8 experts over 8 ranks, top-2 of softmax(N(0,1) logits), renormalised.
    "mixtral": Workload("mixtral", T=8192, H=4096, E=8, R=8, k=2, mode=MODE_HT, fp8=False,
                        scores="normal_logits", weight_mode=W_SOFTMAX_RENORM),
    # Skewed stress: Zipf(1.2) per-expert bias, FP8, full dispatch + combine.
    "skewed": Workload("skewed", T=16384, H=7168, E=256, R=64, k=8, mode=MODE_HT, fp8=True,
                       scores="zipf_bias", weight_mode=W_SCORE_NORM, G=8, kg=4),
}


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Scores fp32 [T][E] and tokens bf16 bits [T][H], drawn in the stated order."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    if w.scores == "uniform_bias":
        scores = uniform_bias_scores(rng, w.T, w.E)
    elif w.scores == "uniform_raw":
        scores = rng.random((w.T, w.E)).astype(np.float32)
    elif w.scores == "zipf_bias":
        scores = zipf_bias_scores(rng, w.T, w.E)
    elif w.scores == "normal_logits":
        scores = normal_logits(rng, w.T, w.E)
    else:
        raise ValueError(w.scores)
    x = tokens_bf16(rng, w.T, w.H)
    return {"scores": scores, "x": x}

"""Benchmark: MoE expert-parallel dispatch + combine on one GB300 (libmoeep).

One step = one pass of the whole path over one batch: route (node-limited
top-k) + layout (counts, offsets) -> dispatch (+ row map) -> combine ->
receive-count query (HT: the one host synchronisation), with identity experts
(combine reads the dispatched rows; the FP8 variant's combine reads a bf16
expert-output buffer of the receive layout).

Prints one JSON line.  `value` is tokens/s of whole steps with inputs resident
in HBM; `e2e` adds, every step, the host->device copy of the step's inputs
(scores, tokens) from pinned memory and the device->host copy of the combined
output.  `roofline` is for the dominant kernel, from CUDA events recorded
around its launches on the launching stream, in a second pass of the same K
timed steps (events between kernels end the overlap of a launch with the
previous kernel's tail, so the `value` pass carries none).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ht_prefill]
  python bench.py --impl reference ...   # the CPU oracle on the host cores
Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (tokens are independent: no data-path collective), and rank 0
prints the aggregate over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from combine_layout_gb300 import synth  # noqa: E402

METRIC = "dispatch+combine tokens/s at T=4096,H=7168,top-8; achieved HBM GB/s vs peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
KERNELS_PER_STEP = 3  # route (+ layout), dispatch (+ row map), combine
# --path dedup: route, rank layout, dedup dispatch, expand, row map, partials, combine
KERNELS_PER_STEP_DEDUP = 7


# ------------------------------------------------------------------ helpers
def algorithmic_bytes(w: synth.Workload) -> dict:
    """Bytes each kernel must move per launch (DRAM, once each)."""
    T, H, k, E = w.T, w.H, w.k, w.E
    payload = H if w.fp8 else 2 * H
    scales = (H // 128) * 4 if w.fp8 else 0
    # dispatch: read the token once and its k row ids; write k rows (+ scales) and k source ids
    dispatch = T * (2 * H + k * 4) + T * k * (payload + scales + 4)
    # combine: read k rows of bf16 expert output, k row ids and k weights; write the token
    combine = T * k * (2 * H + 4 + 4) + T * 2 * H
    route = T * E * 4 + T * k * 8 + ((T + 31) // 32) * E * 4
    return {"dispatch": dispatch, "combine": combine, "route": route}


def algorithmic_bytes_dedup(w: synth.Workload, nd: int) -> dict:
    """Per-rank dedup path, nd dedup rows: dispatch = one copy per (token,
    rank) (payload, scales, token, mask) + the receiver's expansion into the
    T*k expert rows; combine = the k gathered rows and weights read, one BF16
    partial per dedup row written and read back, the token written."""
    T, H, k = w.T, w.H, w.k
    payload = H if w.fp8 else 2 * H
    scales = (H // 128) * 4 if w.fp8 else 0
    dispatch = (T * (2 * H + k * 4) + nd * (payload + scales + 8)
                + nd * (payload + scales + 8) + T * k * (payload + scales + 4))
    combine = T * k * (2 * H + 4 + 4) + 2 * nd * 2 * H + T * 2 * H
    return {"dispatch": dispatch, "combine": combine}


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload_config(w: synth.Workload, world: int, rows: int) -> dict:
    """The `config` of both arms' JSON lines (rows: receive-buffer rows)."""
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "ranks": w.R, "k": w.k,
            "nodes": w.G, "max_nodes": w.kg,
            "mode": "HT" if w.mode == synth.MODE_HT else "LL", "fp8": w.fp8,
            "l2": "inputs larger than L2: each step writes and reads a "
                  f"{rows * w.H * (1 if w.fp8 else 2) / 1e6:.0f} MB receive buffer",
            "parallelism": f"replicas x{world} (logical ranks inside each GPU)"}


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments and with whitespace runs folded:
    a comment edit does not change the kernel (string literals in these
    sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(kernel: str) -> str:
    """Hash of the code (not the comments) of a kernel's source file and of
    the shared headers it includes."""
    csrc = os.path.join(ROOT, "combine_layout_gb300", "csrc")
    h = hashlib.sha256()
    for name in (f"{kernel}.cu", "common.cuh", "layout_dev.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel, if
    the summary was taken on the current source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_b = re.search(r"traffic_bytes_per_launch_full:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != kernel_source_sha(kernel):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def rank_env() -> tuple[int, int, int]:
    """(world size, rank, local rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max_over_ranks(v: float, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, world: int, steps: int, ms: float) -> float:
    """Tokens per second of the whole job: every rank's tokens over the
    max-over-ranks time of `steps` steps."""
    return tokens_per_rank * world * steps / (ms / 1e3)


# ------------------------------------------------------------------ GPU arm
def run_gpu(args) -> dict | None:
    import torch
    import torch.distributed as dist

    from combine_layout_gb300 import moe_ep as ep
    from combine_layout_gb300.pipeline import BoundStep, EpPipeline

    world, rank, local = rank_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w, seed=w.seed + rank)
    scores_h = torch.from_numpy(inp["scores"]).pin_memory()
    x_h = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    scores = scores_h.to(dev)
    x = x_h.to(dev)
    # x is resident (or, end to end, uploaded) before each step's route and
    # nothing writes it between the route and the dispatch: the MoE-layer
    # order, so the dispatch may read its tokens while the router finishes
    p = EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k, fp8=w.fp8, device=dev,
                   x_before_route=True)
    if w.fp8:
        g = torch.Generator(device=dev)
        g.manual_seed(1234 + rank)
        y = torch.randn((p.rows, w.H), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    else:
        y = p.recv_x
    ht = w.mode == ep.MOE_EP_HT
    stream = torch.cuda.current_stream(dev)

    # The HT receive-count query (the mode's one host synchronisation) comes
    # last: the receive buffers hold the worst case (T*k rows), so neither the
    # dispatch nor the combine launch waits for the count, and the sync overlaps
    # the step's GPU work instead of splitting it.
    bs = BoundStep(p, scores, x, y, w.T, w.G, w.kg, 0, w.weight_mode, stream)

    dedup = args.path == "dedup"
    if dedup and not ht:
        raise SystemExit("--path dedup needs an HT workload")

    def step(ev=None):
        bs.route()
        if ev is not None:
            ev[0].record(stream)
        if dedup:
            p.dispatch_dedup(x, stream)
            p.expand(stream)
        else:
            bs.dispatch()
        if ev is not None:
            ev[1].record(stream)
        if dedup:
            p.combine_dedup(y, stream=stream)
        else:
            bs.combine()
        if ev is not None:
            ev[2].record(stream)
        if ht:
            bs.num_recv_tokens()

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        return reduce_max_over_ranks(v, dev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # --- device-resident timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    uuid = str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(uuid)
    time.sleep(0.05)
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms_local = t0.elapsed_time(t1)
    ms = max_over_ranks(ms_local)
    # Per-kernel durations for the roofline: the same K steps again, with
    # events recorded between the kernels.  An event between two kernels ends
    # the overlap of the second kernel's launch with the first one's tail
    # (every kernel is launched with programmatic stream serialization), so
    # these durations are taken in a pass of their own.
    barrier()
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier()
    d_ms = [e[0].elapsed_time(e[1]) for e in evs]
    c_ms = [e[1].elapsed_time(e[2]) for e in evs]

    nd = int(p.rank_off[-1].item()) if dedup else None
    if dedup:                       # the direct path's end-to-end leg only
        p.close()
        if world > 1:
            dist.destroy_process_group()
        if rank != 0:
            return None
        return _line(args, w, world, ms, d_ms, c_ms, clk, p.rows, ht, None, None, nd)

    # --- end to end: every step copies its inputs (scores, tokens) from pinned
    # host memory and its combined output back.  Inputs and outputs are double
    # buffered on the device, so the copies of neighbouring steps run on their
    # own streams while this step's kernels run.
    out_h = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    sc_d = [scores, torch.empty_like(scores)]
    x_d = [x, torch.empty_like(x)]
    out_d = [p.out, torch.empty_like(p.out)]
    steps_b = [BoundStep(p, sc_d[b], x_d[b], y, w.T, w.G, w.kg, 0, w.weight_mode, stream,
                         out=out_d[b]) for b in range(2)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_used[b])      # step i-2 is done with these input buffers
            sc_d[b].copy_(scores_h, non_blocking=True)
            x_d[b].copy_(x_h, non_blocking=True)
            ev_in[b].record(s_in)

    def e2e_step(i):
        # step i+1's inputs are enqueued before this step's count query can
        # block the host, so the host-to-device copies never wait on it
        b = i % 2
        upload(i + 1)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])         # step i-2's output has reached the host
        bs_b = steps_b[b]
        bs_b.route()
        bs_b.dispatch()
        bs_b.combine()
        ev_used[b].record(stream)
        if ht:
            bs_b.num_recv_tokens()
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_used[b])
            out_h[b].copy_(out_d[b][: w.T], non_blocking=True)
            ev_out[b].record(s_out)

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    nw = min(3, args.warmup)
    upload(0)
    for i in range(nw):
        e2e_step(i)
    torch.cuda.synchronize(dev)      # (the upload for step nw is done too)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # The timed region holds e2e_steps uploads, steps and read-backs: the
    # first timed step's inputs were uploaded before it, and its last step
    # uploads one step past the end (the same bytes); the end waits for that
    # upload too.
    e0.record(s_in)
    for i in range(nw, nw + e2e_steps):
        e2e_step(i)
    s_out.wait_event(ev_in[(nw + e2e_steps) % 2])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    out_last = out_h[(nw + e2e_steps - 1) % 2]

    # --- correctness spot check of the last step (no oracle: round trip property)
    if not w.fp8:
        rt = (out_last.float() - x_h.float()).abs().max().item()
    else:
        rt = None

    p.close()
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    e2e = {"value": whole_job_rate(w.T, world, e2e_steps, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": scores_h.numel() * 4 + x_h.numel() * 2,
           "d2h_bytes_per_step": out_h[0].numel() * 2, "steps": e2e_steps,
           "overlap": "double-buffered inputs/outputs; copies on their own streams; each "
                      "step enqueues the next step's upload before its count query"}
    return _line(args, w, world, ms, d_ms, c_ms, clk, p.rows, ht, e2e, rt, None)


def _line(args, w, world, ms, d_ms, c_ms, clk, rows, ht, e2e, rt, nd):
    """The JSON line of one timed run (nd: dedup rows of the dedup path, else None)."""
    value = whole_job_rate(w.T, world, args.steps, ms)
    ab = algorithmic_bytes(w) if nd is None else algorithmic_bytes_dedup(w, nd)
    d_avg = statistics.mean(d_ms)
    c_avg = statistics.mean(c_ms)
    dom = "dispatch" if d_avg >= c_avg else "combine"
    dom_ms = d_avg if dom == "dispatch" else c_avg
    peak, peak_src = measured_peak_gbs()
    achieved = ab[dom] / (dom_ms / 1e3) / 1e9
    traffic = profiled_traffic(dom, w.name) if nd is None else None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e4m3 dispatch payload, bf16 combine (fp32 accumulate)" if w.fp8
                  else "bf16 (fp32 combine accumulate)"),
        "data": "synthetic (seeded numpy: U[0,1)+U[0,0.5) per-expert bias scores, N(0,1) bf16 tokens)",
        "config": {**workload_config(w, world, rows),
                   **({} if nd is None else {"path": "dedup", "dedup_rows": nd})},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_source": f"{peak_src} hbm_gbs (copy, burst)", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": ab[dom]},
        "breakdown": {
            "timing": "second pass of the same K steps with CUDA events between the kernels",
            "dispatch_us": d_avg * 1e3, "combine_us": c_avg * 1e3,
            "dispatch_GBps": ab["dispatch"] / (d_avg / 1e3) / 1e9,
            "combine_GBps": ab["combine"] / (c_avg / 1e3) / 1e9,
            "dispatch_frac": ab["dispatch"] / (d_avg / 1e3) / 1e9 / peak,
            "combine_frac": ab["combine"] / (c_avg / 1e3) / 1e9 / peak,
            "route_layout_query_us_by_difference": (ms / args.steps - d_avg - c_avg) * 1e3,
            "dispatch_combine_tokens_per_s": w.T / ((d_avg + c_avg) / 1e3),
        },
        "e2e": e2e,
        "gpu_launches": (KERNELS_PER_STEP if nd is None else KERNELS_PER_STEP_DEDUP) * args.steps,
        "x_before_route": True,
        "clocks": clk,
        "round_trip_max_abs_err": rt,
    }
    return line


# ------------------------------------------------------------------ CPU oracle
def oracle_step(orc, w: synth.Workload, scores, x, T):
    idx, wts = orc.route(scores[:T], w.k, w.G, w.kg, weight_mode=w.weight_mode)
    L, _ = orc.layout(idx, w.E, w.R, w.mode, w.slots)
    rows = w.E * w.slots if w.mode == synth.MODE_LL else T * w.k
    rx, rs, _ = orc.dispatch(x[:T], L["row"], rows, w.fp8)
    y = rx if not w.fp8 else x[:T][np.arange(rows) % T]   # identity expert (bf16 expert outputs)
    orc.combine(y, L["row"], wts.astype(np.float32))


def cpu_oracle_rate(w: synth.Workload, sample_tokens: int, seconds: float):
    import oracle as orc
    orc.build()
    inp = synth.make_inputs(w)
    T = min(sample_tokens, w.T)
    oracle_step(orc, w, inp["scores"], inp["x"], min(T, 8))   # warm caches / build
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(orc, w, inp["scores"], inp["x"], T)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return T * n / el, T, n, el


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle as orc
    orc.build()
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w)
    # per-token cost, then a sample size that keeps the whole run to ~90 s
    t0 = time.perf_counter()
    oracle_step(orc, w, inp["scores"], inp["x"], 32)
    per_tok = (time.perf_counter() - t0) / 32
    budget = 90.0 / max(1, args.steps + args.warmup)
    T = int(max(1, min(w.T, budget / per_tok)))
    for _ in range(args.warmup):
        oracle_step(orc, w, inp["scores"], inp["x"], T)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(orc, w, inp["scores"], inp["x"], T)
    el = time.perf_counter() - t0
    value = T * args.steps / el
    sample = f"first {T} of {w.T} tokens per step (full H, E, k), {args.steps} steps"
    rows = w.E * w.slots if w.mode == synth.MODE_LL else w.T * w.k
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 oracle (fp32 FP8 decisions)",
            "data": "synthetic (seeded numpy)", "impl": "reference",
            "config": workload_config(w, args.gpus, rows),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ht_prefill", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-sample-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="direct", choices=["direct", "dedup"],
                    help="dedup: one copy per (token, rank), expanded on the receiver, "
                         "two-stage combine (HT workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")

    if args.impl == "reference":
        line = run_reference(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    line = run_gpu(args)
    if line is None:
        return
    if not args.no_cpu_baseline and line["n_gpus"] == 1:
        rate, T, n, el = cpu_oracle_rate(synth.WORKLOADS[args.workload], args.cpu_sample_tokens,
                                         args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{n} oracle steps of the first {T} tokens "
                                          f"(full H, E, k) in {el:.1f} s, single thread"}
    else:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

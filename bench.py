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
previous kernel's tail, so the `value` pass carries none).  Each workload's
entry also carries its kernels launched back to back (launches overlapping,
as in a step) and, for LL workloads, the step replayed from a CUDA graph.

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


L2_BYTES_NOMINAL = 126 * 2**20  # GB300 (the device's own figure is used when known)


def step_bytes(w: synth.Workload) -> int:
    """Bytes one step touches (route, dispatch and combine: the algorithmic bytes)."""
    ab = algorithmic_bytes(w)
    return ab["route"] + ab["dispatch"] + ab["combine"]


def flushes_l2(w: synth.Workload, l2_bytes: int = L2_BYTES_NOMINAL) -> bool:
    """A step that touches less than twice the L2 would find its inputs there
    from the step before: such workloads flush the L2 before every timed step."""
    return step_bytes(w) < 2 * l2_bytes


def workload_config(w: synth.Workload, world: int, rows: int) -> dict:
    """The `config` of both arms' JSON lines (rows: receive-buffer rows)."""
    if flushes_l2(w):
        l2 = (f"step touches {step_bytes(w) / 1e6:.0f} MB, less than twice L2: L2 flushed "
              "(a read of a buffer twice its size) before every timed step, each step timed "
              "between its own events")
    else:
        l2 = ("inputs larger than L2: each step writes and reads a "
              f"{rows * w.H * (1 if w.fp8 else 2) / 1e6:.0f} MB receive buffer "
              f"({step_bytes(w) / 1e6:.0f} MB touched per step)")
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "ranks": w.R, "k": w.k,
            "nodes": w.G, "max_nodes": w.kg,
            "mode": "HT" if w.mode == synth.MODE_HT else "LL", "fp8": w.fp8,
            "l2": l2, "parallelism": f"replicas x{world} (logical ranks inside each GPU)"}


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


# ------------------------------------------------------------------ timing
def agreed_passes(first_pass_ms: float, min_seconds: float, max_passes: int = 2000,
                  device=None) -> int:
    """Timed passes of K steps every rank runs: enough for min_seconds of GPU
    time at the slowest rank's first-pass time, at least 3.  Every rank gets
    the same number (the barriers around each pass must pair up)."""
    ms = reduce_max_over_ranks(max(first_pass_ms, 1e-3), device)
    return int(min(max_passes, max(3, -(-min_seconds * 1e3 // ms))))


def numa_of_buffer(addr: int, nbytes: int) -> dict:
    """NUMA nodes holding the pages of [addr, addr + nbytes): pages per node,
    from /proc/self/maps and /proc/self/numa_maps (Linux)."""
    try:
        spans = []
        with open("/proc/self/maps") as f:
            for line in f:
                a, b = line.split()[0].split("-")
                spans.append((int(a, 16), int(b, 16)))
        nodes: dict[str, int] = {}
        with open("/proc/self/numa_maps") as f:
            for line, (a, b) in zip(f, spans):
                if b <= addr or a >= addr + nbytes:
                    continue
                for tok in line.split()[1:]:
                    m = re.fullmatch(r"N(\d+)=(\d+)", tok)
                    if m:
                        nodes[m.group(1)] = nodes.get(m.group(1), 0) + int(m.group(2))
        return nodes
    except Exception as e:   # not Linux, or the files are not readable
        return {"unknown": str(e)}


def gpu_numa_node(pci_bus_id: str | None) -> int | None:
    """The NUMA node the GPU's PCI function reports (-1: none)."""
    if not pci_bus_id:
        return None
    bus = pci_bus_id.lower()
    if bus.count(":") == 2 and len(bus.split(":")[0]) == 8:
        bus = bus[4:]                                   # 00000000:xx:... -> 0000:xx:...
    try:
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            return int(f.read().strip())
    except Exception:
        return None


def measure_link(dev, nbytes: int = 256 << 20, reps: int = 5) -> dict:
    """Host<->device copy bandwidth with pinned host memory: host->device,
    device->host and both directions at once (two streams), best of `reps`,
    CUDA events; and where the pinned pages live."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_in.fill_(1)
    h_out.fill_(2)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, streams):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0 = [torch.cuda.Event(enable_timing=True) for _ in streams]
            e1 = [torch.cuda.Event(enable_timing=True) for _ in streams]
            for s, e in zip(streams, e0):
                e.record(s)
            fn()
            for s, e in zip(streams, e1):
                e.record(s)
            torch.cuda.synchronize(dev)
            t = max(e0[0].elapsed_time(b) for b in e1)
            best = min(best, t)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in = timed(h2d, [s1])
    t_out = timed(d2h, [s2])
    t_both = timed(both, [s1, s2])
    props = torch.cuda.get_device_properties(dev)
    bus = None
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=uuid,pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout
        uuid = str(props.uuid).replace("GPU-", "")
        for line in out.splitlines():
            u, b = [x.strip() for x in line.split(",")]
            if uuid in u:
                bus = b
    except Exception:
        pass
    cpus = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else []
    return {"h2d_GBps": nbytes / (t_in / 1e3) / 1e9, "d2h_GBps": nbytes / (t_out / 1e3) / 1e9,
            "both_GBps": 2 * nbytes / (t_both / 1e3) / 1e9, "bytes_per_copy": nbytes,
            "how": f"pinned host memory (torch pin_memory), copy_ on its own stream, best of {reps}; "
                   "both = one copy each way at once on two streams",
            "numa": {"pinned_in_pages_by_node": numa_of_buffer(h_in.data_ptr(), nbytes),
                     "pinned_out_pages_by_node": numa_of_buffer(h_out.data_ptr(), nbytes),
                     "gpu_pci": bus, "gpu_numa_node": gpu_numa_node(bus),
                     "cpus_allowed": f"{cpus[0]}-{cpus[-1]} ({len(cpus)})" if cpus else None}}


# ------------------------------------------------------------------ GPU arm
class WorkloadRun:
    """One workload on fixed buffers: its pipeline, inputs and bound step."""

    def __init__(self, w: synth.Workload, dev, stream, rank: int, dedup: bool = False):
        import torch

        from combine_layout_gb300 import moe_ep as ep
        from combine_layout_gb300.pipeline import BoundStep, EpPipeline
        self.w, self.dev, self.stream, self.dedup = w, dev, stream, dedup
        inp = synth.make_inputs(w, seed=w.seed + rank)
        self.scores_h = torch.from_numpy(inp["scores"]).pin_memory()
        self.x_h = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
        self.scores = self.scores_h.to(dev)
        self.x = self.x_h.to(dev)
        # x is resident (or, end to end, uploaded) before each step's route and
        # nothing writes it between the route and the dispatch: the MoE-layer
        # order, so the dispatch may read its tokens while the router finishes
        self.p = EpPipeline(w.mode, w.E, w.R, w.max_tokens, w.H, w.k, fp8=w.fp8, device=dev,
                            x_before_route=True)
        if w.fp8:
            g = torch.Generator(device=dev)
            g.manual_seed(1234 + rank)
            self.y = torch.randn((self.p.rows, w.H), generator=g, device=dev,
                                 dtype=torch.float32).to(torch.bfloat16)
        else:
            self.y = self.p.recv_x
        self.ht = w.mode == ep.MOE_EP_HT
        if dedup and not self.ht:
            raise SystemExit("--path dedup needs an HT workload")
        # The HT receive-count query (the mode's one host synchronisation)
        # comes last: the receive buffers hold the worst case (T*k rows), so
        # neither the dispatch nor the combine launch waits for the count,
        # and the sync overlaps the step's GPU work instead of splitting it.
        self.bs = BoundStep(self.p, self.scores, self.x, self.y, w.T, w.G, w.kg, 0,
                            w.weight_mode, stream)
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES_NOMINAL
        self.flush = (torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
                      if flushes_l2(w, l2) else None)

    def flush_l2(self):
        """Read a buffer twice the L2's size on the launching stream: the L2
        then holds none of the step's data, and only clean lines to evict."""
        if self.flush is not None:
            self.flush.max()

    def step(self, ev=None):
        p, bs, s = self.p, self.bs, self.stream
        if ev is not None:
            ev[0].record(s)
        bs.route()
        if ev is not None:
            ev[1].record(s)
        if self.dedup:
            p.dispatch_dedup(self.x, s)
            p.expand(s)
        else:
            bs.dispatch()
        if ev is not None:
            ev[2].record(s)
        if self.dedup:
            p.combine_dedup(self.y, stream=s)
        else:
            bs.combine()
        if ev is not None:
            ev[3].record(s)
        if self.ht:
            bs.num_recv_tokens()

    def timed(self, steps: int, warmup: int, min_seconds: float, barrier, uuid) -> dict:
        """W warm-up steps; passes of exactly K steps, each bracketed by a
        barrier and a synchronize and timed with CUDA events on the launching
        stream, repeated (the same count on every rank) until min_seconds of
        GPU time; then one more K-step pass with events between the kernels.
        Clocks are sampled over all of it."""
        import torch
        dev, s = self.dev, self.stream
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(uuid)
        time.sleep(0.1)

        ea = eb = None
        if self.flush is not None:
            ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]

        def one_pass():
            barrier()
            torch.cuda.synchronize(dev)
            if self.flush is None:
                t0.record(s)
                for _ in range(steps):
                    self.step()
                t1.record(s)
                torch.cuda.synchronize(dev)
                barrier()
                return t0.elapsed_time(t1)
            # a small step: the L2 is flushed before each step, outside its events
            for i in range(steps):
                self.flush_l2()
                ea[i].record(s)
                self.step()
                eb[i].record(s)
            torch.cuda.synchronize(dev)
            barrier()
            return sum(ea[i].elapsed_time(eb[i]) for i in range(steps))

        passes = [one_pass()]
        n = agreed_passes(passes[0], min_seconds, device=dev)
        passes += [one_pass() for _ in range(n - 1)]
        warm = None
        if self.flush is not None:
            # context only: the same K steps back to back with no flush (the
            # step's data stays in L2 from one step to the next)
            barrier()
            torch.cuda.synchronize(dev)
            t0.record(s)
            for _ in range(steps):
                self.step()
            t1.record(s)
            torch.cuda.synchronize(dev)
            barrier()
            warm = t0.elapsed_time(t1)
        # Per-kernel durations for the roofline: one more K-step pass with
        # events recorded between the kernels.  An event between two kernels
        # ends the overlap of the second kernel's launch with the first one's
        # tail (every kernel is launched with programmatic stream
        # serialization), so these durations are taken in a pass of their own.
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        barrier()
        torch.cuda.synchronize(dev)
        for i in range(steps):
            self.flush_l2()
            self.step(evs[i])
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        barrier()
        return {"pass_ms": passes, "clocks": clk, "warm_pass_ms": warm,
                "r_ms": [e[0].elapsed_time(e[1]) for e in evs],
                "d_ms": [e[1].elapsed_time(e[2]) for e in evs],
                "c_ms": [e[2].elapsed_time(e[3]) for e in evs]}

    def back_to_back(self, reps: int = 3) -> dict:
        """Each kernel launched n times in a row between two CUDA events on the
        launching stream, median of reps: microseconds per launch.  Launches
        overlap the previous launch's tail, as the kernels of a step do, so
        these durations carry no event gap (the event-timed ones do)."""
        import torch
        n = 200 if self.w.T <= 1024 else 50
        out = {"launches": n, "how": "n launches of one kernel back to back between two CUDA "
                                     "events on the launching stream, per launch, median of "
                                     f"{reps}" + ("; the same inputs each launch, so a step "
                                                  "smaller than L2 runs from L2 here"
                                                  if self.flush is not None else "")}
        for name, fn in (("route_us", self.bs.route), ("dispatch_us", self.bs.dispatch),
                         ("combine_us", self.bs.combine)):
            t = []
            for _ in range(reps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize(self.dev)
                a.record(self.stream)
                for _ in range(n):
                    fn()
                b.record(self.stream)
                torch.cuda.synchronize(self.dev)
                t.append(a.elapsed_time(b) * 1e3 / n)
            out[name] = statistics.median(t)
        return out

    def close(self):
        self.p.close()


def graph_step_us(w: synth.Workload, dev, rank: int, n: int = 200) -> dict:
    """An LL workload's step (route, dispatch, combine: no host synchronisation)
    replayed from a CUDA graph on a side stream, without host launches (how a
    decode loop runs it): `us`, a one-step graph replayed n times, each replay
    between its own events after an L2 flush (when the step is smaller than
    L2), the mean; `us_l2_warm` (context), a graph of 20 steps replayed back
    to back, per step."""
    import torch
    s = torch.cuda.Stream(dev)
    out = {}
    with torch.cuda.stream(s):
        r = WorkloadRun(w, dev, s, rank)
        for _ in range(3):
            r.step()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            r.step()
        g.replay()
        torch.cuda.synchronize(dev)
        ea = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        eb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            r.flush_l2()
            ea[i].record(s)
            g.replay()
            eb[i].record(s)
        torch.cuda.synchronize(dev)
        out["us"] = statistics.mean(ea[i].elapsed_time(eb[i]) * 1e3 for i in range(n))
        del g
        g20 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g20, stream=s):
            for _ in range(20):
                r.step()
        g20.replay()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(10):
            g20.replay()
        b.record(s)
        torch.cuda.synchronize(dev)
        out["us_l2_warm"] = a.elapsed_time(b) * 1e3 / 200
        del g20
        r.close()
    return out


def secondary_line(w: synth.Workload, r: dict, steps: int) -> dict:
    """Per-workload figures for the `secondary` object: the step time (median
    pass), each kernel's event-timed duration and its algorithmic bandwidth
    against the measured copy peak and the nominal 8 TB/s."""
    ab = algorithmic_bytes(w)
    peak, _ = measured_peak_gbs()
    step_ms = statistics.median(r["pass_ms"]) / steps
    d = statistics.mean(r["d_ms"])
    c = statistics.mean(r["c_ms"])
    ro = statistics.mean(r["r_ms"])
    gbs = lambda b, ms: b / (ms / 1e3) / 1e9  # noqa: E731
    total = ab["route"] + ab["dispatch"] + ab["combine"]
    return {"T": w.T, "H": w.H, "E": w.E, "k": w.k,
            "mode": "HT" if w.mode == synth.MODE_HT else "LL", "fp8": w.fp8,
            "step_us": step_ms * 1e3, "tokens_per_s": w.T / (step_ms / 1e3),
            "passes": len(r["pass_ms"]),
            "route_us": ro * 1e3, "dispatch_us": d * 1e3, "combine_us": c * 1e3,
            "dispatch_GBps": gbs(ab["dispatch"], d), "combine_GBps": gbs(ab["combine"], c),
            "dispatch_frac": gbs(ab["dispatch"], d) / peak,
            "combine_frac": gbs(ab["combine"], c) / peak,
            "dispatch_frac_of_8TBps": gbs(ab["dispatch"], d) / 8000.0,
            "combine_frac_of_8TBps": gbs(ab["combine"], c) / 8000.0,
            "step_GBps": gbs(total, step_ms),
            "route_layout_query_us_by_difference": (step_ms - d - c) * 1e3,
            "event_timing": "route, dispatch and combine each between CUDA events (no launch "
                            "overlap) in one more pass of K steps",
            "algorithmic_bytes": ab, "l2": workload_config(w, 1, w.recv_rows())["l2"],
            **({"step_us_l2_warm": r["warm_pass_ms"] / steps * 1e3}
               if r.get("warm_pass_ms") is not None else {}),
            "back_to_back": r.get("b2b"), "clocks": r["clocks"]}


def run_gpu(args) -> dict | None:
    import torch
    import torch.distributed as dist

    world, rank, local = rank_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    uuid = str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        return reduce_max_over_ranks(v, dev)

    w = synth.WORKLOADS[args.workload]
    dedup = args.path == "dedup"
    run = WorkloadRun(w, dev, stream, rank, dedup)
    p = run.p
    r = run.timed(args.steps, args.warmup, args.min_seconds, barrier, uuid)
    b2b = None if dedup or args.no_b2b else run.back_to_back()
    # the job's time: each rank's median pass, the slowest rank's
    ms = max_over_ranks(statistics.median(r["pass_ms"]))
    d_ms, c_ms, clk = r["d_ms"], r["c_ms"], r["clocks"]
    clk["route_us_event_timed"] = statistics.mean(r["r_ms"]) * 1e3
    clk["passes"] = len(r["pass_ms"])

    nd = int(p.rank_off[-1].item()) if dedup else None
    if dedup:                       # the direct path's end-to-end leg only
        run.close()
        if world > 1:
            dist.destroy_process_group()
        if rank != 0:
            return None
        return _line(args, w, world, ms, d_ms, c_ms, clk, p.rows, run.ht, None, None, nd)

    # --- end to end: every step copies its inputs (scores, tokens) from pinned
    # host memory and its combined output back.  Inputs and outputs are double
    # buffered on the device, so the copies of neighbouring steps run on their
    # own streams while this step's kernels run.
    from combine_layout_gb300.pipeline import BoundStep
    scores_h, x_h, scores, x, y, ht = run.scores_h, run.x_h, run.scores, run.x, run.y, run.ht
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

    # its own step count (not K): the double-buffered pipeline's fill and
    # drain are a small share of 200 steps, a large one of 20
    e2e_steps = max(1, args.e2e_steps)
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

    run.close()
    del sc_d, x_d, out_d, steps_b, run, p
    torch.cuda.empty_cache()
    link = measure_link(dev) if world == 1 else None   # one process: nothing else on the link
    graph = (graph_step_us(w, dev, rank)
             if w.mode == synth.MODE_LL and not args.no_b2b and world == 1 else None)

    # --- the other workloads, same process and GPU, one line's `secondary`
    secondary = {}
    if world == 1 and args.secondary:
        for name in args.secondary.split(","):
            if name == w.name:
                continue
            ws = synth.WORKLOADS[name]
            rs = WorkloadRun(ws, dev, stream, rank)
            r2 = rs.timed(args.steps, args.warmup, args.secondary_seconds, barrier, uuid)
            r2["b2b"] = None if args.no_b2b else rs.back_to_back()
            rs.close()
            del rs
            torch.cuda.empty_cache()
            secondary[name] = secondary_line(ws, r2, args.steps)
            if ws.mode == synth.MODE_LL and not args.no_b2b:
                gr = graph_step_us(ws, dev, rank)
                secondary[name]["step_graph_us"] = gr["us"]
                secondary[name]["step_graph_us_l2_warm"] = gr["us_l2_warm"]
                torch.cuda.empty_cache()

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    h2d = scores_h.numel() * 4 + x_h.numel() * 2
    d2h = out_h[0].numel() * 2
    e2e = {"value": whole_job_rate(w.T, world, e2e_steps, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "overlap": "double-buffered inputs/outputs; copies on their own streams; each "
                      "step enqueues the next step's upload before its count query",
           "link_GBps": (h2d + d2h) / (e2e_ms / e2e_steps / 1e3) / 1e9}
    if link is not None:
        e2e["link_peak"] = link
        e2e["link_frac_of_both"] = e2e["link_GBps"] / link["both_GBps"]
    line = _line(args, w, world, ms, d_ms, c_ms, clk, w.recv_rows(), ht, e2e, rt, None)
    line["breakdown"]["back_to_back"] = b2b
    if graph is not None:
        line["breakdown"]["step_graph_us"] = graph["us"]
        line["breakdown"]["step_graph_us_l2_warm"] = graph["us_l2_warm"]
    if r.get("warm_pass_ms") is not None:
        line["breakdown"]["step_us_l2_warm"] = r["warm_pass_ms"] / args.steps * 1e3
    if secondary:
        line["secondary"] = secondary
    return line


def _line(args, w, world, ms, d_ms, c_ms, clk, rows, ht, e2e, rt, nd):
    """The JSON line of one timed run (nd: dedup rows of the dedup path, else None)."""
    value = whole_job_rate(w.T, world, args.steps, ms)
    ab = algorithmic_bytes(w) if nd is None else algorithmic_bytes_dedup(w, nd)
    d_avg = statistics.mean(d_ms)
    c_avg = statistics.mean(c_ms)
    route_us = clk.pop("route_us_event_timed", None)
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
        "timing": {"passes": clk.get("passes"),
                   "how": "passes of exactly K steps, each bracketed by a barrier and a "
                          "synchronize and timed with CUDA events on the launching stream, "
                          "repeated until >= --min-seconds of GPU time; ms_per_step is the "
                          "median pass / K (max over ranks)" +
                          ("; a step smaller than L2: the L2 flushed before every step and "
                           "each step timed between its own events, a pass being their sum"
                           if flushes_l2(w) else ""),
                   "sm_kcycles_per_step": (ms / args.steps * clk["sm_mhz"]
                                           if clk.get("sm_mhz") else None)},
        "breakdown": {
            "timing": "one more pass of K steps with CUDA events between the kernels",
            "route_us": route_us, "dispatch_us": d_avg * 1e3, "combine_us": c_avg * 1e3,
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
                             "host_cores": os.cpu_count(), "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _oracle_worker(name: str, scores, x, seconds: float):
    """One process of the all-core CPU baseline: the oracle on its own copy of
    the token sample, repeated for `seconds`.  Returns (tokens, seconds)."""
    import oracle as orc
    w = synth.WORKLOADS[name]
    T = x.shape[0]
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(orc, w, scores, x, T)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return T * n, el


def cpu_oracle_rate_all_cores(w: synth.Workload, sample_tokens: int, seconds: float):
    """The oracle on every host core at once (one spawned process per core,
    each on the same token sample): tokens of all processes over the longest
    one's time."""
    import multiprocessing as mp

    import oracle as orc
    orc.build()
    n = os.cpu_count() or 1
    inp = synth.make_inputs(w)
    T = min(sample_tokens, w.T)
    args = [(w.name, inp["scores"][:T].copy(), inp["x"][:T].copy(), seconds)] * n
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.starmap(_oracle_worker, args)
    return sum(r[0] for r in res) / max(r[1] for r in res), n


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ht_prefill", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--cpu-all-core-seconds", type=float, default=4.0)
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="repeat the K-step timed pass until this much GPU time has passed")
    ap.add_argument("--secondary", default="ht_prefill_fp8,skewed,mixtral,ll_decode",
                    help="other workloads measured in the same process (N = 1), '' for none")
    ap.add_argument("--secondary-seconds", type=float, default=0.25)
    ap.add_argument("--link-peak", action="store_true",
                    help="only measure the host<->device copy bandwidth and print it")
    ap.add_argument("--cpu-sample-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-b2b", action="store_true",
                    help="skip the back-to-back kernel and CUDA-graph step timings "
                         "(profiling runs: fewer launches)")
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
    if args.link_peak:
        import torch
        link = measure_link(torch.device("cuda", 0))
        print(json.dumps({"metric": "host<->device copy GB/s (pinned host memory)", **link}),
              flush=True)
        return

    line = run_gpu(args)
    if line is None:
        return
    if not args.no_cpu_baseline and line["n_gpus"] == 1:
        rate, T, n, el = cpu_oracle_rate(synth.WORKLOADS[args.workload], args.cpu_sample_tokens,
                                         args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "host_cores": os.cpu_count(),
                                "sample": f"{n} oracle steps of the first {T} tokens "
                                          f"(full H, E, k) in {el:.1f} s, single thread"}
        if args.cpu_all_core_seconds > 0:
            rate_all, ncores = cpu_oracle_rate_all_cores(
                synth.WORKLOADS[args.workload], args.cpu_sample_tokens, args.cpu_all_core_seconds)
            line["cpu_baseline"]["all_cores"] = {
                "value": rate_all, "cores": ncores,
                "sample": f"one process per host core, each repeating the oracle on the first "
                          f"{min(args.cpu_sample_tokens, synth.WORKLOADS[args.workload].T)} "
                          f"tokens for {args.cpu_all_core_seconds:.0f} s"}
    else:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

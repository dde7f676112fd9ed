"""Host logic of the benchmark's N > 1 path, on CPU with world-size-2 gloo:
every rank runs an independent replica (tokens are independent), the job time
is the slowest rank's, and the rate counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.rank_env()
        assert (w, r, l) == (world, rank, rank)
        ms = bench.reduce_max_over_ranks(10.0 + rank)   # rank 1 is the slowest
        # every rank must run the same number of timed passes (barriers pair up)
        n = bench.agreed_passes(2.0 + 3.0 * rank, 0.5)
        out[rank] = (ms, bench.whole_job_rate(4096, world, 100, ms), n)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == 11.0
    assert out[0][1] == pytest.approx(4096 * 2 * 100 / 11e-3)
    assert out[0][2] == out[1][2] == 100     # 500 ms at the slower rank's 5 ms per pass


def test_single_process_defaults(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    assert bench.reduce_max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(4096, 1, 10, 2.0) == pytest.approx(4096 * 10 / 2e-3)


def test_algorithmic_bytes_per_unit():
    import bench
    from combine_layout_gb300 import synth
    w = synth.WORKLOADS["ht_prefill"]
    ab = bench.algorithmic_bytes(w)
    per_token = 2 * 7168 + 4 * 8 + 8 * (2 * 7168 + 4)
    assert ab["dispatch"] == 4096 * per_token == 528_744_448
    assert ab["combine"] == 4096 * (8 * (2 * 7168 + 8) + 2 * 7168)
    ab8 = bench.algorithmic_bytes(synth.WORKLOADS["ht_prefill_fp8"])
    assert ab8["dispatch"] == 4096 * (2 * 7168 + 32 + 8 * (7168 + 7168 // 32 + 4))


def test_algorithmic_bytes_of_the_dedup_path():
    """One copy per (token, rank) and its expansion; the two-stage combine
    writes and reads one BF16 partial per dedup row.  With one dedup row per
    pair (nothing to dedup) the dispatch side is the direct dispatch plus
    every row written once more and read back (payload, token, mask), and
    the combine side the direct combine plus the partials' round trip."""
    import bench
    from combine_layout_gb300 import synth
    w = synth.WORKLOADS["ht_prefill"]
    T, H, k = w.T, w.H, w.k
    nd = 30574
    ab = bench.algorithmic_bytes_dedup(w, nd)
    assert ab["dispatch"] == T * (2 * H + 4 * k) + 2 * nd * (2 * H + 8) + T * k * (2 * H + 4)
    assert ab["combine"] == T * k * (2 * H + 8) + 2 * nd * 2 * H + T * 2 * H
    full = bench.algorithmic_bytes_dedup(w, T * k)
    direct = bench.algorithmic_bytes(w)
    assert full["dispatch"] == direct["dispatch"] + 2 * T * k * (2 * H + 8)
    assert full["combine"] == direct["combine"] + 2 * T * k * 2 * H


def test_profile_hash_ignores_comments_only():
    """The hash tying an ncu summary to its kernel source sees code changes,
    not comment or whitespace edits."""
    import bench
    a = "int f(int x) {\n    return x + 1;  // add one\n}\n/* block\n comment */"
    b = "int f(int x)\n{\n  return x + 1;\n}\n// other words"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_agreed_passes_single_process():
    import bench
    assert bench.agreed_passes(3.4, 0.5) == 148      # ceil(500 / 3.4)
    assert bench.agreed_passes(400.0, 0.5) == 3      # at least three passes
    assert bench.agreed_passes(0.0001, 0.5, max_passes=2000) == 2000


def test_numa_of_buffer_reads_this_process():
    import numpy as np

    import bench
    a = np.ones(1 << 22, np.uint8)                   # 4 MiB, touched
    nodes = bench.numa_of_buffer(a.ctypes.data, a.nbytes)
    assert isinstance(nodes, dict)
    if "unknown" not in nodes:
        assert sum(nodes.values()) >= 1
    assert bench.gpu_numa_node(None) is None


def test_small_steps_flush_the_l2():
    """Workloads whose step touches less than twice the L2 (the LL ones) are
    timed step by step after an L2 flush; the large ones stream from HBM."""
    import bench
    from combine_layout_gb300 import synth
    W = synth.WORKLOADS
    for name in ("tiny_ll", "ll_decode"):
        assert bench.flushes_l2(W[name]), name
        assert "flushed" in bench.workload_config(W[name], 1, W[name].recv_rows())["l2"]
    for name in ("ht_prefill", "ht_prefill_fp8", "mixtral", "skewed"):
        assert not bench.flushes_l2(W[name]), name
        assert bench.step_bytes(W[name]) > 2 * bench.L2_BYTES_NOMINAL
    # the per-step bytes are the three kernels' algorithmic bytes
    ab = bench.algorithmic_bytes(W["ll_decode"])
    assert bench.step_bytes(W["ll_decode"]) == ab["route"] + ab["dispatch"] + ab["combine"]

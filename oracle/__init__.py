"""CPU oracle for MoE expert-parallel dispatch / combine (ctypes over moe_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library (``combine_layout_gb300``) never imports it and shares no code
with it.

Each wrapper follows a passage of the source pages (cited in moe_oracle.c):
  route    -- "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式" (node-limited
              routing: 4 nodes by the sum of each node's top-2 scores, then top-8)
  layout   -- same page, "高吞吐模式" (count tokens per rank and expert) and
              "低延迟模式" (fixed slots); "NCCL EP 论文解读", "算法模式"/"Tensor Layouts"
  dispatch -- same pages: HT 2D / LL 3D expert-major receive layout, FP8 e4m3 with
              one fp32 scale per 128 elements ("高吞吐模式")
  combine  -- "NCCL EP 论文解读", "核心功能函数" (un-permute with the handle's routing
              state and reduce to token order); "高吞吐模式" (BF16 weighted sum)
  node_layout -- "高吞吐模式": one copy per remote node (same-position GPU), then
              forwarding to the GPUs holding the experts; the routing statistics
  rank_layout / expand / combine_dedup -- "高吞吐模式" routing simulation, "按目标卡去重"
              (one copy per destination GPU), and BF16 weighted sums sent back
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoeoracle.so")

OK, ERR_INVALID, ERR_OVERFLOW = 0, 1, 2
MODE_LL, MODE_HT = 0, 1
W_SOFTMAX_TOPK, W_SOFTMAX_RENORM, W_SCORE_NORM = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoeoracle.so (plain gcc, IEEE arithmetic)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_double.restype = ctypes.c_double
    lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
    lib.orc_bf16_from_double.restype = ctypes.c_uint16
    lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_double.restype = ctypes.c_double
    lib.orc_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.orc_e4m3_from_float.restype = ctypes.c_uint8
    lib.orc_e4m3_from_float_array.argtypes = [P, i64, P]
    lib.orc_e4m3_from_float_array.restype = None
    lib.orc_quant_row.argtypes = [P, i32, P, P]
    lib.orc_route.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, P, P]
    lib.orc_layout.argtypes = [P, i64, i32, i32, i32, i32, i32, P, P, P, P, P]
    lib.orc_layout_aligned.argtypes = [P, i64, i32, i32, i32, i32, i32, i32, P, P, P, P, P]
    lib.orc_dequant_rows.argtypes = [P, P, i64, i32, P, i64, P]
    lib.orc_dispatch.argtypes = [P, i64, i32, i32, P, i64, i32, P, P, P]
    lib.orc_node_layout.argtypes = [P, i64, i32, i32, i32, i32, i32, P, P, P, P, P]
    lib.orc_combine.argtypes = [P, i64, i32, P, P, i64, i32, P, i64, P]
    lib.orc_rank_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P]
    lib.orc_expand.argtypes = [P, P, i64, i64, i32, P, P, P, i32, i32, P, P, i64, i32, i64, P, P, P]
    lib.orc_combine_dedup.argtypes = [P, i64, i32, P, P, P, i64, i32, i32, i32, P, i64, P, i64, P, P]
    for f in ("orc_quant_row", "orc_route", "orc_layout", "orc_dispatch", "orc_combine",
              "orc_node_layout", "orc_layout_aligned", "orc_dequant_rows", "orc_rank_layout",
              "orc_expand", "orc_combine_dedup"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars
def bf16_to_double(b: int) -> float:
    return _load().orc_bf16_to_double(int(b))


def bf16_from_double(v: float) -> int:
    return int(_load().orc_bf16_from_double(float(v)))


def e4m3_to_double(code: int) -> float:
    return _load().orc_e4m3_to_double(int(code))


def e4m3_from_float(v: float) -> int:
    return int(_load().orc_e4m3_from_float(float(v)))


def e4m3_from_float_array(v) -> np.ndarray:
    v = _c(v, np.float32).reshape(-1)
    out = np.empty(v.shape, np.uint8)
    _load().orc_e4m3_from_float_array(_p(v), v.size, _p(out))
    return out


def quant_row(x_bf16_bits) -> tuple[np.ndarray, np.ndarray]:
    x = _c(x_bf16_bits, np.uint16).reshape(-1)
    H = x.size
    q = np.empty(H, np.uint8)
    s = np.empty(max(H // 128, 1), np.float32)
    st = _load().orc_quant_row(_p(x), H, _p(q), _p(s))
    if st != OK:
        raise ValueError(f"orc_quant_row status {st}")
    return q, s[: H // 128]


# ---------------------------------------------------------------- path
def route(scores, k: int, num_groups: int = 1, topk_groups: int = 1,
          group_topk: int = 0, weight_mode: int = W_SCORE_NORM):
    """Node-limited top-k routing. Returns (topk_idx int32 [T,k], topk_w float64 [T,k])."""
    s = _c(scores, np.float32)
    T, E = s.shape
    if group_topk == 0:
        group_topk = -(-k // topk_groups)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    st = _load().orc_route(_p(s), T, E, num_groups, topk_groups, group_topk, k,
                           weight_mode, _p(idx), _p(w))
    if st != OK:
        raise ValueError(f"orc_route status {st}")
    return idx, w


def layout(topk_idx, experts: int, ranks: int, mode: int, slots: int = 0, align: int = 1):
    """Counts, offsets and the row map (HT expert blocks padded to `align` rows).
    Returns (dict, status)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    cnt = np.empty(experts, np.int32)
    off = np.empty(experts + 1, np.int32)
    rcnt = np.empty(ranks, np.int32)
    roff = np.empty(ranks + 1, np.int32)
    row = np.empty((T, k), np.int32)
    if align == 1:
        st = _load().orc_layout(_p(idx), T, k, experts, ranks, mode, slots,
                                _p(cnt), _p(off), _p(rcnt), _p(roff), _p(row))
    else:
        st = _load().orc_layout_aligned(_p(idx), T, k, experts, ranks, mode, slots, align,
                                        _p(cnt), _p(off), _p(rcnt), _p(roff), _p(row))
    return dict(cnt=cnt, off=off, rcnt=rcnt, roff=roff, row=row), st


def dequant_rows(q, scale, rows) -> np.ndarray:
    """bf16 bits of float(q) * scale (fp32 product) for the listed rows, zeros elsewhere."""
    q = _c(q, np.uint8)
    nrows, H = q.shape
    sc = _c(scale, np.float32)
    r = _c(rows, np.int64).reshape(-1)
    y = np.zeros((nrows, H), np.uint16)
    st = _load().orc_dequant_rows(_p(q), _p(sc), nrows, H, _p(r), r.size, _p(y))
    if st != OK:
        raise ValueError(f"orc_dequant_rows status {st}")
    return y


def node_layout(topk_idx, experts: int, ranks: int, nodes: int, src_node: int = 0):
    """Node-level (two-hop) layout and the routing statistics.
    Returns dict(cnt, off, src, mask, stats[4])."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    cnt = np.empty(nodes, np.int32)
    off = np.empty(nodes + 1, np.int32)
    rows = T * min(k, nodes)
    src = np.full(max(rows, 1), -1, np.int32)
    mask = np.zeros(max(rows, 1), np.uint32)
    stats = np.zeros(4, np.int64)
    st = _load().orc_node_layout(_p(idx), T, k, experts, ranks, nodes, src_node, _p(cnt), _p(off),
                                 _p(src), _p(mask), _p(stats))
    if st != OK:
        raise ValueError(f"orc_node_layout status {st}")
    n = int(off[-1])
    return dict(cnt=cnt, off=off, src=src[:n], mask=mask[:n], stats=stats)


def dispatch(x_bf16_bits, row, nrows: int, fp8: bool, recv_x=None, recv_scale=None,
             recv_src=None):
    """Pack tokens into the receive layout. Returns (recv_x, recv_scale, recv_src)."""
    x = _c(x_bf16_bits, np.uint16)
    T, H = x.shape
    row = _c(row, np.int32)
    k = row.shape[1]
    if recv_x is None:
        recv_x = np.zeros((nrows, H), np.uint8 if fp8 else np.uint16)
    if recv_scale is None:
        recv_scale = np.zeros((nrows, max(H // 128, 1)), np.float32)
    if recv_src is None:
        recv_src = np.full(nrows, -1, np.int32)
    st = _load().orc_dispatch(_p(x), T, H, k, _p(row), nrows, int(bool(fp8)),
                              _p(recv_x), _p(recv_scale), _p(recv_src))
    if st != OK:
        raise ValueError(f"orc_dispatch status {st}")
    return recv_x, recv_scale, recv_src


def combine(y_bf16_bits, row, w, tokens=None) -> np.ndarray:
    """Weighted un-permute back to token order. Returns bf16 bits [T or len(tokens), H]."""
    y = _c(y_bf16_bits, np.uint16)
    nrows, H = y.shape
    row = _c(row, np.int32)
    T, k = row.shape
    w = _c(w, np.float32)
    if tokens is None:
        tk, ntok, n = None, 0, T
    else:
        tk = _c(tokens, np.int64).reshape(-1)
        ntok = n = tk.size
    out = np.empty((n, H), np.uint16)
    st = _load().orc_combine(_p(y), nrows, H, _p(row), _p(w), T, k,
                             None if tk is None else _p(tk), ntok, _p(out))
    if st != OK:
        raise ValueError(f"orc_combine status {st}")
    return out


def rank_layout(topk_idx, experts: int, ranks: int):
    """Per-rank dedup layout.  Returns (dict(cnt, off, drow, src, mask), status)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    cnt = np.empty(ranks, np.int32)
    off = np.empty(ranks + 1, np.int32)
    drow = np.empty((T, k), np.int32)
    cap = max(T * min(k, ranks), 1)
    src = np.full(cap, -1, np.int32)
    mask = np.zeros(cap, np.uint32)
    st = _load().orc_rank_layout(_p(idx), T, k, experts, ranks, _p(cnt), _p(off), _p(drow),
                                 _p(src), _p(mask))
    if st == ERR_INVALID and (experts % ranks or experts // ranks > 32):
        raise ValueError("orc_rank_layout: bad shape")
    n = int(off[-1])
    return dict(cnt=cnt, off=off, drow=drow, src=src[:n], mask=mask[:n]), st


def expand(dx, dscale, dsrc, dmask, rank_off, experts: int, topk_idx, row, nrows: int):
    """Receiver-side expansion of dedup rows (bf16 [nd][H] or e4m3 [nd][H] with
    dscale [nd][H/128]) into the expert-major rows.  Returns (recv_x, recv_scale, recv_src)."""
    dx = np.ascontiguousarray(dx)
    nd = dx.shape[0]
    row_bytes = dx.shape[1] * dx.itemsize
    fp8 = dscale is not None
    nscale = dscale.shape[1] if fp8 else 0
    recv_x = np.zeros((nrows,) + dx.shape[1:], dx.dtype)
    recv_scale = np.zeros((nrows, max(nscale, 1)), np.float32)
    recv_src = np.full(nrows, -1, np.int32)
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    R = len(rank_off) - 1
    st = _load().orc_expand(_p(dx), _p(_c(dscale, np.float32)) if fp8 else None, nd, row_bytes,
                            nscale, _p(_c(dsrc, np.int32)), _p(_c(dmask, np.uint32)),
                            _p(_c(rank_off, np.int32)), R, experts, _p(idx), _p(_c(row, np.int32)),
                            T, k, nrows, _p(recv_x), _p(recv_scale), _p(recv_src))
    if st != OK:
        raise ValueError(f"orc_expand status {st}")
    return recv_x, (recv_scale if fp8 else None), recv_src


def combine_dedup(y_bf16_bits, topk_idx, row, w, experts: int, ranks: int, drow, nd: int,
                  tokens=None, want_partial: bool = False):
    """Two-stage combine over dedup rows.  Returns out [T or len(tokens), H]
    (and the partial rows [nd][H] when want_partial)."""
    y = _c(y_bf16_bits, np.uint16)
    nrows, H = y.shape
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    if tokens is None:
        tk, ntok, n = None, 0, T
    else:
        tk = _c(tokens, np.int64).reshape(-1)
        ntok = n = tk.size
    out = np.empty((n, H), np.uint16)
    partial = np.zeros((max(nd, 1), H), np.uint16) if want_partial else None
    st = _load().orc_combine_dedup(_p(y), nrows, H, _p(idx), _p(_c(row, np.int32)),
                                   _p(_c(w, np.float32)), T, k, experts, ranks,
                                   _p(_c(drow, np.int32)), nd, None if tk is None else _p(tk),
                                   ntok, None if partial is None else _p(partial), _p(out))
    if st != OK:
        raise ValueError(f"orc_combine_dedup status {st}")
    return (out, partial[:nd]) if want_partial else out

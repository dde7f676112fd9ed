"""Thin Python binding of libmoeep (ctypes): argument marshalling only.

Every function has the name of the C entry point it calls (include/moe_ep.h)
and takes torch CUDA tensors (or None for NULL).  All work runs in the CUDA
kernels of libmoeep; nothing here computes.  Importing this module loads the
library and fails loudly if it has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeep.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "moe_ep.h")

MOE_EP_LL, MOE_EP_HT = 0, 1
(MOE_EP_OK, MOE_EP_ERR_INVALID, MOE_EP_ERR_OVERFLOW, MOE_EP_ERR_CUDA, MOE_EP_ERR_DEVICE,
 MOE_EP_ERR_TIMEOUT) = range(6)
MOE_EP_W_SOFTMAX_TOPK, MOE_EP_W_SOFTMAX_RENORM, MOE_EP_W_SCORE_NORM = 0, 1, 2
MOE_EP_DEVERR_EXPERT_RANGE, MOE_EP_DEVERR_DUPLICATE, MOE_EP_DEVERR_TIMEOUT = 1, 2, 4


class MoeEpError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: status {status} ({status_string(status)})")


class RouteOpts(ctypes.Structure):
    _fields_ = [("topk", ctypes.c_int), ("num_groups", ctypes.c_int),
                ("topk_groups", ctypes.c_int), ("group_topk", ctypes.c_int),
                ("weight_mode", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoeep is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    PP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "moe_ep_create_group": [PP, I, I, I, I, I],
        "moe_ep_destroy_group": [P],
        "moe_ep_create_handle": [P, I, PP],
        "moe_ep_destroy_handle": [P],
        "moe_ep_route": [P, P, I, ctypes.POINTER(RouteOpts), P, P, P],
        "moe_ep_get_num_recv_tokens": [P, ctypes.POINTER(ctypes.c_int64), P, P, P],
        "moe_ep_dispatch": [P, P, I, P, P, P, P, I64, P],
        "moe_ep_combine": [P, P, P, P, I64, P],
        "moe_ep_copy_layout": [P, P, P, P, P, P, P],
        "moe_ep_get_device_errors": [P, ctypes.POINTER(ctypes.c_uint32)],
        "moe_ep_clear_device_errors": [P],
        "moe_ep_node_layout": [P, I, I, P, P, P, P, I64, P, P],
        "moe_ep_set_row_align": [P, I],
        "moe_ep_set_x_before_route": [P, I],
        "moe_ep_dispatch_send": [P, P, I, P, P, P, P, I64, P],
        "moe_ep_combine_send": [P, P, P, P, I64, P],
        "moe_ep_complete": [P, P],
        "moe_ep_signal_add": [P, P, ctypes.c_uint32, P],
        "moe_ep_wait_signal": [P, P, ctypes.c_uint32, I64, P],
        "moe_ep_dequant": [P, P, P, P, I64, P],
        "moe_ep_route_layout_static": [P, I, I, I, I, I, ctypes.POINTER(RouteOpts), P, P, P, P, P,
                                       P, P, P],
        "moe_ep_dispatch_dedup": [P, P, I, P, P, P, P, P, P, I64, P],
        "moe_ep_expand": [P, P, P, P, P, I, P, P, P, I64, P],
        "moe_ep_combine_dedup": [P, P, P, P, P, P, I64, I64, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.moe_ep_status_string.argtypes = [I]
    lib.moe_ep_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


def declared_symbols() -> list[str]:
    """Entry points declared in include/moe_ep.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*MOE_EP_API\s+(?:int|const char\*)\s+(moe_ep_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return _lib.moe_ep_status_string(int(status)).decode()


def _check(name: str, st: int):
    if st != MOE_EP_OK:
        raise MoeEpError(name, st)


def _ptr(t) -> ctypes.c_void_p | None:
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_contiguous():
        raise ValueError("libmoeep takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ------------------------------------------------------------------ entry points
def moe_ep_create_group(mode: int, experts: int, ranks: int, max_tokens: int, hidden: int) -> int:
    out = ctypes.c_void_p()
    _check("moe_ep_create_group",
           _lib.moe_ep_create_group(ctypes.byref(out), mode, experts, ranks, max_tokens, hidden))
    return out.value


def moe_ep_destroy_group(group: int) -> None:
    _check("moe_ep_destroy_group", _lib.moe_ep_destroy_group(ctypes.c_void_p(group)))


def moe_ep_create_handle(group: int, max_topk: int) -> int:
    out = ctypes.c_void_p()
    _check("moe_ep_create_handle",
           _lib.moe_ep_create_handle(ctypes.c_void_p(group), max_topk, ctypes.byref(out)))
    return out.value


def moe_ep_destroy_handle(handle: int) -> None:
    _check("moe_ep_destroy_handle", _lib.moe_ep_destroy_handle(ctypes.c_void_p(handle)))


def moe_ep_route(handle: int, scores, num_tokens: int, topk: int, topk_idx, topk_w=None,
                 num_groups: int = 1, topk_groups: int = 1, group_topk: int = 0,
                 weight_mode: int = MOE_EP_W_SCORE_NORM, stream=None) -> None:
    opts = RouteOpts(topk, num_groups, topk_groups, group_topk, weight_mode)
    _check("moe_ep_route", _lib.moe_ep_route(ctypes.c_void_p(handle), _ptr(scores), num_tokens,
                                             ctypes.byref(opts), _ptr(topk_idx), _ptr(topk_w),
                                             _stream(stream)))


def moe_ep_get_num_recv_tokens(handle: int, ranks: int | None = None, experts: int | None = None,
                               stream=None):
    """Returns (total, per_rank list or None, per_expert list or None)."""
    total = ctypes.c_int64()
    pr = (ctypes.c_int32 * ranks)() if ranks else None
    pe = (ctypes.c_int32 * experts)() if experts else None
    _check("moe_ep_get_num_recv_tokens",
           _lib.moe_ep_get_num_recv_tokens(ctypes.c_void_p(handle), ctypes.byref(total),
                                           ctypes.cast(pr, ctypes.c_void_p) if pr else None,
                                           ctypes.cast(pe, ctypes.c_void_p) if pe else None,
                                           _stream(stream)))
    return total.value, (list(pr) if pr else None), (list(pe) if pe else None)


def moe_ep_dispatch(handle: int, x, fp8: bool, recv_x, recv_scale=None, recv_src=None,
                    recv_cnt=None, recv_rows: int | None = None, stream=None) -> None:
    if recv_rows is None:
        recv_rows = recv_x.shape[0]
    _check("moe_ep_dispatch",
           _lib.moe_ep_dispatch(ctypes.c_void_p(handle), _ptr(x), int(bool(fp8)), _ptr(recv_x),
                                _ptr(recv_scale), _ptr(recv_src), _ptr(recv_cnt), recv_rows,
                                _stream(stream)))


def moe_ep_combine(handle: int, y, topk_w, out, recv_rows: int | None = None, stream=None) -> None:
    if recv_rows is None:
        recv_rows = y.shape[0]
    _check("moe_ep_combine",
           _lib.moe_ep_combine(ctypes.c_void_p(handle), _ptr(y), _ptr(topk_w), _ptr(out),
                               recv_rows, _stream(stream)))


def moe_ep_copy_layout(handle: int, cnt=None, off=None, rcnt=None, roff=None, row=None,
                       stream=None) -> None:
    _check("moe_ep_copy_layout",
           _lib.moe_ep_copy_layout(ctypes.c_void_p(handle), _ptr(cnt), _ptr(off), _ptr(rcnt),
                                   _ptr(roff), _ptr(row), _stream(stream)))


def moe_ep_dispatch_send(handle: int, x, fp8: bool, recv_x, recv_scale=None, recv_src=None,
                         recv_cnt=None, recv_rows: int | None = None, stream=None) -> None:
    if recv_rows is None:
        recv_rows = recv_x.shape[0]
    _check("moe_ep_dispatch_send",
           _lib.moe_ep_dispatch_send(ctypes.c_void_p(handle), _ptr(x), int(bool(fp8)),
                                     _ptr(recv_x), _ptr(recv_scale), _ptr(recv_src),
                                     _ptr(recv_cnt), recv_rows, _stream(stream)))


def moe_ep_combine_send(handle: int, y, topk_w, out, recv_rows: int | None = None,
                        stream=None) -> None:
    if recv_rows is None:
        recv_rows = y.shape[0]
    _check("moe_ep_combine_send",
           _lib.moe_ep_combine_send(ctypes.c_void_p(handle), _ptr(y), _ptr(topk_w), _ptr(out),
                                    recv_rows, _stream(stream)))


def moe_ep_complete(handle: int, stream=None) -> None:
    _check("moe_ep_complete", _lib.moe_ep_complete(ctypes.c_void_p(handle), _stream(stream)))


def moe_ep_signal_add(group: int, signal, value: int, stream=None) -> None:
    """signal: a one-element uint32 / int32 device tensor."""
    _check("moe_ep_signal_add", _lib.moe_ep_signal_add(ctypes.c_void_p(group), _ptr(signal),
                                                       value, _stream(stream)))


def moe_ep_wait_signal(group: int, signal, expected: int, timeout_ns: int, stream=None) -> None:
    _check("moe_ep_wait_signal", _lib.moe_ep_wait_signal(ctypes.c_void_p(group), _ptr(signal),
                                                         expected, timeout_ns, _stream(stream)))


def moe_ep_set_row_align(handle: int, align: int) -> None:
    _check("moe_ep_set_row_align", _lib.moe_ep_set_row_align(ctypes.c_void_p(handle), align))


def moe_ep_set_x_before_route(handle: int, on: bool) -> None:
    _check("moe_ep_set_x_before_route",
           _lib.moe_ep_set_x_before_route(ctypes.c_void_p(handle), 1 if on else 0))


def moe_ep_dequant(handle: int, recv_q, recv_scale, y, recv_rows: int | None = None,
                   stream=None) -> None:
    if recv_rows is None:
        recv_rows = recv_q.shape[0]
    _check("moe_ep_dequant",
           _lib.moe_ep_dequant(ctypes.c_void_p(handle), _ptr(recv_q), _ptr(recv_scale), _ptr(y),
                               recv_rows, _stream(stream)))


def moe_ep_node_layout(handle: int, num_nodes: int, src_node: int, node_cnt, node_off,
                       node_src, node_mask, stats=None, node_rows: int | None = None,
                       stream=None) -> None:
    if node_rows is None:
        node_rows = node_src.shape[0] if node_src is not None else 0
    _check("moe_ep_node_layout",
           _lib.moe_ep_node_layout(ctypes.c_void_p(handle), num_nodes, src_node, _ptr(node_cnt),
                                   _ptr(node_off), _ptr(node_src), _ptr(node_mask), node_rows,
                                   _ptr(stats), _stream(stream)))


def moe_ep_dispatch_dedup(handle: int, x, fp8: bool, drecv_x, drecv_scale=None, drecv_src=None,
                          drecv_mask=None, rank_cnt=None, rank_off=None,
                          drecv_rows: int | None = None, stream=None) -> None:
    if drecv_rows is None:
        drecv_rows = drecv_x.shape[0]
    _check("moe_ep_dispatch_dedup",
           _lib.moe_ep_dispatch_dedup(ctypes.c_void_p(handle), _ptr(x), int(bool(fp8)),
                                      _ptr(drecv_x), _ptr(drecv_scale), _ptr(drecv_src),
                                      _ptr(drecv_mask), _ptr(rank_cnt), _ptr(rank_off),
                                      drecv_rows, _stream(stream)))


def moe_ep_expand(handle: int, drecv_x, drecv_scale, drecv_src, drecv_mask, fp8: bool, recv_x,
                  recv_scale=None, recv_src=None, recv_rows: int | None = None,
                  stream=None) -> None:
    if recv_rows is None:
        recv_rows = recv_x.shape[0]
    _check("moe_ep_expand",
           _lib.moe_ep_expand(ctypes.c_void_p(handle), _ptr(drecv_x), _ptr(drecv_scale),
                              _ptr(drecv_src), _ptr(drecv_mask), int(bool(fp8)), _ptr(recv_x),
                              _ptr(recv_scale), _ptr(recv_src), recv_rows, _stream(stream)))


def moe_ep_combine_dedup(handle: int, y, topk_w, drecv_src, partial, out,
                         recv_rows: int | None = None, drecv_rows: int | None = None,
                         stream=None) -> None:
    if recv_rows is None:
        recv_rows = y.shape[0]
    if drecv_rows is None:
        drecv_rows = partial.shape[0]
    _check("moe_ep_combine_dedup",
           _lib.moe_ep_combine_dedup(ctypes.c_void_p(handle), _ptr(y), _ptr(topk_w),
                                     _ptr(drecv_src), _ptr(partial), _ptr(out), recv_rows,
                                     drecv_rows, _stream(stream)))


def moe_ep_get_device_errors(group: int) -> int:
    bits = ctypes.c_uint32()
    _check("moe_ep_get_device_errors",
           _lib.moe_ep_get_device_errors(ctypes.c_void_p(group), ctypes.byref(bits)))
    return bits.value


def moe_ep_clear_device_errors(group: int) -> None:
    _check("moe_ep_clear_device_errors", _lib.moe_ep_clear_device_errors(ctypes.c_void_p(group)))


def moe_ep_route_layout_static(scores, num_tokens: int, experts: int, ranks: int, mode: int,
                               slots: int, topk: int, topk_idx, topk_w, row, cnt, off, rcnt, roff,
                               num_groups: int = 1, topk_groups: int = 1, group_topk: int = 0,
                               weight_mode: int = MOE_EP_W_SCORE_NORM, stream=None) -> None:
    """Routing + layout into caller buffers with no device allocation (the
    library's static scratch array); see include/moe_ep.h."""
    opts = RouteOpts(topk, num_groups, topk_groups, group_topk, weight_mode)
    _check("moe_ep_route_layout_static",
           _lib.moe_ep_route_layout_static(_ptr(scores), num_tokens, experts, ranks, mode, slots,
                                           ctypes.byref(opts), _ptr(topk_idx), _ptr(topk_w),
                                           _ptr(row), _ptr(cnt), _ptr(off), _ptr(rcnt), _ptr(roff),
                                           _stream(stream)))

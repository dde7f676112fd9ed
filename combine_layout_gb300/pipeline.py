"""One group + one handle with their receive buffers (torch device memory).

Allocation and argument marshalling only: every step runs in libmoeep's
kernels through the C ABI (``moe_ep``).  The order of calls is the one on
"NCCL EP 论文解读", item "使用方式": create the group once, then per forward
route -> (HT: receive-count query) -> dispatch -> experts -> combine.
"""
from __future__ import annotations

import torch

from . import moe_ep as ep


class EpPipeline:
    def __init__(self, mode: int, experts: int, ranks: int, max_tokens: int, hidden: int,
                 topk: int, fp8: bool = False, device: str | int = "cuda", align: int = 1,
                 x_before_route: bool = False):
        self.mode, self.E, self.R, self.S, self.H, self.k = mode, experts, ranks, max_tokens, hidden, topk
        self.fp8 = fp8
        self.device = torch.device(device)
        self.group = ep.moe_ep_create_group(mode, experts, ranks, max_tokens, hidden)
        self.handle = ep.moe_ep_create_handle(self.group, topk)
        if align != 1:
            ep.moe_ep_set_row_align(self.handle, align)
        if x_before_route:
            ep.moe_ep_set_x_before_route(self.handle, True)
        self.align = align
        self.rows = (experts * max_tokens if mode == ep.MOE_EP_LL
                     else max_tokens * topk + experts * (align - 1))
        dev = self.device
        self.topk_idx = torch.empty((max_tokens, topk), dtype=torch.int32, device=dev)
        self.topk_w = torch.empty((max_tokens, topk), dtype=torch.float32, device=dev)
        self.recv_x = torch.empty((self.rows, hidden), dtype=torch.uint8 if fp8 else torch.bfloat16,
                                  device=dev)
        self.recv_scale = (torch.empty((self.rows, hidden // 128), dtype=torch.float32, device=dev)
                           if fp8 else None)
        self.recv_src = torch.empty(self.rows, dtype=torch.int32, device=dev)
        self.recv_cnt = torch.empty(experts, dtype=torch.int32, device=dev)
        self.out = torch.empty((max_tokens, hidden), dtype=torch.bfloat16, device=dev)
        self.T = 0

    # ---------------------------------------------------------------- steps
    def route(self, scores, num_tokens: int, num_groups: int = 1, topk_groups: int = 1,
              group_topk: int = 0, weight_mode: int = ep.MOE_EP_W_SCORE_NORM, stream=None):
        self.T = num_tokens
        ep.moe_ep_route(self.handle, scores, num_tokens, self.k, self.topk_idx, self.topk_w,
                        num_groups, topk_groups, group_topk, weight_mode, stream)

    def route_given(self, topk_idx, stream=None):
        """Lay out caller-made routing (topk_idx [T][k] int32 on the device)."""
        T = topk_idx.shape[0]
        self.topk_idx[:T].copy_(topk_idx)
        self.T = T
        ep.moe_ep_route(self.handle, None, T, self.k, self.topk_idx, None, stream=stream)

    def num_recv_tokens(self, stream=None):
        return ep.moe_ep_get_num_recv_tokens(self.handle, self.R, self.E, stream)

    def dispatch(self, x, stream=None):
        ep.moe_ep_dispatch(self.handle, x, self.fp8, self.recv_x, self.recv_scale, self.recv_src,
                           self.recv_cnt, self.rows, stream)

    def combine(self, y, topk_w=None, out=None, stream=None):
        if topk_w is None:
            topk_w = self.topk_w
        if out is None:
            out = self.out
        ep.moe_ep_combine(self.handle, y, topk_w, out, y.shape[0], stream)
        return out[: self.T]

    def dequant(self, y=None, stream=None):
        """bf16 expert-major rows from the FP8 receive buffers (defined rows only)."""
        if y is None:
            y = torch.zeros((self.rows, self.H), dtype=torch.bfloat16, device=self.device)
        ep.moe_ep_dequant(self.handle, self.recv_x, self.recv_scale, y, self.rows, stream)
        return y

    # ------------------------------------------------- per-rank dedup (HT)
    def _dedup_buffers(self):
        if getattr(self, "drows", None) is None:
            dev = self.device
            self.drows = self.S * min(self.k, self.R)
            self.drecv_x = torch.empty((self.drows, self.H),
                                       dtype=torch.uint8 if self.fp8 else torch.bfloat16, device=dev)
            self.drecv_scale = (torch.empty((self.drows, self.H // 128), dtype=torch.float32,
                                            device=dev) if self.fp8 else None)
            self.drecv_src = torch.empty(self.drows, dtype=torch.int32, device=dev)
            self.drecv_mask = torch.empty(self.drows, dtype=torch.int32, device=dev)
            self.rank_cnt = torch.empty(self.R, dtype=torch.int32, device=dev)
            self.rank_off = torch.empty(self.R + 1, dtype=torch.int32, device=dev)
            self.partial = torch.empty((self.drows, self.H), dtype=torch.bfloat16, device=dev)

    def dispatch_dedup(self, x, stream=None):
        """One copy per (token, destination rank) into drecv_*; rank_cnt / rank_off."""
        self._dedup_buffers()
        ep.moe_ep_dispatch_dedup(self.handle, x, self.fp8, self.drecv_x, self.drecv_scale,
                                 self.drecv_src, self.drecv_mask, self.rank_cnt, self.rank_off,
                                 self.drows, stream)

    def expand(self, stream=None):
        """Receiver side: the dedup rows into recv_x / recv_scale / recv_src."""
        ep.moe_ep_expand(self.handle, self.drecv_x, self.drecv_scale, self.drecv_src,
                         self.drecv_mask, self.fp8, self.recv_x, self.recv_scale, self.recv_src,
                         self.rows, stream)

    def combine_dedup(self, y, topk_w=None, out=None, stream=None):
        if topk_w is None:
            topk_w = self.topk_w
        if out is None:
            out = self.out
        ep.moe_ep_combine_dedup(self.handle, y, topk_w, self.drecv_src, self.partial, out,
                                y.shape[0], self.drows, stream)
        return out[: self.T]

    def layout(self, stream=None) -> dict:
        dev = self.device
        L = dict(cnt=torch.empty(self.E, dtype=torch.int32, device=dev),
                 off=torch.empty(self.E + 1, dtype=torch.int32, device=dev),
                 rcnt=torch.empty(self.R, dtype=torch.int32, device=dev),
                 roff=torch.empty(self.R + 1, dtype=torch.int32, device=dev),
                 row=torch.empty((max(self.T, 1), self.k), dtype=torch.int32, device=dev))
        ep.moe_ep_copy_layout(self.handle, L["cnt"], L["off"], L["rcnt"], L["roff"], L["row"], stream)
        L["row"] = L["row"][: self.T]
        return L

    def device_errors(self) -> int:
        return ep.moe_ep_get_device_errors(self.group)

    def clear_device_errors(self):
        ep.moe_ep_clear_device_errors(self.group)

    def close(self):
        if self.handle:
            ep.moe_ep_destroy_handle(self.handle)
            self.handle = None
        if self.group:
            ep.moe_ep_destroy_group(self.group)
            self.group = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BoundStep:
    """One forward on fixed buffers with every C-ABI argument marshalled once.

    For callers that repeat the same shapes (a serving loop, the benchmark):
    each call is then a bare ctypes call into libmoeep, so the host adds as
    little as possible between the kernels of a step.
    """

    def __init__(self, p: EpPipeline, scores, x, y, num_tokens: int, num_groups: int = 1,
                 topk_groups: int = 1, group_topk: int = 0,
                 weight_mode: int = ep.MOE_EP_W_SCORE_NORM, stream=None, out=None):
        import ctypes

        V = ctypes.c_void_p
        if stream is None:
            stream = torch.cuda.current_stream(p.device)
        lib = ep._lib
        h = V(p.handle)
        s = V(stream.cuda_stream)
        ptr = (lambda t: None if t is None else V(t.data_ptr()))
        for t in (scores, x, y):
            if not t.is_contiguous():
                raise ValueError("libmoeep takes contiguous tensors")
        self.p = p
        self._opts = ep.RouteOpts(p.k, num_groups, topk_groups, group_topk, weight_mode)
        self._total = ctypes.c_int64()
        self._per_rank = (ctypes.c_int32 * p.R)()
        self._route = (lib.moe_ep_route, (h, ptr(scores), num_tokens, ctypes.byref(self._opts),
                                          ptr(p.topk_idx), ptr(p.topk_w), s))
        self._dispatch = (lib.moe_ep_dispatch, (h, ptr(x), int(p.fp8), ptr(p.recv_x),
                                                ptr(p.recv_scale), ptr(p.recv_src),
                                                ptr(p.recv_cnt), p.rows, s))
        out = p.out if out is None else out
        if not out.is_contiguous() or out.shape[0] < num_tokens:
            raise ValueError("out must be contiguous with room for the tokens")
        self.out = out
        self._combine = (lib.moe_ep_combine, (h, ptr(y), ptr(p.topk_w), ptr(out), y.shape[0], s))
        self._query = (lib.moe_ep_get_num_recv_tokens,
                       (h, ctypes.byref(self._total),
                        ctypes.cast(self._per_rank, ctypes.c_void_p), None, s))
        p.T = num_tokens

    @staticmethod
    def _call(fa, name):
        st = fa[0](*fa[1])
        if st != ep.MOE_EP_OK:
            raise ep.MoeEpError(name, st)

    def route(self):
        self._call(self._route, "moe_ep_route")

    def dispatch(self):
        self._call(self._dispatch, "moe_ep_dispatch")

    def combine(self):
        self._call(self._combine, "moe_ep_combine")

    def num_recv_tokens(self) -> int:
        self._call(self._query, "moe_ep_get_num_recv_tokens")
        return self._total.value

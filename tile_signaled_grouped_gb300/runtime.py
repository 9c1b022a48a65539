"""Owner of the device memory one plan needs, on top of the C ABI.

PyTorch provides the allocations and the streams; every computation is a
launch of the library's kernels through capi. Each logical rank gets its own
allocations (rank workspace, receive buffer, output).
"""
from __future__ import annotations

import torch

from . import capi


def _stream_handle(s) -> int:
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


class ExpertCombine:
    """One MoE layer split over W logical ranks on the current CUDA device."""

    def __init__(self, W, L, topk, T, d_model, d_ff, tb_M, mgb=1, consumer_ctas=8,
                 timeout_ns=0, producer_pairs=1, device=None):
        self.device = torch.device(device or "cuda")
        self.cfg = capi.moe_cfg(W, L, topk, T, d_model, d_ff, tb_M, mgb, consumer_ctas,
                                timeout_ns, producer_pairs)
        self.W, self.L, self.k, self.T, self.D, self.F = W, L, topk, T, d_model, d_ff
        plan_bytes, rank_bytes, recv_rows = capi.moe_workspace_size(self.cfg)
        self.plan_bytes, self.rank_bytes, self.recv_rows = plan_bytes, rank_bytes, recv_rows
        dev = self.device
        self.plan_ws = torch.zeros(plan_bytes, dtype=torch.uint8, device=dev)
        # rank workspaces: 1024-byte aligned views of separate allocations
        self._rank_raw, self.rank_ws = [], []
        for _ in range(W):
            raw = torch.empty(rank_bytes + 1024, dtype=torch.uint8, device=dev)
            off = (-raw.data_ptr()) % 1024
            self._rank_raw.append(raw)
            self.rank_ws.append(raw[off:off + rank_bytes])
        self.recv = [torch.zeros(max(recv_rows, 1), d_model, dtype=torch.bfloat16, device=dev)
                     for _ in range(W)]
        self.out = [torch.empty(T, d_model, dtype=torch.bfloat16, device=dev) for _ in range(W)]
        self.ids = torch.empty(W, T, topk, dtype=torch.int32, device=dev)
        self.w = torch.empty(W, T, topk, dtype=torch.float32, device=dev)
        with torch.cuda.device(dev):
            self.plan = capi.moe_plan_create(self.cfg, self.plan_ws.data_ptr(), plan_bytes,
                                             [t.data_ptr() for t in self.rank_ws], rank_bytes)

    def close(self):
        if getattr(self, "plan", None):
            capi.moe_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ path
    def route(self, logits, forced_ids=None, stream=None):
        capi.moe_route(self.plan, logits.data_ptr(),
                       None if forced_ids is None else forced_ids.data_ptr(),
                       self.ids.data_ptr(), self.w.data_ptr(), _stream_handle(stream))
        return self.ids, self.w

    def plan_build(self, x, ids=None, stream=None):
        ids = self.ids if ids is None else ids
        capi.moe_plan_build(self.plan, ids.data_ptr(), [t.data_ptr() for t in x],
                            _stream_handle(stream))

    def expert_combine(self, w_gate, w_up, w_down, producer=None, consumer=None):
        sp = _stream_handle(producer)
        sc = sp if consumer is None else _stream_handle(consumer)
        capi.moe_expert_combine(self.plan, [t.data_ptr() for t in w_gate],
                                [t.data_ptr() for t in w_up], [t.data_ptr() for t in w_down],
                                [t.data_ptr() for t in self.recv], sp, sc)

    def scale(self, w=None, stream=None):
        w = self.w if w is None else w
        capi.moe_scale(self.plan, w.data_ptr(), [t.data_ptr() for t in self.recv],
                       [t.data_ptr() for t in self.out], _stream_handle(stream))
        return self.out

    def forward(self, x, w_gate, w_up, w_down, logits, forced_ids=None, producer=None,
                consumer=None):
        """route -> plan -> overlapped FFN and combine -> scale; all on the GPU."""
        self.route(logits, forced_ids, producer)
        self.plan_build(x, stream=producer)
        self.expert_combine(w_gate, w_up, w_down, producer, consumer)
        return self.scale(stream=producer)

    # ------------------------------------------------------------- inspection
    def status(self, stream=None):
        return capi.moe_status(self.plan, _stream_handle(stream))

    def clear_status(self, stream=None):
        capi.moe_status_clear(self.plan, _stream_handle(stream))

    def field(self, field: int) -> torch.Tensor:
        """View of a plan array (int32) inside the plan workspace."""
        off, cnt = capi.moe_field(self.cfg, field)
        return self.plan_ws[off:off + 4 * cnt].view(torch.int32)

    def rank_field(self, field: int, rank: int) -> torch.Tensor:
        off, cnt = capi.moe_field(self.cfg, field)
        cols = self.F if field == capi.MOE_RANK_H else self.D
        return self.rank_ws[rank][off:off + 2 * cnt].view(torch.bfloat16).view(-1, cols)

    def launch_info(self):
        """(producer_ctas, consumer_ctas, num_sms, pair_clusters) of the overlapped schedule."""
        return capi.moe_launch_info(self.plan)

    def set_timing(self, enable=True):
        capi.moe_set_timing(self.plan, enable)

    def timings(self):
        return capi.moe_timings(self.plan, 6)

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

    def __init__(self, W, L, topk, T, d_model, d_ff, tb_M, mgb=1,
                 consumer_ctas=capi.MOE_CONSUMER_FUSED, timeout_ns=0, producer_pairs=1,
                 device=None, scale_mode="after"):
        """consumer_ctas: MOE_CONSUMER_FUSED (-1, the copy runs in a warp of every pair
        producer CTA), 0 (serial), or the consumer CTAs beside the producer.
        scale_mode: "after" (moe_scale once the combine is done) or "gated"
        (moe_scale_gated: the scale starts beside the producer and waits on the device
        for each token's group signals and ready flags)."""
        if scale_mode not in ("after", "gated"):
            raise ValueError(f"scale_mode {scale_mode!r}")
        self.scale_mode = scale_mode
        # The moe_gate splits argument of forward() and HostPipeline steps routed from a
        # router: 0 picks the kernel; MOE_GATE_BESIDE (E <= 16) takes CTAs that fit
        # beside a running producer, for batches in flight.
        self.gate_splits = 0
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
        # The zero fills above ran on the current stream, and the layer's kernels run on
        # the caller's streams, which torch creates non-blocking: without this wait a
        # first combine could start while the plan workspace (counters, flags, status)
        # or a receive buffer is still being zeroed.
        torch.cuda.synchronize(dev)

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

    def gate(self, x, w_router, forced_ids=None, stream=None, logits_out=None, splits=0):
        """Router scores of the token rows and their routing, in one kernel.

        x: W tensors [T, D] bf16; w_router: [E, D] bf16 (E <= 256). logits_out: an
        optional [W, T, E] fp32 tensor that receives the scores. splits: 0 picks the
        kernel (for E <= 16 the one that streams the token rows into registers, else
        the tcgen05 kernel with the K split it picks); 1, 2, 4 or 8 force the tcgen05
        kernel with that K split; capi.DEFINES["MOE_GATE_BESIDE"] (E <= 16) takes the
        small CTAs that fit beside a running producer CTA."""
        capi.moe_gate(self.plan, [t.data_ptr() for t in x], w_router.data_ptr(),
                      None if forced_ids is None else forced_ids.data_ptr(),
                      self.ids.data_ptr(), self.w.data_ptr(),
                      None if logits_out is None else logits_out.data_ptr(), splits,
                      _stream_handle(stream))
        return self.ids, self.w

    def plan_build(self, x, ids=None, stream=None, from_gate=False):
        """from_gate: build from the routing of the last gate() call, whose routing
        tail already set the plan's token bitmaps (one plan kernel fewer)."""
        if from_gate:
            capi.moe_plan_build(self.plan, None, [t.data_ptr() for t in x], _stream_handle(stream))
            return
        ids = self.ids if ids is None else ids
        capi.moe_plan_build(self.plan, ids.data_ptr(), [t.data_ptr() for t in x],
                            _stream_handle(stream))

    def expert_combine(self, w_gate, w_up, w_down, producer=None, consumer=None):
        sp = _stream_handle(producer)
        sc = sp if consumer is None else _stream_handle(consumer)
        capi.moe_expert_combine(self.plan, [t.data_ptr() for t in w_gate],
                                [t.data_ptr() for t in w_up], [t.data_ptr() for t in w_down],
                                [t.data_ptr() for t in self.recv], sp, sc)

    def scale(self, w=None, stream=None, out=None):
        """out: W tensors [T, D] bf16 to write (default: the layer's own outputs)."""
        w = self.w if w is None else w
        out = self.out if out is None else out
        capi.moe_scale(self.plan, w.data_ptr(), [t.data_ptr() for t in self.recv],
                       [t.data_ptr() for t in out], _stream_handle(stream))
        return out

    def scale_gated(self, w=None, stream=None, out=None):
        """The scale overlapped with the combine just enqueued on `stream` (its producer
        stream): same results as scale()."""
        w = self.w if w is None else w
        out = self.out if out is None else out
        capi.moe_scale_gated(self.plan, w.data_ptr(), [t.data_ptr() for t in self.recv],
                             [t.data_ptr() for t in out], _stream_handle(stream))
        return out

    def scale_step(self, stream=None, out=None):
        """The scale of a step, in the layer's scale_mode."""
        if self.scale_mode == "gated":
            return self.scale_gated(stream=stream, out=out)
        return self.scale(stream=stream, out=out)

    def forward(self, x, w_gate, w_up, w_down, logits=None, forced_ids=None, producer=None,
                consumer=None, out=None, w_router=None):
        """route -> plan -> overlapped FFN and combine -> scale; all on the GPU.

        The routing comes from the gate logits, or, given w_router instead, from the
        router's scores of x (gate()). Every call is enqueued on `producer` (and
        `consumer`): inputs written on another stream must be complete before it (an
        event or a synchronize)."""
        if (logits is None) == (w_router is None):
            raise ValueError("give exactly one of logits and w_router")
        if w_router is not None:
            self.gate(x, w_router, forced_ids, producer, splits=self.gate_splits)
        else:
            self.route(logits, forced_ids, producer)
        self.plan_build(x, stream=producer, from_gate=w_router is not None)
        self.expert_combine(w_gate, w_up, w_down, producer, consumer)
        return self.scale_step(stream=producer, out=out)

    def capture(self, x, w_gate, w_up, w_down, logits=None, forced_ids=None, producer=None,
                consumer=None, out=None, w_router=None):
        """Records one step (route, plan, combine, scale) into a CUDA graph over these
        tensors. Replaying it (graph.replay()) runs the step on whatever the tensors hold
        then, with one launch from the host. Every call the step makes is asynchronous
        and allocates nothing, so the whole path is capturable; the event fork and join
        between the producer and consumer streams become graph edges."""
        sp = producer if producer is not None else torch.cuda.Stream(device=self.device)
        sc = consumer if consumer is not None else torch.cuda.Stream(device=self.device,
                                                                     priority=-1)
        torch.cuda.synchronize(self.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=sp):
            self.forward(x, w_gate, w_up, w_down, logits, forced_ids, sp, sc, out=out,
                         w_router=w_router)
        return graph

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

    def set_schedule(self, consumer_ctas: int, mgb: int):
        """Consumer partition (0 = serial) and segment merge width; the next plan build
        and combine use them."""
        capi.moe_set_schedule(self.plan, consumer_ctas, mgb)
        self.cfg.consumer_ctas, self.cfg.mgb = consumer_ctas, mgb

    def tune(self, x, w_gate, w_up, w_down, logits, forced_ids=None, producer=None,
             consumer=None, candidates=((-1, 1), (0, 1), (4, 1), (8, 1), (14, 1), (4, 2)),
             steps=6, rounds=3):
        """Adaptive schedule: times whole steps on these inputs for each (consumer_ctas,
        mgb) candidate and keeps the fastest. Returns (consumer_ctas, mgb, {candidate:
        median ms per step}). Candidates the shape does not support are skipped. The
        candidates take turns over `rounds` rounds, each in a rotated order, and each
        keeps its median: the GPU's clocks follow its power draw, so a candidate timed
        right after a slow (low-power) one would otherwise start at higher clocks."""
        sp = producer if producer is not None else torch.cuda.Stream(device=self.device)
        sc = consumer if consumer is not None else torch.cuda.Stream(device=self.device,
                                                                     priority=-1)
        keep = (self.cfg.consumer_ctas, self.cfg.mgb)
        usable = []
        for cand in candidates:
            try:
                self.set_schedule(*cand)
            except capi.MoeError:
                continue
            usable.append(tuple(cand))
        samples = {c: [] for c in usable}
        run = lambda: self.forward(x, w_gate, w_up, w_down, logits, forced_ids, sp, sc)
        for r in range(max(1, rounds)):
            k = r % len(usable) if usable else 0
            for cc, mgb in usable[k:] + usable[:k]:
                self.set_schedule(cc, mgb)
                run()
                run()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(sp)
                for _ in range(steps):
                    run()
                e1.record(sp)
                e1.synchronize()
                if self.status() != (0, 0):
                    raise capi.MoeError(f"device status {self.status()} while tuning {cc, mgb}")
                samples[(cc, mgb)].append(e0.elapsed_time(e1) / steps)
        times = {c: sorted(v)[len(v) // 2] for c, v in samples.items()}
        best = min(times, key=times.get) if times else keep
        self.set_schedule(*best)
        return best[0], best[1], times

    def launch_info(self):
        """(producer_ctas, consumer_ctas, num_sms, pair_clusters) of the overlapped schedule."""
        return capi.moe_launch_info(self.plan)

    def set_timing(self, enable=True):
        """True/1: CUDA events and device-clock records; 2: device-clock records only
        (nothing enters the streams); False/0: off."""
        capi.moe_set_timing(self.plan, enable)

    def timings(self):
        """[route or gate, plan, producer, consumer, scale, gather, producer span,
        scale span, scale time before the producer's end, gate span, consumer-kernel
        span, gather span] in ms (-1: none)."""
        return capi.moe_timings(self.plan, 12)

    def producer_spans(self):
        """[(start_ns, end_ns)] of the producer launches recorded while timing (device
        clock), oldest first."""
        return capi.moe_producer_spans(self.plan)

    def combine_overlap(self):
        """(share of the combine's bytes landed before the producer's last tile, µs from
        that tile to the last copy, bytes copied) of the last combine recorded."""
        return capi.moe_combine_overlap(self.plan)


class HostPipeline:
    """Steps of one MoE layer fed from and returned to pinned host memory, with the
    copies overlapped with compute: step i+1's inputs are copied in while step i
    computes, and step i's outputs are copied out while step i+1 computes.

    Two sets of device inputs (tokens, logits, forced ids) and two sets of outputs
    alternate; one copy stream per direction. Events order everything on the GPU:
    a set's inputs are overwritten only after the plan build of the step that read
    them, and its outputs only after their copy to the host finished. Every step
    still moves all of its input and output bytes; nothing is cached across steps.

    `layer` may also be a list of ExpertCombine instances of the same layer (same
    shape, own workspaces): step i then runs on instance i % len, on its own streams,
    so the routing, plan and gather of one batch overlap the expert FFN of the
    previous one (batches in flight).
    """

    def __init__(self, layer, producer=None, consumer=None, forced=False):
        self.layers = list(layer) if isinstance(layer, (list, tuple)) else [layer]
        lay0 = self.layers[0]
        dev = lay0.device
        W, T, D, E, k = lay0.W, lay0.T, lay0.D, lay0.W * lay0.L, lay0.k
        n = max(2, len(self.layers))
        self.nbuf = n
        self.sp = [producer or torch.cuda.Stream(device=dev)] + \
            [torch.cuda.Stream(device=dev) for _ in self.layers[1:]]
        self.sc = [consumer or torch.cuda.Stream(device=dev, priority=-1)] + \
            [torch.cuda.Stream(device=dev, priority=-1) for _ in self.layers[1:]]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.x = [[torch.empty(T, D, dtype=torch.bfloat16, device=dev) for _ in range(W)]
                  for _ in range(n)]
        self.logits = [torch.empty(W, T, E, dtype=torch.float32, device=dev) for _ in range(n)]
        self.forced = [torch.empty(W, T, k, dtype=torch.int32, device=dev) if forced else None
                       for _ in range(n)]
        self.out = [[torch.empty(T, D, dtype=torch.bfloat16, device=dev) for _ in range(W)]
                    for _ in range(n)]
        ev = lambda: [torch.cuda.Event() for _ in range(n)]
        self.ev_in, self.ev_free, self.ev_done, self.ev_out = ev(), ev(), ev(), ev()
        self.started = [False] * n
        self.i = 0

    @property
    def sp0(self):
        return self.sp[0]

    def step(self, hx, hlogits, hforced, hout, w_gate, w_up, w_down, start_after=None,
             w_router=None):
        """Enqueue one step. hx: W pinned [T, D] bf16; hlogits: pinned [W, T, E] fp32;
        hforced: pinned [W, T, k] int32 or None; hout: W pinned [T, D] bf16 written when
        the step's output copy completes (after self.done_event() of this step).
        start_after: an event the first copy must follow (for timing). With w_router
        (a device [E, D] bf16 tensor) the routing comes from the gate kernel on the
        copied tokens and hlogits must be None: no logits cross the host link."""
        if (hlogits is None) == (w_router is None):
            raise ValueError("give exactly one of hlogits and w_router")
        b = self.i % self.nbuf
        li = self.i % len(self.layers)
        lay, sp, sc = self.layers[li], self.sp[li], self.sc[li]
        if start_after is not None:
            self.s_in.wait_event(start_after)
        if self.started[b]:
            self.s_in.wait_event(self.ev_free[b])
        with torch.cuda.stream(self.s_in):
            for d, h in zip(self.x[b], hx):
                d.copy_(h, non_blocking=True)
            if hlogits is not None:
                self.logits[b].copy_(hlogits, non_blocking=True)
            if hforced is not None:
                self.forced[b].copy_(hforced, non_blocking=True)
        self.ev_in[b].record(self.s_in)
        sp.wait_event(self.ev_in[b])
        fid = self.forced[b] if hforced is not None else None
        if w_router is not None:
            lay.gate(self.x[b], w_router, fid, sp, splits=lay.gate_splits)
        else:
            lay.route(self.logits[b], fid, sp)
        lay.plan_build(self.x[b], stream=sp, from_gate=w_router is not None)
        self.ev_free[b].record(sp)
        # The output set is rewritten only after its previous copy to the host; the wait
        # comes before the combine, so nothing separates the combine from the scale.
        if self.started[b]:
            sp.wait_event(self.ev_out[b])
        lay.expert_combine(w_gate, w_up, w_down, sp, sc)
        lay.scale_step(stream=sp, out=self.out[b])
        self.ev_done[b].record(sp)
        self.s_out.wait_event(self.ev_done[b])
        with torch.cuda.stream(self.s_out):
            for h, o in zip(hout, self.out[b]):
                h.copy_(o, non_blocking=True)
        self.ev_out[b].record(self.s_out)
        self.started[b] = True
        self.i += 1
        return self.ev_out[b]

    def done_event(self):
        """Event completed when the last enqueued step's outputs are on the host."""
        return self.ev_out[(self.i - 1) % self.nbuf]

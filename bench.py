"""Throughput of the tile-signalled MoE expert-combine path on GB300.

One step = the whole path over one batch of synthetic input: gate routing,
plan build (layout, schedule, combine plan) with the layout gather, the
overlapped expert FFN producer and combine consumer, and the scale. The
workload is the 4-rank A100-paper-like layer (W=4, 2 experts/rank, top-2,
4096 tokens/rank, d_model 2048, d_ff 8192, tb_M 128, balanced routing).

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle on the
host cores instead (a bounded sample of the same workload).
Multi-GPU: the path does not shard across GPUs (all logical ranks live on one
GPU), so `--gpus N` runs N independent replicas, one per GPU.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "a100_like"
METRIC = "MoE combine-layer tokens/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons. Only samples
    stamped between mark_start() and mark_end() (host clock) are summarised: those the
    sampler takes while the program is idle or warming up would read as full clocks."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index  # physical index or "GPU-<uuid>"
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def mark_start(self):
        import datetime
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        import datetime
        self.t1 = datetime.datetime.now()

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        import datetime
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == 8:
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    except ValueError:
                        continue
                    rows.append((ts, parts[1:]))
        os.unlink(self.file.name)
        inside = [r for ts, r in rows
                  if (self.t0 is None or ts >= self.t0) and (self.t1 is None or ts <= self.t1)]
        window = "timed region"
        if not inside:  # a region shorter than the sampling interval
            inside, window = [r for _, r in rows], "whole sampler run (none inside the region)"
        if not inside:
            return None
        sm = [float(r[0]) for r in inside if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


def source_fingerprint(names) -> str:
    """First 16 hex digits of the sha256 of the code of the named csrc files, with their
    comments and blank lines left out (a change to a comment does not change a kernel)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in names:
        text = open(os.path.join(ROOT, "tile_signaled_grouped_gb300", "csrc", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*", "", line).rstrip()
            if code.strip():
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def producer_traffic(wl_name: str, reduced: bool, pairs: int):
    """DRAM bytes (read + write) per producer launch, from the committed ncu summary of the
    A100-like full-size run of the producer in use, while its sources and the plan build
    that orders its tiles still have the fingerprint recorded there (source_fingerprint);
    None otherwise (changed kernel or tile order, other workload)."""
    import re

    if wl_name != WORKLOAD or reduced:
        return None
    summary, srcs = (("ffn_pair_a100_like.md", ("ffn_pair.cu", "combine_copy.cuh")) if pairs
                     else ("ffn_producer_a100_like.md", ("ffn.cu",)))
    try:
        text = open(os.path.join(ROOT, "profiles", summary)).read()
        # plan.cu fixes the order the producer takes its tiles in, so it is part of it.
        fp = source_fingerprint(srcs + ("moe_common.cuh", "plan.cu"))
    except OSError:
        return None
    m1 = re.search(r"traffic_bytes_per_launch: (\d+)", text)
    m2 = re.search(r"source_fingerprint: (\w+)", text)
    if not (m1 and m2) or fp != m2.group(1):
        return None
    return int(m1.group(1))


def producer_launch_ms(spans) -> float:
    """Device-clock time per producer launch: the union of the launches' spans
    [(start_ns, end_ns)] over their number (consecutive launches of batches in flight
    overlap; the union counts every moment once)."""
    busy, cur = 0, None
    for s_, e in sorted(spans):
        if cur is None or s_ > cur[1]:
            busy += 0 if cur is None else cur[1] - cur[0]
            cur = [s_, e]
        else:
            cur[1] = max(cur[1], e)
    busy += cur[1] - cur[0]
    return busy / len(spans) * 1e-6


def pick_bf16_peak(region_s: float, clocks, burst: float, sustained: float):
    """(peak, "burst" | "sustained", capped): the measured bf16 peak whose conditions match
    the timed region's. The burst figure (cuBLAS timed alone) fits a region run at full
    clocks; once the GPU holds its power cap (a region of a second or more, or a shorter
    one whose clock samples show sw_power_cap with the SM clock below its maximum) the
    sustained figure, measured in the same regime, does."""
    capped = bool(clocks and clocks.get("window") == "timed region"
                  and "sw_power_cap" in clocks.get("reasons", [])
                  and clocks.get("sm_mhz") and clocks.get("sm_max_mhz")
                  and clocks["sm_mhz"] < clocks["sm_max_mhz"])
    if region_s >= 1.0 or capped:
        return sustained, "sustained", capped
    return burst, "burst", capped


def max_over_ranks(v: float, device="cpu") -> float:
    """Largest value over the ranks of the default process group (v itself alone)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_replica: int, ms_step_max: float) -> float:
    """Whole-job throughput: every replica's tokens over the slowest replica's step."""
    return world * tokens_per_replica / (ms_step_max * 1e-3)


# --------------------------------------------------------------------------- GPU arm

def gpu_arm(args, rank, world, local_rank):
    import torch

    from tile_signaled_grouped_gb300 import capi
    from tile_signaled_grouped_gb300.runtime import ExpertCombine
    from tile_signaled_grouped_gb300.workloads import get_workload, make_inputs

    torch.cuda.set_device(local_rank)
    wl = get_workload(args.workload)
    reduced = bool(args.tokens_per_rank or args.experts_per_rank)
    if reduced:  # a smaller case of the shape (profiling): a name of its own
        over = {}
        if args.tokens_per_rank:
            over["T"] = args.tokens_per_rank
        if args.experts_per_rank:
            over["L"] = args.experts_per_rank
        wl = get_workload(args.workload, **over)
        wl = dataclasses.replace(wl, name=f"{wl.name}_L{wl.L}_T{wl.T}")
    W, T, D, F, k = wl.W, wl.T, wl.d_model, wl.d_ff, wl.topk
    inp = make_inputs(wl, device="cuda")
    # --route gate: every step routes from the token rows with the gate kernel (router
    # scores, softmax and top-k in one launch; a prescribed routing keeps its ids), and
    # the plan starts from the token bitmaps the gate's routing tail set.
    wr = None
    if args.route == "gate":
        from tile_signaled_grouped_gb300.workloads import router_weights
        if wl.E > 256:
            raise SystemExit(f"the gate kernel takes E <= 256 experts ({wl.name} has {wl.E})")
        wr = router_weights(wl, device="cuda")
    torch.cuda.synchronize()  # inputs are drawn on the default stream; the steps run on sp/sc
    # Batches in flight: instance i % n (own plan and workspaces, own streams) runs
    # step i, so one batch's routing, plan and gather overlap the previous batch's
    # expert FFN. Every step still runs the whole path on its own batch.
    n_fly = max(1, args.batches_in_flight)
    layers = [ExpertCombine(W, wl.L, k, T, D, F, wl.tb_M, wl.mgb, args.consumer_ctas,
                            producer_pairs=args.producer_pairs, scale_mode=args.scale)
              for _ in range(n_fly)]
    # With batches in flight a batch's gate overlaps the previous batch's producer:
    # for E <= 16 it takes CTAs that fit beside a producer CTA (MOE_GATE_BESIDE).
    gate_splits = {"auto": capi.DEFINES["MOE_GATE_BESIDE"] if n_fly > 1 and wl.E <= 16 else 0,
                   "default": 0, "beside": capi.DEFINES["MOE_GATE_BESIDE"]}[args.gate_shape]
    for lay in layers:
        lay.gate_splits = gate_splits
    layer = layers[0]
    sps = [torch.cuda.Stream() for _ in range(n_fly)]
    scs = [torch.cuda.Stream(priority=-1) for _ in range(n_fly)]
    sp, sc = sps[0], scs[0]
    step_i = [0]

    def step():
        j = step_i[0] % n_fly
        step_i[0] += 1
        layers[j].forward(inp.x, inp.w_gate, inp.w_up, inp.w_down,
                          None if wr is not None else inp.logits, inp.forced_ids,
                          producer=sps[j], consumer=scs[j], w_router=wr)

    for _ in range(max(args.warmup, n_fly)):
        step()
    torch.cuda.synchronize()
    for lay in layers:
        code, detail = lay.status()
        if code != 0:
            raise RuntimeError(f"device status {code} detail {detail}")

    # Counts for the algorithmic work of one step (read once, outside the timed region).
    rank_rows = layer.field(capi.MOE_PLAN_RANK_ROWS).cpu().tolist()
    recv_rows = layer.field(capi.MOE_PLAN_RECV_ROWS).cpu().tolist()
    rows_exec = sum(rank_rows)
    valid_rows = W * T * k
    flops_exec = 6.0 * rows_exec * D * F
    flops_valid = 6.0 * valid_rows * D * F

    # ---- timed region: K steps, inputs resident in HBM ------------------------------
    # The library keeps device-clock records of each combine (timing mode 2: no CUDA
    # event enters the streams, so kernels overlap exactly as untimed): the producer's
    # execution span for the roofline, the overlapped scale's span, and when each
    # combine copy chunk landed.
    for lay in layers:  # every batch's producer launches, for their union below
        lay.set_timing(2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        gpu_id = str(local_rank)
    with ClockSampler(gpu_id) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        t_wall = time.perf_counter()
        ev0.record(sp)
        for s_ in sps[1:]:
            s_.wait_event(ev0)
        for _ in range(args.steps):
            step()
        for s_ in sps[1:]:
            sp.wait_stream(s_)
        ev1.record(sp)
        torch.cuda.synchronize()
        clk.mark_end()
        if world > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - t_wall
    kernel_ms = layer.timings()
    landed, tail_us, copy_bytes = layer.combine_overlap()
    spans = [iv for lay in layers for iv in lay.producer_spans()]
    for lay in layers:
        lay.set_timing(False)
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, device="cuda")
    for lay in layers:
        code, detail = lay.status()
        if code != 0:
            raise RuntimeError(f"device status {code} detail {detail} after the timed region")

    # ---- e2e through the C ABI with host buffers, right after the timed region (the
    # same power state: the GPU sits at its power cap within a fraction of a second) ---
    e2e = e2e_arm(layers, inp, wl, sp, sc, args, wr) if not args.no_e2e else None

    # ---- stage measurements (outside the timed region) --------------------------------
    # They time kernels one at a time against the burst peaks, so they start from a
    # rested GPU: after the timed region and the e2e leg the power limiter holds the
    # clocks down for a while, and a few idle seconds release it.
    stages = None
    if not args.no_stages:
        torch.cuda.synchronize()
        time.sleep(3.0)
        stages = stage_times(layer, inp, wl, sp, sc, args)

    hbm, bf16, bf16_sus, src = _peaks()
    launch = layer.launch_info()
    # The producer's launch duration from the device clock: with batches in flight the
    # event pair around a launch also counts the time the kernel waits for the previous
    # batch's producer to leave the SMs, and consecutive launches overlap (the next
    # batch's first CTAs start on the SMs the previous one frees), so a launch's own
    # span (first CTA start to last CTA end) counts those moments twice. The time any
    # producer CTA runs, the union of all recorded launches' spans, over the number of
    # launches counts each moment once.
    prod_span_mean = sum(e - s_ for s_, e in spans) / len(spans) * 1e-6
    prod_avg = producer_launch_ms(spans)
    achieved = flops_exec / (prod_avg * 1e-3) / 1e12
    # Consecutive producer spans overlap a little (the next batch's producer starts as
    # the previous one drains), so the span rate is beside the rate per step: the
    # executed FLOPs of one step over the whole step time, which can never overlap.
    per_step = flops_exec / (ms_step * 1e-3) / 1e12
    region_s = ms_step * args.steps * 1e-3
    clocks = clk.summary()
    peak, peak_kind, capped = pick_bf16_peak(region_s, clocks, bf16, bf16_sus)
    result = {
        "metric": METRIC,
        "value": job_tokens_per_s(world, W * T, ms_step),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: x~N(0,1), weights~N(0,0.02), logits~N(0,1), balanced routing)",
        "config": {"workload": wl.name, "W": W, "experts_per_rank": wl.L, "topk": k,
                   "tokens_per_rank": T, "d_model": D, "d_ff": F, "tb_M": wl.tb_M,
                   "mgb": wl.mgb, "consumer_ctas": args.consumer_ctas,
                   "batches_in_flight": n_fly,
                   "schedule": ("fused (copy warp in every producer CTA)" if args.consumer_ctas < 0
                                else "serial" if args.consumer_ctas == 0
                                else "overlapped (consumer kernel on its own SMs)"),
                   "producer": "CTA pairs (cta_group::2, M=256)" if args.producer_pairs
                   else "one CTA per tile (M=128)",
                   "scale": ("overlapped with the producer (moe_scale_gated)"
                             if args.scale == "gated" else "after the combine (moe_scale)"),
                   "routing": (("gate kernel from the token rows (seeded router), "
                                + ("CTAs that fit beside the producer" if gate_splits < 0
                                   else "moe_gate's own choice of CTAs"))
                               if wr is not None else "from the drawn gate logits"),
                   "producer_ctas": launch[0], "consumer_ctas_launched": launch[1],
                   "num_sms": launch[2], "pair_clusters_resident": launch[3],
                   "parallelism": f"{W} logical EP ranks on 1 GPU; replicas x{world}",
                   "l2": "inputs larger than L2: 768 MB of expert weights read every step"},
        "roofline": {"kernel": ("ffn_pair (CTA pairs, " if args.producer_pairs else "ffn_producer (")
                     + "GEMM1+SiLU+GEMM2, executed rows)",
                     "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": producer_traffic(wl.name, reduced, args.producer_pairs),
                     "peak_source": (f"{src} bf16 {peak_kind} (timed region {region_s:.3f} s"
                                     + (", clocks held at the power cap" if capped else "")
                                     + "; burst below 1 s at full clocks, sustained otherwise)"),
                     "frac_of_burst": achieved / bf16, "frac_of_sustained": achieved / bf16_sus,
                     "flops_per_launch": flops_exec, "launch_ms": prod_avg,
                     "launch_ms_source": ("device clock: the union of the spans (first CTA start "
                                          "to last CTA end) of the producer launches of every "
                                          "batch in the timed region, over their number"),
                     "launches_recorded": len(spans), "launches_timed": args.steps,
                     "span_mean_ms": prod_span_mean,
                     "span_mean_frac": flops_exec / (prod_span_mean * 1e-3) / 1e12 / peak,
                     "per_step_tflops": per_step, "per_step_frac": per_step / peak,
                     "per_step_source": "executed FLOPs of one step / ms_per_step"},
        "e2e": e2e,
        # route 1 + plan 5 + gather 1 + producer 1 + scale 1, + consumer kernel 1 unless
        # fused; routed by the gate: gate 1 + plan 4 (the gate set the token bitmaps)
        "gpu_launches": ((9 if wr is None else 8) + (0 if args.consumer_ctas < 0 else 1))
        * args.steps,
        "clocks": clocks,
        "stages": stages,
        "work": {"rows_executed": rows_exec, "rows_valid": valid_rows,
                 "tflop_executed": flops_exec / 1e12, "tflop_valid": flops_valid / 1e12,
                 "recv_rows": recv_rows},
        "timed_wall_s": wall,
        "device_clock_ms_in_timed_region": {
            "producer_span": kernel_ms[6], "scale_span": kernel_ms[7],
            "scale_before_producer_end": kernel_ms[8]},
        # TileMoE notes 7.3: how much of the second all-to-all the FFN hides. Here: the
        # share of the combine's bytes whose copies had landed when the producer
        # finished its last output tile (last combine of the timed region).
        "combine_overlap": {"landed_before_last_tile": landed, "last_copy_after_last_tile_us": tail_us,
                            "copy_bytes": copy_bytes},
    }
    for lay in layers:
        lay.close()
    del layers, inp
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if not args.no_other_workloads and not reduced:
        result["other_workloads"] = other_workloads(args, wl.name)
    return result


class L2Flush:
    """Evicts the L2 (129 MB) before a timed kernel: a 512 MB write, then a read of the
    same 512 MB. The write alone would leave up to the L2's size in dirty lines, whose
    write-back then lands inside the next timed kernel and counts against it (the gate
    on A100-like measured 15.6 us after a write and 13.0 us after a write and a read);
    the read replaces them with clean lines of a buffer no timed kernel touches."""

    def __init__(self, nbytes=512 << 20):
        import torch

        self.buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.words = self.buf.view(torch.int32)
        self.out = torch.empty((), dtype=torch.int64, device="cuda")

    def __call__(self, stream=None):
        import torch

        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            self.buf.zero_()
            torch.sum(self.words, dim=0, dtype=torch.int64, out=self.out)


def other_workloads(args, skip):
    """The other workload shapes at full size, each with the bench's default schedule
    (fused producer and copy, two batches in flight): whole-step time from CUDA events
    over a few steps (device inputs; but for the tiny shape the expert weights are
    larger than L2 and stream from HBM every step), the producer's device-clock span and
    its share of the bf16 burst peak, and the combine overlap."""
    import torch

    from tile_signaled_grouped_gb300 import capi
    from tile_signaled_grouped_gb300.runtime import ExpertCombine
    from tile_signaled_grouped_gb300.workloads import WORKLOADS, make_inputs

    _, bf16, _, src = _peaks()
    out = {}
    for name, wl in WORKLOADS.items():
        if name == skip:
            continue
        inp = make_inputs(wl, device="cuda")
        torch.cuda.synchronize()
        lays = [ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb,
                              args.consumer_ctas, producer_pairs=args.producer_pairs,
                              scale_mode=args.scale) for _ in range(2)]
        sps = [torch.cuda.Stream(), torch.cuda.Stream()]
        scs = [torch.cuda.Stream(priority=-1), torch.cuda.Stream(priority=-1)]

        def run(i):
            lays[i % 2].forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits,
                                inp.forced_ids, producer=sps[i % 2], consumer=scs[i % 2])

        for i in range(4):
            run(i)
        torch.cuda.synchronize()
        steps = 10
        for lay in lays:
            lay.set_timing(2)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(sps[0])
        sps[1].wait_event(ev0)
        for i in range(steps):
            run(i)
        sps[0].wait_stream(sps[1])
        ev1.record(sps[0])
        torch.cuda.synchronize()
        for lay in lays:
            if lay.status() != (0, 0):
                raise RuntimeError(f"device status {lay.status()} on {name}")
        landed, tail_us, copy_bytes = lays[0].combine_overlap()
        prod_ms = producer_launch_ms([iv for lay in lays for iv in lay.producer_spans()])
        rows = int(lays[0].field(capi.MOE_PLAN_RANK_ROWS).sum().item())
        flops = 6.0 * rows * wl.d_model * wl.d_ff
        ms = ev0.elapsed_time(ev1) / steps
        out[name] = {
            "ms_per_step": ms, "tokens_per_s": wl.W * wl.T / (ms * 1e-3), "steps": steps,
            "producer_launch_ms": prod_ms,
            "producer_tflops": flops / (prod_ms * 1e-3) / 1e12,
            "producer_frac": flops / (prod_ms * 1e-3) / 1e12 / bf16,
            "per_step_frac": flops / (ms * 1e-3) / 1e12 / bf16,
            "peak": f"{src} bf16 burst {bf16}",
            "tflop_executed": flops / 1e12,
            "tflop_valid": 6.0 * wl.W * wl.T * wl.topk * wl.d_model * wl.d_ff / 1e12,
            "combine_landed_before_last_tile": landed,
        }
        for lay in lays:
            lay.close()
        del lays, inp
        torch.cuda.empty_cache()
    return out


def measure_gate(lay, x, wl, stream, iters, warmup, hbm, splits=0):
    """The gate (router scores + softmax + top-k in one launch) on the tokens x with the
    workload's seeded router, L2 flushed before each launch (L2Flush); CUDA events of
    the library around each launch (launch latency included) and the kernel's
    device-clock span, medians. splits 0: the kernel moe_gate picks (for E <= 16 the
    one that streams the token rows into registers); 1-8: the tcgen05 kernel."""
    import torch

    from tile_signaled_grouped_gb300.workloads import router_weights

    W, T, D, k = wl.W, wl.T, wl.d_model, wl.topk
    wr = router_weights(wl, device="cuda")
    flush = L2Flush()
    lay.set_timing(False)
    for _ in range(warmup):
        lay.gate(x, wr, stream=stream, splits=splits)
    torch.cuda.synchronize()
    # Right after seconds of the producer's tensor work at the power cap the same launch
    # measured about 6 % slower (A100-like rows gate: 13.7 against 12.9 us) for a few
    # milliseconds; a pause lets the GPU settle so the kernel is measured on its own.
    time.sleep(0.2)
    g, gs = [], []
    for _ in range(iters):
        flush(stream)
        lay.set_timing(True)
        lay.gate(x, wr, stream=stream, splits=splits)
        t = lay.timings()
        g.append(t[0])
        gs.append(t[9])
        lay.set_timing(False)
    code, detail = lay.status()
    if code != 0:
        raise RuntimeError(f"device status {code} detail {detail} in the gate kernel")
    ms = statistics.median(g)
    span = statistics.median(gs)
    nbytes = 2.0 * D * W * T + 2.0 * D * wl.E + 8.0 * W * T * k
    flops = 2.0 * W * T * D * wl.E
    kernel = "gate_rows_kernel" if splits == 0 and wl.E <= 16 else "gate_kernel"
    return {"kernel": kernel, "splits": splits,
            "ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "tflops": flops / (ms * 1e-3) / 1e12,
            "timing": "CUDA events around the launch (launch latency included), "
                      "L2 flushed (512 MB write, then read) before each, median of %d, "
                      "0.2 s after any earlier work" % iters,
            "span_ms": span, "span_gbs": nbytes / (span * 1e-3) / 1e9,
            "span_frac_hbm": nbytes / (span * 1e-3) / 1e9 / hbm,
            "span_timing": "device clock, first CTA start to last CTA end, median"}


def gate_arm(args):
    """--gate-only: the gate kernel alone on the workload's tokens (its own routing,
    seeded router, no expert weights allocated), one JSON line."""
    import dataclasses

    import torch

    from tile_signaled_grouped_gb300.runtime import ExpertCombine
    from tile_signaled_grouped_gb300.workloads import get_workload, make_inputs

    wl = get_workload(args.workload, routing="gate")
    if args.tokens_per_rank:
        wl = dataclasses.replace(wl, T=args.tokens_per_rank)
    if wl.E > 256:
        raise SystemExit(f"the gate kernel takes E <= 256 experts ({wl.name} has {wl.E})")
    torch.cuda.set_device(0)
    inp = make_inputs(wl, device="cuda", with_weights=False)
    torch.cuda.synchronize()
    lay = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb)
    sp = torch.cuda.Stream()
    hbm, _, _, src = _peaks()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(0).uuid)
    except Exception:
        gpu_id = "0"
    with ClockSampler(gpu_id) as clk:
        clk.mark_start()
        g = measure_gate(lay, inp.x, wl, sp, args.steps, args.warmup, hbm)
        clk.mark_end()
    # The tcgen05 kernel on the same tokens, for comparison, where the automatic
    # choice is the other kernel.
    other = (measure_gate(lay, inp.x, wl, sp, args.steps, args.warmup, hbm, splits=1)
             if wl.E <= 16 else None)
    lay.close()
    ntok = wl.W * wl.T
    return {
        "metric": "gate tokens/s", "value": ntok / (g["ms"] * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": g["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded: x~N(0,1), router~N(0,1/D))",
        "config": {"workload": wl.name, "kernel": g["kernel"], "W": wl.W,
                   "experts": wl.E, "topk": wl.topk, "tokens_per_rank": wl.T,
                   "d_model": wl.d_model,
                   "l2": "flushed before each launch (512 MB write, then read)"},
        "roofline": {"kernel": g["kernel"], "bound": "hbm", "achieved": g["gbs"],
                     "peak": hbm, "unit": "GB/s", "frac": g["frac_hbm"], "traffic": None,
                     "span_ms": g["span_ms"], "span_achieved": g["span_gbs"],
                     "span_frac": g["span_frac_hbm"], "span_timing": g["span_timing"],
                     "peak_source": f"{src} HBM copy", "bytes_per_launch": g["bytes"],
                     "launch_ms": g["ms"], "launch_ms_source": g["timing"]},
        "tflops": g["tflops"],
        "tcgen05_gate_split1": None if other is None else {
            k: other[k] for k in ("ms", "span_ms", "span_frac_hbm", "frac_hbm")},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }


def _frac(nbytes, ms, peak_gbs):
    """Fraction of the peak HBM rate that nbytes in ms reach (None without a time)."""
    return nbytes / (ms * 1e-3) / 1e9 / peak_gbs if ms and ms > 0 else None


def stage_times(layer, inp, wl, sp, sc, args, iters=12):
    """Per-kernel times of one step, and the producer alone on every SM (serial mode)."""
    import torch

    from tile_signaled_grouped_gb300 import capi

    W, T, D, k = wl.W, wl.T, wl.d_model, wl.topk
    hbm, bf16, bf16_sus, _ = _peaks()
    layer.set_timing(True)
    acc = {}
    for _ in range(iters):
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                      producer=sp, consumer=sc)
        t = layer.timings()
        for i, name in enumerate(["route", "plan", "producer", "consumer", "scale", "gather"]):
            acc.setdefault(name, []).append(t[i])
    over = {n: statistics.median(v) for n, v in acc.items()}
    # Serial mode, each stage from a cold L2 (L2Flush before it): the producer on
    # all SMs, then the consumer on all SMs with every flag set (it follows the producer
    # on one stream, so nothing flushes between the two), the routing, the plan with
    # its gather, and the scale.
    ser = {}
    from tile_signaled_grouped_gb300.runtime import ExpertCombine
    lay2 = ExpertCombine(W, wl.L, k, T, D, wl.d_ff, wl.tb_M, wl.mgb, 0,
                         producer_pairs=args.producer_pairs)
    flush = L2Flush()

    def cold():
        flush(sp)

    lay2.set_timing(True)
    for _ in range(iters):
        cold()
        lay2.route(inp.logits, inp.forced_ids, stream=sp)
        cold()
        lay2.plan_build(inp.x, stream=sp)
        cold()
        lay2.expert_combine(inp.w_gate, inp.w_up, inp.w_down, sp, sp)
        cold()
        lay2.scale(stream=sp)
        t = lay2.timings()
        for i, name in enumerate(["route", "plan", "producer", "consumer", "scale", "gather"]):
            ser.setdefault(name, []).append(t[i])
        # Device-clock spans of the same launches (the means over the records so far;
        # the last iteration's values are the means over all of them).
        ser_span = {"producer": t[6], "scale": t[7], "consumer": t[10], "gather": t[11]}
    ser = {n: statistics.median(v) for n, v in ser.items()}
    del flush
    # Whole-step time of each schedule: consumer CTAs beside the producer (-1 fused,
    # 0 serial, n CTAs), and the scale after the combine or overlapped with it
    # (moe_scale_gated) with one batch at a time or two in flight. The GPU's clocks
    # drift as it settles at its power cap, so the configurations take turns: rounds
    # of a few steps each, the median over the rounds.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pair = [ExpertCombine(W, wl.L, k, T, D, wl.d_ff, wl.tb_M, wl.mgb, -1,
                          producer_pairs=args.producer_pairs) for _ in range(2)]
    sps = [sp, torch.cuda.Stream()]
    scs = [sc, torch.cuda.Stream(priority=-1)]
    configs = [("cc", c, "after", 1) for c in args.ccta_sweep if c >= -1] + \
              [("scale", args.consumer_ctas, m, n) for n in (1, 2) for m in ("after", "gated")]
    times = {c: [] for c in configs}
    import random
    for _round in range(4):
        # A slow configuration (one consumer CTA) draws less power, so the one after it
        # starts at higher clocks: each round takes the configurations in its own
        # (seeded) order, so that no configuration always follows the same one.
        order = list(configs)
        random.Random(_round).shuffle(order)
        for cfg in order:
            kind, cc, mode, n_fly = cfg
            for lay in pair:
                lay.set_schedule(cc, wl.mgb)
                lay.scale_mode = mode

            def run(i):
                j = i % n_fly
                pair[j].forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits,
                                inp.forced_ids, producer=sps[j], consumer=scs[j])

            for i in range(2 * n_fly):
                run(i)
            torch.cuda.synchronize()
            ev0.record(sp)
            sps[1].wait_event(ev0)
            for i in range(iters):
                run(i)
            sp.wait_stream(sps[1])
            ev1.record(sp)
            torch.cuda.synchronize()
            times[cfg].append(ev0.elapsed_time(ev1) / iters)
    for lay in pair:
        if lay.status() != (0, 0):
            raise RuntimeError(f"device status {lay.status()} in the schedule sweep")
        lay.close()
    del pair
    sweep = {str(c[1]): statistics.median(v) for c, v in times.items() if c[0] == "cc"}
    sweep_range = {str(c[1]): [min(v), max(v)] for c, v in times.items() if c[0] == "cc"}
    scale_sweep = {f"{c[2]}_x{c[3]}": statistics.median(v) for c, v in times.items()
                   if c[0] == "scale"}
    # The same step captured once into a CUDA graph and replayed (one host launch per step).
    layer.set_timing(False)
    graph = layer.capture(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                          producer=sp, consumer=sc)
    with torch.cuda.stream(sp):
        for _ in range(3):
            graph.replay()
        ev0.record(sp)
        for _ in range(iters * 4):
            graph.replay()
        ev1.record(sp)
    torch.cuda.synchronize()
    graph_ms = ev0.elapsed_time(ev1) / (iters * 4)
    del graph
    # The gate (router scores + softmax + top-k in one launch) on this shape's tokens
    # with seeded router weights, L2 flushed before each launch. It is not part of the
    # step (the workload's routing comes from its gate logits).
    gate = measure_gate(lay2, inp.x, wl, sp, 30, 3, hbm) if wl.E <= 256 else {}
    rank_rows = layer.field(capi.MOE_PLAN_RANK_ROWS).cpu().tolist()
    recv_rows = layer.field(capi.MOE_PLAN_RECV_ROWS).cpu().tolist()
    rows = sum(rank_rows)
    valid = W * T * k
    flops = 6.0 * rows * D * wl.d_ff
    cons_bytes = 4.0 * D * sum(recv_rows)
    scale_bytes = 2.0 * D * k * W * T + 2.0 * D * W * T + 8.0 * W * T * k
    # The layout gather's least DRAM traffic: every token row read once (its k copies in
    # X come from the same source row) and every valid X row written; zero rows that
    # were already zero after the previous gather are not rewritten.
    gather_bytes = 2.0 * D * (W * T + valid)
    lay2.close()
    return {
        "overlapped_ms": over,
        "serial_ms": ser,
        "step_ms_by_consumer_ctas": sweep,
        "step_ms_by_scale_and_batches_in_flight": scale_sweep,
        "step_ms_by_consumer_ctas_min_max": sweep_range,
        "schedule_sweep_timing": ("whole steps, CUDA events; 4 interleaved rounds of "
                                  f"{iters} steps per configuration, each round in its own "
                                  "seeded order, median"),
        "step_ms_graph_replay": graph_ms,
        "producer_alone_tflops": flops / (ser["producer"] * 1e-3) / 1e12,
        "producer_alone_frac_burst": flops / (ser["producer"] * 1e-3) / 1e12 / bf16,
        "producer_overlapped_tflops": flops / (over["producer"] * 1e-3) / 1e12,
        "overlap_vs_gemm_alone": max(over["producer"], over["consumer"]) / ser["producer"],
        "consumer_standalone_gbs": cons_bytes / (ser["consumer"] * 1e-3) / 1e9,
        "consumer_standalone_frac": cons_bytes / (ser["consumer"] * 1e-3) / 1e9 / hbm,
        "scale_gbs": scale_bytes / (ser["scale"] * 1e-3) / 1e9,
        "scale_frac": scale_bytes / (ser["scale"] * 1e-3) / 1e9 / hbm,
        "gather_gbs": gather_bytes / (ser["gather"] * 1e-3) / 1e9,
        "gather_frac": gather_bytes / (ser["gather"] * 1e-3) / 1e9 / hbm,
        "serial_span_ms": ser_span,
        "consumer_standalone_span_frac": _frac(cons_bytes, ser_span["consumer"], hbm),
        "scale_span_frac": _frac(scale_bytes, ser_span["scale"], hbm),
        "gather_span_frac": _frac(gather_bytes, ser_span["gather"], hbm),
        "span_timing": ("device clock, first CTA start to last CTA end, mean over the serial "
                        "iterations (no launch latency, unlike the CUDA events)"),
        "hbm_stage_timing": ("serial schedule, CUDA events around each kernel, L2 flushed "
                             "(512 MB write, then read) before the routing, the plan build (the gather "
                             "is its last kernel), the producer and the scale; the consumer "
                             "follows the producer on one stream with no flush between them"),
        "scale_in_step_gbs": (scale_bytes / (over["scale"] * 1e-3) / 1e9
                              if over["scale"] > 0 else None),  # no events around a gated scale
        "gather_in_step_gbs": gather_bytes / (over["gather"] * 1e-3) / 1e9,
        "gate": gate,
    }


def e2e_arm(layers, inp, wl, sp, sc, args, wr=None):
    """Same metric through the public API with pinned host buffers: every step copies its
    inputs in and its output out inside the timed region. The runtime's HostPipeline
    overlaps step i+1's input copy and step i-1's output copy with step i's compute."""
    import torch

    from tile_signaled_grouped_gb300.runtime import HostPipeline

    W, T, D = wl.W, wl.T, wl.d_model
    hx = [t.cpu().pin_memory() for t in inp.x]
    hl = None if wr is not None else inp.logits.cpu().pin_memory()  # the gate needs no logits
    hf = None if inp.forced_ids is None else inp.forced_ids.cpu().pin_memory()
    hout = [torch.empty(T, D, dtype=torch.bfloat16).pin_memory() for _ in range(W)]
    h2d = sum(t.numel() * t.element_size() for t in hx) + (0 if hl is None else hl.numel() * 4) + \
        (0 if hf is None else hf.numel() * 4)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    pipe = HostPipeline(layers, sp, sc, forced=hf is not None)

    def step(start_after=None):
        pipe.step(hx, hl, hf, hout, inp.w_gate, inp.w_up, inp.w_down, start_after=start_after,
                  w_router=wr)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, args.steps)
    ev0.record(sp)
    for i in range(n):
        step(ev0 if i == 0 else None)
    sp.wait_event(pipe.done_event())
    ev1.record(sp)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / n
    return {"value": W * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "pinned host buffers; step i+1's inputs and step i-1's output copied "
                      "while step i computes (two copy streams, double-buffered device sets)"}


# --------------------------------------------------------------------------- CPU oracle

def cpu_baseline(wl, seconds=15.0, max_tokens=None):
    """The oracle, as it stands, on the host cores: route, plan, FFN, combine and scale
    of the same workload with the first n tokens of every rank (n sized to run for
    about `seconds`). Returns tokens/s."""
    import numpy as np

    from oracle import moe_oracle as O
    from tile_signaled_grouped_gb300.workloads import make_inputs

    inp = make_inputs(wl, device="cpu")
    f64 = lambda t: t.float().numpy().astype(np.float64)
    xs = [f64(t) for t in inp.x]
    wg = [f64(t) for t in inp.w_gate]
    wu = [f64(t) for t in inp.w_up]
    wd = [f64(t) for t in inp.w_down]
    lg = inp.logits.numpy()
    forced = None if inp.forced_ids is None else inp.forced_ids.numpy()

    def run(n):
        t0 = time.perf_counter()
        O.forward([x[:n] for x in xs], wg, wu, wd, lg[:, :n], wl.topk, wl.L, wl.tb_M, wl.mgb,
                  None if forced is None else forced[:, :n])
        return time.perf_counter() - t0

    n = min(wl.T, 64)
    t = run(n)
    if max_tokens is None:
        max_tokens = wl.T
    n2 = int(min(max_tokens, max(n, n * seconds / max(t, 1e-3))))
    if n2 > n:
        n = n2
        t = run(n)
    return {"value": wl.W * n / t, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens of each of the {wl.W} ranks "
                      f"(route, plan, fp64 FFN, combine, scale), {t:.1f} s"}


def reference_arm(args):
    from tile_signaled_grouped_gb300.workloads import get_workload

    wl = get_workload(args.workload)
    per_step = max(5.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        cpu_baseline(wl, seconds=1.0, max_tokens=16)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(wl, seconds=per_step))
    wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "W": wl.W, "experts_per_rank": wl.L, "topk": wl.topk,
                   "tokens_per_rank": wl.T, "d_model": wl.d_model, "d_ff": wl.d_ff,
                   "tb_M": wl.tb_M, "mgb": wl.mgb},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "kind": "oracle",
                         "cores": vals[0]["cores"], "sample": vals[-1]["sample"]},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--consumer-ctas", type=int, default=-1,
                    help="-1: the copy runs in a warp of every pair-producer CTA (fused); "
                         "0: producer then consumer, serially; n > 0: n consumer CTAs beside "
                         "the producer (two kernels, two streams)")
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="override T of the workload (smaller cases for profiling)")
    ap.add_argument("--experts-per-rank", type=int, default=0,
                    help="override L of the workload (smaller cases for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stages", action="store_true",
                    help="skip the per-kernel stage measurements and schedule sweeps (short "
                         "runs, e.g. under a profiler)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg through host buffers")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the short runs of the other workload shapes")
    ap.add_argument("--batches-in-flight", type=int, default=2,
                    help="layer instances (own plan and workspaces) that take steps in turn, so "
                         "one batch's routing, plan and gather overlap the previous batch's FFN")
    ap.add_argument("--scale", default="after", choices=["after", "gated"],
                    help="after: moe_scale once the combine is done; gated: moe_scale_gated, "
                         "launched behind the producer, waits on the device for each token's "
                         "group signals and ready flags")
    ap.add_argument("--gate-shape", default="auto", choices=["auto", "default", "beside"],
                    help="with --route gate: moe_gate's own choice (default, splits 0) or, for "
                         "E <= 16, CTAs that fit beside a producer CTA (beside); auto: beside "
                         "with batches in flight")
    ap.add_argument("--route", default="logits", choices=["logits", "gate"],
                    help="logits: route from the drawn gate logits; gate: the gate kernel scores "
                         "the token rows with a seeded router (softmax and top-k in the same "
                         "launch) and sets the plan's token bitmaps")
    ap.add_argument("--producer-pairs", type=int, default=1, choices=[0, 1],
                    help="1: the CTA-pair producer (clusters of two, tcgen05 cta_group::2)")
    ap.add_argument("--gate-only", action="store_true",
                    help="time the gate kernel alone (router scores + softmax + top-k) on the "
                         "workload's tokens; one GPU")
    ap.add_argument("--ccta-sweep", type=lambda v: [int(x) for x in v.split(",") if x],
                    default=[-1, 0, 2, 4, 8, 14],
                    help="consumer-CTA counts whose step time is reported (outside the timed "
                         "region); 0 is the serial schedule")
    args = ap.parse_args()
    if args.consumer_ctas < 0 and not args.producer_pairs:
        ap.error("--consumer-ctas -1 (fused) needs the pair producer (--producer-pairs 1)")
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return
    if args.gate_only:
        if world > 1:
            ap.error("--gate-only runs on one GPU")
        print(json.dumps(gate_arm(args)), flush=True)
        return

    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

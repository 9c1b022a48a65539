"""Parity of the CUDA path against the CPU oracle, through the C ABI.

Plan arrays (layout, schedule, combine plan, segments, scale map) and the
layout gather and combine copies are compared bit-exactly; every FFN row and
every output token within the tolerance of tests/parity.py (the stated max-abs
2e-2 plus the bf16 rounding of the output, relative L2 5e-3). The workload
shapes at full size are in test_gpu_full_size.py.
"""
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

from tests import parity as P  # noqa: E402
from tile_signaled_grouped_gb300 import capi  # noqa: E402
from tile_signaled_grouped_gb300.workloads import Workload, get_workload  # noqa: E402


def _full_check(wl, mode="overlap", cctas=8):
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode=mode, consumer_ctas=cctas)
    assert layer.status() == (0, 0)
    orc = P.oracle_run(wl, inp)
    P.check_plan(layer, wl, orc.plan, orc.ids, orc.w)
    P.check_order(layer, wl, orc.plan)
    P.check_layout_and_outputs(layer, wl, inp, orc)
    layer.close()


@pytest.mark.parametrize("mode", ["serial", "overlap"])
@pytest.mark.parametrize("mgb", [1, 2])
def test_tiny_full_parity(mode, mgb):
    _full_check(get_workload("tiny", mgb=mgb), mode)


SMALL = [
    # ragged T, every band height, several ranks/experts; d_model 128 uses 128-wide GEMM2 tiles
    Workload("ragged_tb64", W=3, L=3, topk=2, T=77, d_model=256, d_ff=384, tb_M=64, routing="gate", mgb=3),
    Workload("ragged_tb128", W=4, L=2, topk=3, T=130, d_model=128, d_ff=256, tb_M=128, routing="gate"),
    Workload("ragged_tb256", W=2, L=4, topk=2, T=301, d_model=384, d_ff=128, tb_M=256, routing="gate", mgb=2),
    Workload("k_equals_E", W=2, L=2, topk=4, T=40, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("one_rank", W=1, L=3, topk=2, T=50, d_model=128, d_ff=256, tb_M=128, routing="gate"),
    Workload("T1", W=4, L=2, topk=2, T=1, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("skew_small", W=4, L=4, topk=1, T=300, d_model=256, d_ff=256, tb_M=256, routing="zipf"),
    Workload("balanced_small", W=4, L=2, topk=2, T=256, d_model=256, d_ff=512, tb_M=128, routing="balanced"),
    Workload("eight_ranks", W=8, L=4, topk=4, T=64, d_model=256, d_ff=256, tb_M=64, routing="gate", mgb=2),
    # the largest top k the library takes (32), here every expert of every rank
    Workload("k32_every_expert", W=2, L=16, topk=32, T=24, d_model=128, d_ff=128, tb_M=64,
             routing="gate"),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_shapes_full_parity(wl):
    _full_check(wl, "overlap", cctas=4)


# The producer's scheduling units keep an expert's run of tiles whole where it fits (at
# most 32 tiles), cut longer runs into near-equal parts and pack short runs together.
# long_runs: every expert's 48 remote tiles are cut into 24 + 24. mixed_runs (Zipf):
# one rank has remote runs of 48, 29 and 20 tiles (units 24, 24, 29, 20), the other
# 15, 11 and 9 (units 26, 9).
UNIT_SHAPES = [
    Workload("long_runs", W=4, L=1, topk=2, T=4096, d_model=128, d_ff=128, tb_M=128,
             routing="balanced"),
    Workload("mixed_runs", W=2, L=3, topk=2, T=8192, d_model=128, d_ff=128, tb_M=64,
             routing="zipf"),
]


@pytest.mark.parametrize("pairs", [0, 1])
@pytest.mark.parametrize("wl", UNIT_SHAPES, ids=lambda w: w.name)
def test_scheduling_units_with_long_expert_runs(wl, pairs):
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="overlap", consumer_ctas=4, pairs=pairs)
    assert layer.status() == (0, 0)
    orc = P.oracle_run(wl, inp)
    P.check_plan(layer, wl, orc.plan, orc.ids, orc.w)
    P.check_order(layer, wl, orc.plan)
    if pairs:
        P.check_pairs(layer, wl, orc.plan)
    P.check_layout_and_outputs(layer, wl, inp, orc)
    layer.close()


@pytest.mark.parametrize("mode", ["overlap", "fused"])
def test_largest_token_row(mode):
    """d_model = 10240, the largest the library takes: each copy chunk holds exactly one
    20 KB row. Plan bit-exact, copies exact, outputs within tolerance."""
    wl = Workload("D10240", W=2, L=2, topk=2, T=40, d_model=10240, d_ff=128, tb_M=64,
                  routing="gate")
    _full_check(wl, mode, cctas=4)


def test_all_local_routing_sends_nothing():
    wl = Workload("all_local", W=4, L=2, topk=2, T=96, d_model=128, d_ff=256, tb_M=64, routing="balanced")
    inp = P.inputs_for(wl)
    # every token of rank s routes to rank s's two experts
    ids = torch.stack([torch.full((wl.T,), 2 * s, dtype=torch.int32) for s in range(4)])
    inp.forced_ids = torch.stack([ids, ids + 1], dim=-1).cuda()
    layer = P.run_gpu(wl, inp)
    assert layer.status() == (0, 0)
    orc = P.oracle_run(wl, inp)
    assert orc.plan.recv_rows.sum() == 0
    P.check_plan(layer, wl, orc.plan, orc.ids, orc.w)
    P.check_layout_and_outputs(layer, wl, inp, orc)


FULL = ["a100_like", "qwen3_235b_like", "deepseek_v3_like", "stress_skew"]


def test_repeat_runs_are_identical():
    wl = get_workload("tiny")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp)
    first = [layer.field(f).clone() for f in (capi.MOE_PLAN_SCHEDULE, capi.MOE_PLAN_XSRC,
                                              capi.MOE_PLAN_SEG_FIRST, capi.MOE_PLAN_SCALE_SRC)]
    out0 = [t.clone() for t in layer.out]
    for _ in range(5):
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids)
        torch.cuda.synchronize()
        again = [layer.field(f) for f in (capi.MOE_PLAN_SCHEDULE, capi.MOE_PLAN_XSRC,
                                          capi.MOE_PLAN_SEG_FIRST, capi.MOE_PLAN_SCALE_SRC)]
        assert all(torch.equal(a, b) for a, b in zip(first, again))
        assert all(torch.equal(a, b) for a, b in zip(out0, layer.out))
    assert layer.status() == (0, 0)


def test_bad_routing_is_reported_and_recoverable():
    wl = get_workload("tiny")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp)
    bad = layer.ids.clone()
    bad[1, 3, 0] = wl.E + 5  # out of range
    layer.plan_build(inp.x, ids=bad)
    layer.expert_combine(inp.w_gate, inp.w_up, inp.w_down)
    code, detail = layer.status()
    assert code == capi.MOE_DEV_ROUTING and detail == 1 * wl.T + 3
    layer.clear_status()
    layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids)
    assert layer.status() == (0, 0)


def test_device_wait_timeout_is_reported_and_recoverable():
    """A wait bound far shorter than the producer's work makes the consumer's flag
    wait run out: the kernels return, the status says MOE_DEV_TIMEOUT, and the
    context stays usable for a normal run afterwards."""
    wl = get_workload("a100_like")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, timeout_ns=20_000)  # 20 us
    code, _ = layer.status()
    assert code == capi.MOE_DEV_TIMEOUT
    layer.close()
    layer = P.run_gpu(wl, inp)
    assert layer.status() == (0, 0)


def test_host_argument_errors():
    wl = get_workload("tiny")
    cfg = capi.moe_cfg(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, 1, 4, 0)
    pb, rb, _ = capi.moe_workspace_size(cfg)
    plan_ws = torch.zeros(pb, dtype=torch.uint8, device="cuda")
    rank = [torch.zeros(rb + 1024, dtype=torch.uint8, device="cuda") for _ in range(wl.W)]
    ptrs = [t.data_ptr() + (-t.data_ptr()) % 1024 for t in rank]
    with pytest.raises(capi.MoeError, match="WORKSPACE"):
        capi.moe_plan_create(cfg, plan_ws.data_ptr(), pb - 256, ptrs, rb)
    with pytest.raises(capi.MoeError, match="ARG"):
        capi.moe_plan_create(cfg, plan_ws.data_ptr() + 4, pb, ptrs, rb)
    plan = capi.moe_plan_create(cfg, plan_ws.data_ptr(), pb, ptrs, rb)
    with pytest.raises(capi.MoeError, match="ARG"):
        capi.moe_plan_build(plan, 0, [0] * wl.W, 0)
    # Base pointers of int32 and fp32 arrays must be 16-byte aligned too (checked on the host).
    ids = torch.zeros(wl.W * wl.T * wl.topk + 4, dtype=torch.int32, device="cuda")
    x = [torch.zeros(wl.T, wl.d_model, dtype=torch.bfloat16, device="cuda") for _ in range(wl.W)]
    with pytest.raises(capi.MoeError, match="ARG"):
        capi.moe_plan_build(plan, ids.data_ptr() + 4, [t.data_ptr() for t in x], 0)
    w = torch.zeros(wl.W * wl.T * wl.topk + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(capi.MoeError, match="ARG"):
        capi.moe_route(plan, w.data_ptr(), None, ids.data_ptr(), w.data_ptr() + 8, 0)
    capi.moe_plan_destroy(plan)


# One shape per logits-per-lane instantiation of the route kernel (E <= 32, 64, 128,
# 256, 512, 1024): routing ids bit-exact, weights to fp32 rounding, and the whole plan
# bit-exact (the plan kernels hold up to 256 experts per rank).
ROUTE_SHAPES = [
    Workload("E16", W=4, L=4, topk=3, T=40, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("E48", W=4, L=12, topk=4, T=40, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("E96", W=8, L=12, topk=6, T=24, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("E200", W=8, L=25, topk=8, T=24, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("E384", W=8, L=48, topk=8, T=16, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("E1024", W=8, L=128, topk=8, T=16, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    # the limits together: 256 experts per rank (E = 1024) and top 32
    Workload("E1024_L256_k32", W=4, L=256, topk=32, T=16, d_model=128, d_ff=128, tb_M=64,
             routing="gate"),
]


@pytest.mark.parametrize("wl", ROUTE_SHAPES, ids=lambda w: w.name)
def test_route_and_plan_for_every_expert_count(wl):
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="serial")
    assert layer.status() == (0, 0)
    ids, w, plan = P.oracle_plan(wl, inp)
    P.check_plan(layer, wl, plan, ids, w)
    P.check_order(layer, wl, plan)
    layer.close()


@pytest.mark.parametrize("mode", ["overlap", "fused"])
def test_layout_changes_between_builds(mode):
    """The gather leaves rows that were zero and stay zero untouched; with the routing
    changing from build to build (rows turn from token rows into padding and back),
    every build still has exactly its tokens' rows, zero padding rows and exact
    outputs."""
    base = SMALL[0]  # W=3, tb_M=64: many padding rows
    sets = [P.inputs_for(dataclasses.replace(base, seed=s)) for s in (0, 11, 0, 23)]
    w = sets[0]
    cc = 4 if mode == "overlap" else -1
    from tile_signaled_grouped_gb300.runtime import ExpertCombine
    layer = ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff,
                          base.tb_M, base.mgb, cc, 0, 1)
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    for inp in sets:
        inp.w_gate, inp.w_up, inp.w_down = w.w_gate, w.w_up, w.w_down
        torch.cuda.synchronize()
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                      producer=sp, consumer=sc)
        torch.cuda.synchronize()
        assert layer.status() == (0, 0)
        orc = P.oracle_run(base, inp)
        P.check_plan(layer, base, orc.plan, orc.ids, orc.w)
        P.check_layout_and_outputs(layer, base, inp, orc)
    layer.close()

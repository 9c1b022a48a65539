"""The four workload shapes at full size, every row and every token against the
CPU oracle, through the C ABI.

For each shape the oracle runs once (every token row of every owner through its
float64 FFN, h rounded to bf16 and unrounded; combine; scale), and four
schedules of the CUDA path are compared with it completely:

  * the one-CTA producer with the consumer kernel on its own SMs (two streams),
  * the CTA-pair producer with the consumer kernel on its own SMs,
  * the fused schedule the bench times (the copy warp inside the pair producer),
  * the fused schedule with the scale overlapped (moe_scale_gated),

each from a fresh layer with canaries around every buffer. Plan arrays are
bit-exact; X and the combine copies are bit-exact; every Y row and every output
token is within the tolerance of tests/parity.py; the one-CTA and pair producers
give bit-identical h and Y, and both scales the same outputs. Checks follow the
TileMoE notes' correctness validation (section 7.6: per-token outputs against a
serial baseline) and section 4.5 (globally coordinated, non-overlapping receive
offsets).
"""
import gc

import pytest
import torch

pytestmark = pytest.mark.gpu

from tests import parity as P  # noqa: E402
from tests.test_gpu_pairs import check_group_signals  # noqa: E402
from tile_signaled_grouped_gb300 import capi  # noqa: E402
from tile_signaled_grouped_gb300.workloads import get_workload  # noqa: E402

FULL = ["a100_like", "qwen3_235b_like", "deepseek_v3_like", "stress_skew"]

# (mode, consumer CTAs, producer pairs, scale)
SCHEDULES = [("overlap", 16, 0, "after"), ("overlap", 4, 1, "after"), ("fused", -1, 1, "after"),
             ("fused", -1, 1, "gated")]


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity_every_row(name):
    wl = get_workload(name)
    inp = P.inputs_for(wl)
    torch.cuda.synchronize()
    orc = P.oracle_run(wl, inp)
    hy_one = out_one = None
    for mode, cc, pairs, scale in SCHEDULES:
        layer = P.run_gpu(wl, inp, mode=mode, consumer_ctas=cc, pairs=pairs, scale_mode=scale)
        assert layer.status() == (0, 0), (mode, cc, pairs)
        if mode == "fused":  # every SM produces, none is set aside for a consumer
            assert layer.launch_info()[:2] == (layer.launch_info()[2], 0)
        P.check_plan(layer, wl, orc.plan, orc.ids, orc.w)
        P.check_order(layer, wl, orc.plan)
        if pairs:
            P.check_pairs(layer, wl, orc.plan)
        P.check_layout_and_outputs(layer, wl, inp, orc)
        check_group_signals(layer, wl, orc.plan)
        rows = [int(r) for r in orc.plan.rank_rows]
        hy = [(layer.rank_field(capi.MOE_RANK_H, o)[:rows[o]].clone(),
               layer.rank_field(capi.MOE_RANK_Y, o)[:rows[o]].clone()) for o in range(wl.W)]
        if out_one is None:
            out_one = [t.clone() for t in layer.out]
        else:  # one scale arithmetic, whatever the schedule
            for o in range(wl.W):
                assert torch.equal(layer.out[o], out_one[o]), f"out of rank {o}, {mode} {scale}"
        if hy_one is None:
            hy_one = hy
        else:  # both producers add each element's K products in the same order
            for o in range(wl.W):
                assert torch.equal(hy[o][0], hy_one[o][0]), f"h of rank {o}, {mode} {pairs}"
                assert torch.equal(hy[o][1], hy_one[o][1]), f"Y of rank {o}, {mode} {pairs}"
        layer.close()
        del layer, hy
        gc.collect()
    del hy_one, out_one, inp
    gc.collect()
    torch.cuda.empty_cache()

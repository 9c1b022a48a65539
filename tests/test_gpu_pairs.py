"""Parity of the CTA-pair producer (clusters of two CTAs, one tcgen05.mma of
M = 256 over two 128-row tiles of one expert) against the CPU oracle, through
the C ABI: the same checks as the one-CTA producer's parity tests, plus the
pair list itself (unique, so compared exactly)."""
import pytest
import torch

pytestmark = pytest.mark.gpu

from tests import parity as P  # noqa: E402
from tests.test_gpu_parity import SMALL  # noqa: E402
from tile_signaled_grouped_gb300 import capi  # noqa: E402
from tile_signaled_grouped_gb300.workloads import Workload, get_workload  # noqa: E402


def _full_check(wl, mode="overlap", cctas=8):
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode=mode, consumer_ctas=cctas, pairs=1)
    assert layer.status() == (0, 0)
    orc = P.oracle_run(wl, inp)
    P.check_plan(layer, wl, orc.plan, orc.ids, orc.w)
    P.check_order(layer, wl, orc.plan)
    P.check_pairs(layer, wl, orc.plan)
    P.check_layout_and_outputs(layer, wl, inp, orc)
    if mode == "fused" or mode == "overlap":
        check_group_signals(layer, wl, orc.plan)
    layer.close()


def check_group_signals(layer, wl, plan):
    """After a combine, exactly the (sender, destination) groups that sent rows are
    signalled."""
    sig = layer.field(capi.MOE_PLAN_GROUP_SIG).view(wl.W, wl.W).cpu()
    sent = torch.zeros(wl.W, wl.W, dtype=torch.bool)
    for o in range(wl.W):
        for dst in plan.band_dst[o]:
            sent[o, int(dst)] |= int(dst) != o
    assert torch.equal(sig.bool(), sent), "group signals"


@pytest.mark.parametrize("mode", ["serial", "overlap"])
@pytest.mark.parametrize("mgb", [1, 2])
def test_pairs_tiny_full_parity(mode, mgb):
    _full_check(get_workload("tiny", mgb=mgb), mode)


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_pairs_small_shapes_full_parity(wl):
    _full_check(wl, "overlap", cctas=4)


def test_pairs_odd_tile_counts():
    """Experts whose blocks hold an odd number of 128-row tiles leave one tile
    without a partner; its CTA's rows are computed and discarded."""
    # tiles per expert: 4, 3, 2, 2, 1, 1
    wl = Workload("odd_tiles", W=2, L=3, topk=2, T=333, d_model=256, d_ff=256, tb_M=64,
                  routing="zipf")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="serial", pairs=1)
    assert layer.status() == (0, 0)
    orc = P.oracle_run(wl, inp)
    npairs = int(layer.field(capi.MOE_PLAN_TOTALS)[5])
    pr = layer.field(capi.MOE_PLAN_PAIR)[:4 * npairs].view(-1, 4)
    assert (pr[:, 1] < 0).any(), "the shape should leave a tile alone"
    P.check_pairs(layer, wl, orc.plan)
    P.check_layout_and_outputs(layer, wl, inp, orc)


def test_pairs_match_one_cta_producer_bit_for_bit():
    """Both producers accumulate each output element over K in the same order of
    16-wide MMA steps, so h, Y and the outputs are identical."""
    wl = SMALL[0]
    inp = P.inputs_for(wl)
    one = P.run_gpu(wl, inp, mode="serial", pairs=0)
    two = P.run_gpu(wl, inp, mode="serial", pairs=1)
    assert one.status() == (0, 0) and two.status() == (0, 0)
    rows = one.field(capi.MOE_PLAN_RANK_ROWS).tolist()
    for o in range(wl.W):
        for f in (capi.MOE_RANK_H, capi.MOE_RANK_Y):
            a, b = one.rank_field(f, o)[:rows[o]], two.rank_field(f, o)[:rows[o]]
            assert torch.equal(a, b), (o, f, (a.float() - b.float()).abs().max().item())
    for a, b in zip(one.out, two.out):
        assert torch.equal(a, b)


def test_pairs_repeat_runs_are_identical():
    wl = get_workload("tiny")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, pairs=1)
    out0 = [t.clone() for t in layer.out]
    for _ in range(5):
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(out0, layer.out))
    assert layer.status() == (0, 0)


def test_pairs_device_wait_timeout_is_reported_and_recoverable():
    wl = get_workload("a100_like")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, timeout_ns=20_000, pairs=1)
    code, _ = layer.status()
    assert code == capi.MOE_DEV_TIMEOUT
    layer.close()
    layer = P.run_gpu(wl, inp, pairs=1)
    assert layer.status() == (0, 0)


# ---------------------------------------------------------------- fused variant
# consumer_ctas = MOE_CONSUMER_FUSED: no consumer kernel; one warp of every pair
# producer CTA polls the flags and copies.

@pytest.mark.parametrize("mgb", [1, 2])
def test_fused_tiny_full_parity(mgb):
    _full_check(get_workload("tiny", mgb=mgb), "fused")


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_fused_small_shapes_full_parity(wl):
    _full_check(wl, "fused")


def test_fused_device_wait_timeout_is_reported_and_recoverable():
    wl = get_workload("a100_like")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="fused", timeout_ns=20_000)
    code, _ = layer.status()
    assert code == capi.MOE_DEV_TIMEOUT
    layer.close()
    layer = P.run_gpu(wl, inp, mode="fused")
    assert layer.status() == (0, 0)


# ---------------------------------------------------------------- overlapped scale
# moe_scale_gated: launched behind the combine, it starts beside the producer and
# waits on the device for each token's group signals and ready flags.

@pytest.mark.parametrize("mode", ["fused", "serial", "overlap"])
@pytest.mark.parametrize("wl", [get_workload("tiny")] + SMALL, ids=lambda w: w.name)
def test_gated_scale_equals_scale_after(wl, mode):
    """Bit-identical outputs to the scale after the combine, and the complete oracle
    check, for every schedule of the combine (in the two-stream schedule nothing
    overlaps: the producer stream waits for the consumer before the scale)."""
    inp = P.inputs_for(wl)
    after = P.run_gpu(wl, inp, mode=mode, consumer_ctas=4, pairs=1)
    gated = P.run_gpu(wl, inp, mode=mode, consumer_ctas=4, pairs=1, scale_mode="gated")
    assert after.status() == (0, 0) and gated.status() == (0, 0)
    for a, b in zip(after.out, gated.out):
        assert torch.equal(a, b)
    orc = P.oracle_run(wl, inp)
    P.check_layout_and_outputs(gated, wl, inp, orc)
    after.close()
    gated.close()


def test_gated_scale_once_per_combine_on_its_stream():
    wl = get_workload("tiny")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="fused", scale_mode="gated")
    assert layer.status() == (0, 0)
    with pytest.raises(capi.MoeError, match="MOE_ERR_ARG"):
        layer.scale_gated()  # no combine since the last one
    sp, other = torch.cuda.Stream(), torch.cuda.Stream()
    layer.route(inp.logits, inp.forced_ids, stream=sp)
    layer.plan_build(inp.x, stream=sp)
    layer.expert_combine(inp.w_gate, inp.w_up, inp.w_down, sp)
    with pytest.raises(capi.MoeError, match="MOE_ERR_ARG"):
        layer.scale_gated(stream=other)  # not ordered after the combine's zeroing
    layer.scale_gated(stream=sp)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    layer.close()


def test_device_clock_records_of_an_overlapped_step():
    """Timing mode 2 (device clock only): the producer's span, the overlapped scale's
    span and its part before the producer's end, and the combine's overlap record: the
    bytes copied are exactly the remote rows, a share of them landed before the last
    tile, and the last copy landed within the step."""
    wl = get_workload("qwen3_235b_like")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="fused", scale_mode="gated", canaries=False)
    layer.set_timing(2)
    sp = torch.cuda.Stream()
    for _ in range(3):
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                      producer=sp)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    t = layer.timings()
    assert all(v == -1 for v in t[:6]), "no CUDA events in mode 2"
    assert t[6] > 0 and t[7] > 0 and 0 <= t[8] <= t[7] + 1e-3, t
    landed, tail_us, nbytes = layer.combine_overlap()
    recv_rows = int(layer.field(capi.MOE_PLAN_RECV_ROWS).sum())
    assert nbytes == 2.0 * wl.d_model * recv_rows
    assert 0.0 <= landed <= 1.0 and tail_us < 1e3 * t[6], (landed, tail_us)
    layer.close()


@pytest.mark.parametrize("mode", ["overlap", "serial", "fused"])
def test_device_clock_spans_of_every_kernel(mode):
    """Timing mode 2 records each kernel's span (first CTA start to last CTA end): the
    producer, the consumer kernel (none in the fused schedule, whose copy runs inside
    the producer), the scale and the layout gather; outputs are unchanged by it."""
    wl = get_workload("a100_like", T=1024)
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode=mode, consumer_ctas=8, canaries=False)
    ref = [t.clone() for t in layer.out]
    layer.set_timing(2)
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    for _ in range(3):
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                      producer=sp, consumer=None if mode == "serial" else sc)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    t = layer.timings()
    assert len(t) == 12 and all(v == -1 for v in t[:6]), t
    assert t[6] > 0 and t[7] > 0 and t[11] > 0, t
    assert t[9] == -1, t  # no gate
    if mode == "fused":
        assert t[10] == -1, t
    else:
        assert t[10] > 0, t
    if mode == "serial":  # one stream: the scale starts after the producer has ended
        assert t[8] == 0, t
    assert all(torch.equal(a, b) for a, b in zip(ref, layer.out))
    layer.close()


def test_producer_spans_one_interval_per_combine():
    """moe_producer_spans: one (start, end) per combine recorded while timing, oldest
    first, on the device clock (here more launches than a timed region of a few hundred
    steps has per batch); their mean is the producer span of moe_timings slot 6."""
    wl = get_workload("tiny")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="fused", canaries=False)
    sp = torch.cuda.Stream()
    layer.set_timing(2)
    n = 150
    for _ in range(n):
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                      producer=sp)
    torch.cuda.synchronize()
    spans = layer.producer_spans()
    t = layer.timings()
    assert len(spans) == n
    assert all(0 < s0 < e0 for s0, e0 in spans)
    assert all(spans[i][0] >= spans[i - 1][1] for i in range(1, n))  # one stream: in turn
    mean_ms = sum(e0 - s0 for s0, e0 in spans) / n * 1e-6
    assert abs(mean_ms - t[6]) <= 1e-3 * t[6] + 1e-6, (mean_ms, t[6])
    layer.set_timing(0)
    with pytest.raises(capi.MoeError, match="ARG"):  # records are off
        layer.producer_spans()
    layer.close()


def test_gated_scale_device_wait_timeout_is_reported_and_recoverable():
    wl = get_workload("a100_like")
    inp = P.inputs_for(wl)
    layer = P.run_gpu(wl, inp, mode="fused", timeout_ns=20_000, scale_mode="gated")
    code, _ = layer.status()
    assert code == capi.MOE_DEV_TIMEOUT
    layer.close()
    layer = P.run_gpu(wl, inp, mode="fused", scale_mode="gated")
    assert layer.status() == (0, 0)

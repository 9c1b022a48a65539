"""HostPipeline: steps fed from and returned to pinned host memory with the copies
overlapped with compute. Each step's host output must equal the output of a plain
forward on device inputs, bit for bit, although consecutive steps use different
inputs and the double-buffered device sets alternate."""
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu

from tile_signaled_grouped_gb300.runtime import ExpertCombine, HostPipeline  # noqa: E402
from tile_signaled_grouped_gb300.workloads import get_workload, make_inputs  # noqa: E402


@pytest.mark.parametrize("n_layers,cctas,scale", [(1, 4, "after"), (2, 4, "after"),
                                                  (2, -1, "after"), (2, -1, "gated")])
@pytest.mark.parametrize("name", ["tiny", "a100_like"])
def test_pipelined_steps_equal_plain_forward(name, n_layers, cctas, scale):
    base = get_workload(name)
    sets = [make_inputs(get_workload(name, seed=s), device="cuda", with_weights=s == 0)
            for s in (0, 3, 5)]
    w = sets[0]  # one set of expert weights for every step
    torch.cuda.synchronize()  # inputs are drawn on the default stream; the layer runs on others
    mk = lambda: ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff,
                               base.tb_M, base.mgb, consumer_ctas=cctas, scale_mode=scale)
    ref_layer = mk()
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    want = []
    for inp in sets:
        out = ref_layer.forward(inp.x, w.w_gate, w.w_up, w.w_down, inp.logits, inp.forced_ids,
                                producer=sp, consumer=sc)
        torch.cuda.synchronize()
        assert ref_layer.status() == (0, 0)
        want.append([t.cpu().clone() for t in out])
    layers = [mk() for _ in range(n_layers)]  # 2: batches in flight, each on its own instance
    forced = sets[0].forced_ids is not None
    pipe = HostPipeline(layers if n_layers > 1 else layers[0], forced=forced)
    order = [0, 1, 2, 1, 0, 2, 2]
    houts = []
    for i in order:
        inp = sets[i]
        hx = [t.cpu().pin_memory() for t in inp.x]
        hl = inp.logits.cpu().pin_memory()
        hf = inp.forced_ids.cpu().pin_memory() if forced else None
        hout = [torch.empty(base.T, base.d_model, dtype=torch.bfloat16).pin_memory()
                for _ in range(base.W)]
        pipe.step(hx, hl, hf, hout, w.w_gate, w.w_up, w.w_down)
        houts.append(hout)
    pipe.done_event().synchronize()
    torch.cuda.synchronize()
    assert all(lay.status() == (0, 0) for lay in layers)
    for i, hout in zip(order, houts):
        for got, ref in zip(hout, want[i]):
            assert torch.equal(got, ref), f"step with input set {i}"


@pytest.mark.parametrize("n_layers", [1, 2])
def test_pipelined_steps_routed_by_the_gate(n_layers):
    """The same with the routing taken by the gate kernel from the copied tokens (no
    logits cross the host link): every step equals a plain forward with the router."""
    from tile_signaled_grouped_gb300.workloads import router_weights

    name = "tiny"
    base = get_workload(name)
    sets = [make_inputs(get_workload(name, seed=s), device="cuda", with_weights=s == 0)
            for s in (0, 3, 5)]
    w = sets[0]
    wr = router_weights(base, device="cuda")
    torch.cuda.synchronize()
    mk = lambda: ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff,
                               base.tb_M, base.mgb)
    ref_layer = mk()
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    want = []
    for inp in sets:
        out = ref_layer.forward(inp.x, w.w_gate, w.w_up, w.w_down, w_router=wr, producer=sp,
                                consumer=sc)
        torch.cuda.synchronize()
        assert ref_layer.status() == (0, 0)
        want.append([t.cpu().clone() for t in out])
    layers = [mk() for _ in range(n_layers)]
    pipe = HostPipeline(layers if n_layers > 1 else layers[0])
    order = [0, 1, 2, 2, 0]
    houts = []
    for i in order:
        hx = [t.cpu().pin_memory() for t in sets[i].x]
        hout = [torch.empty(base.T, base.d_model, dtype=torch.bfloat16).pin_memory()
                for _ in range(base.W)]
        pipe.step(hx, None, None, hout, w.w_gate, w.w_up, w.w_down, w_router=wr)
        houts.append(hout)
    pipe.done_event().synchronize()
    torch.cuda.synchronize()
    assert all(lay.status() == (0, 0) for lay in layers)
    for i, hout in zip(order, houts):
        for got, ref in zip(hout, want[i]):
            assert torch.equal(got, ref), f"step with input set {i}"


def test_tuned_schedule_keeps_results_exact():
    """The adaptive schedule picks one of its candidates; the plan it then builds (new
    mgb) matches the oracle bit for bit, and the outputs the one-shot forward's."""
    from tests import parity as P
    from tile_signaled_grouped_gb300 import capi

    from tests.test_gpu_parity import SMALL
    wl = SMALL[0]  # W=3, tb_M=64, mgb=3
    inp = P.inputs_for(wl)
    torch.cuda.synchronize()
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb,
                          consumer_ctas=4)
    cands = ((-1, 1), (0, 1), (4, 1), (2, 2), (8, 3))
    cc, mgb, times = layer.tune(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits,
                                inp.forced_ids, candidates=cands, steps=2)
    assert (cc, mgb) in times and set(times) == set(cands)
    assert layer.launch_info()[1] == max(cc, 0)  # the fused schedule runs no consumer CTAs
    sp = torch.cuda.Stream()
    layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                  producer=sp, consumer=torch.cuda.Stream(priority=-1))
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    wl_t = dataclasses.replace(wl, mgb=mgb)
    orc = P.oracle_run(wl_t, inp)
    P.check_plan(layer, wl_t, orc.plan, orc.ids, orc.w)
    P.check_layout_and_outputs(layer, wl_t, inp, orc)
    with pytest.raises(capi.MoeError, match="ARG"):
        layer.set_schedule(-3, 1)
    with pytest.raises(capi.MoeError, match="ARG"):
        layer.set_schedule(4, 0)


@pytest.mark.parametrize("cctas,scale", [(-1, "after"), (4, "after"), (-1, "gated")])
def test_captured_graph_replays_exactly(cctas, scale):
    """A whole step captured into a CUDA graph (fused, or producer and consumer on two
    streams joined by events; the overlapped scale becomes a programmatic edge) and
    replayed with new inputs written into the captured tensors gives, replay by replay,
    exactly the eager step's outputs."""
    name = "tiny"
    base = get_workload(name)
    sets = [make_inputs(get_workload(name, seed=s), device="cuda") for s in (0, 4)]
    w = sets[0]
    torch.cuda.synchronize()
    eager = ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff, base.tb_M,
                          base.mgb, consumer_ctas=cctas, scale_mode=scale)
    want = []
    for inp in sets:
        out = eager.forward(inp.x, w.w_gate, w.w_up, w.w_down, inp.logits, inp.forced_ids)
        torch.cuda.synchronize()
        want.append([t.clone() for t in out])
    layer = ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff, base.tb_M,
                          base.mgb, consumer_ctas=cctas, scale_mode=scale)
    x = [t.clone() for t in sets[0].x]
    logits = sets[0].logits.clone()
    graph = layer.capture(x, w.w_gate, w.w_up, w.w_down, logits)
    for i in (1, 0, 1):
        for dst, src in zip(x, sets[i].x):
            dst.copy_(src)
        logits.copy_(sets[i].logits)
        graph.replay()
        torch.cuda.synchronize()
        assert layer.status() == (0, 0)
        for got, ref in zip(layer.out, want[i]):
            assert torch.equal(got, ref), f"replay with input set {i}"


def test_new_layer_runs_at_once_on_a_side_stream():
    """A layer used on a side stream right after construction: its zero-filled plan
    workspace and receive buffers are ready before the first combine (the fills run on
    the current stream, and torch's side streams do not wait for it). Layers are
    created where the previous one's memory was just freed, the case that raced."""
    wl = get_workload("qwen3_235b_like")
    inp = make_inputs(wl, device="cuda")
    torch.cuda.synchronize()
    first = None
    for _ in range(4):
        layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb)
        sp = torch.cuda.Stream()
        layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                      producer=sp)
        torch.cuda.synchronize()
        assert layer.status() == (0, 0)
        out = [t.clone() for t in layer.out]
        if first is None:
            first = out
        assert all(torch.equal(a, b) for a, b in zip(first, out))
        layer.close()
        del layer
        torch.cuda.empty_cache()

"""HostPipeline: steps fed from and returned to pinned host memory with the copies
overlapped with compute. Each step's host output must equal the output of a plain
forward on device inputs, bit for bit, although consecutive steps use different
inputs and the double-buffered device sets alternate."""
import pytest
import torch

pytestmark = pytest.mark.gpu

from tile_signaled_grouped_gb300.runtime import ExpertCombine, HostPipeline  # noqa: E402
from tile_signaled_grouped_gb300.workloads import get_workload, make_inputs  # noqa: E402


@pytest.mark.parametrize("name", ["tiny", "a100_like"])
def test_pipelined_steps_equal_plain_forward(name):
    base = get_workload(name)
    sets = [make_inputs(get_workload(name, seed=s), device="cuda", with_weights=s == 0)
            for s in (0, 3, 5)]
    w = sets[0]  # one set of expert weights for every step
    torch.cuda.synchronize()  # inputs are drawn on the default stream; the layer runs on others
    mk = lambda: ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff,
                               base.tb_M, base.mgb, consumer_ctas=4)
    ref_layer = mk()
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    want = []
    for inp in sets:
        out = ref_layer.forward(inp.x, w.w_gate, w.w_up, w.w_down, inp.logits, inp.forced_ids,
                                producer=sp, consumer=sc)
        torch.cuda.synchronize()
        assert ref_layer.status() == (0, 0)
        want.append([t.cpu().clone() for t in out])
    layer = mk()
    forced = sets[0].forced_ids is not None
    pipe = HostPipeline(layer, forced=forced)
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
    assert layer.status() == (0, 0)
    for i, hout in zip(order, houts):
        for got, ref in zip(hout, want[i]):
            assert torch.equal(got, ref), f"step with input set {i}"

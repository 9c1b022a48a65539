"""moe_plan_build_noalloc: the plan build for callers that cannot allocate device
memory (a serving loop that reserved all of its memory up front, or a runtime
whose device memory comes from an allocator it does not own). It must produce
exactly the plan that moe_plan_build produces for the same routing, call after
call, although its internal scratch is a fixed array inside the library that
every call reuses; and that plan must drive moe_expert_combine and moe_scale.

Kept in a file of its own that pytest collects last."""
import pytest
import torch

from tests import parity as P

pytestmark = pytest.mark.gpu

from tile_signaled_grouped_gb300 import capi  # noqa: E402
from tile_signaled_grouped_gb300.runtime import ExpertCombine  # noqa: E402
from tile_signaled_grouped_gb300.workloads import get_workload, make_inputs  # noqa: E402

FIELDS = [name for name in capi.ENUMS if name.startswith("MOE_PLAN_")
          and name not in ("MOE_PLAN_NFIELDS", "MOE_PLAN_FLAGS", "MOE_PLAN_GROUP_SIG")]


def _reference_plan(wl, inp):
    """The plan of the existing entry point (routing on the GPU, then moe_plan_build)."""
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb, 4)
    layer.route(inp.logits, inp.forced_ids)
    layer.plan_build(inp.x)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    return layer


@pytest.mark.parametrize("name", ["tiny", "qwen3_235b_like", "deepseek_v3_like"])
def test_noalloc_plan_equals_plan_build_on_two_calls_in_a_row(name):
    wl = get_workload(name)
    out = None
    for call, seed in enumerate([0, 7]):
        wl_call = get_workload(name, seed=seed)
        inp = make_inputs(wl_call, device="cuda", with_weights=False)
        ref = _reference_plan(wl_call, inp)
        if out is None:
            out = torch.full((ref.plan_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
            # the plan's status word must start clear; it is an output of the call
            off, cnt = capi.moe_field(ref.cfg, capi.MOE_PLAN_STATUS)
            out[off:off + 4 * cnt] = 0
        capi.moe_plan_build_noalloc(ref.cfg, ref.ids.data_ptr(), out.data_ptr(), ref.plan_bytes,
                                    torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        for f in FIELDS:
            off, cnt = capi.moe_field(ref.cfg, capi.ENUMS[f])
            got = out[off:off + 4 * cnt].view(torch.int32)
            want = ref.field(capi.ENUMS[f])
            # Arrays are compared over what the plan defines; the tails past the
            # per-rank counts are never written by either call.
            if f in ("MOE_PLAN_BAND_EXPERT", "MOE_PLAN_BAND_DST", "MOE_PLAN_BAND_VALID",
                     "MOE_PLAN_BAND_DST_ROW", "MOE_PLAN_SCHEDULE", "MOE_PLAN_SEG_FIRST",
                     "MOE_PLAN_SEG_NBANDS", "MOE_PLAN_XSRC", "MOE_PLAN_TILE_ROW",
                     "MOE_PLAN_TILE_EXPERT", "MOE_PLAN_SEG_ORDER", "MOE_PLAN_TOTALS",
                     "MOE_PLAN_PAIR"):
                continue
            assert torch.equal(got, want), f"call {call}: {f}"
        _compare_prefixes(ref, out, wl_call)
        ref.close()


def _compare_prefixes(ref, out, wl):
    """Per-rank arrays up to their defined lengths, global lists up to their totals."""
    def view(f):
        off, cnt = capi.moe_field(ref.cfg, capi.ENUMS[f])
        return out[off:off + 4 * cnt].view(torch.int32)

    W = wl.W
    nb = (ref.field(capi.MOE_PLAN_RANK_ROWS) // wl.tb_M).tolist()
    nseg = ref.field(capi.MOE_PLAN_RANK_NSEG).tolist()
    rows = ref.field(capi.MOE_PLAN_RANK_ROWS).tolist()
    nbm = ref.field(capi.MOE_PLAN_SCHEDULE).numel() // W
    rm = ref.field(capi.MOE_PLAN_XSRC).numel() // W
    for o in range(W):
        for f, n, stride in [("MOE_PLAN_BAND_EXPERT", nb[o], nbm), ("MOE_PLAN_BAND_DST", nb[o], nbm),
                             ("MOE_PLAN_BAND_VALID", nb[o], nbm), ("MOE_PLAN_BAND_DST_ROW", nb[o], nbm),
                             ("MOE_PLAN_SCHEDULE", nb[o], nbm), ("MOE_PLAN_SEG_FIRST", nseg[o], nbm),
                             ("MOE_PLAN_SEG_NBANDS", nseg[o], nbm), ("MOE_PLAN_XSRC", rows[o], rm)]:
            a = view(f)[o * stride:o * stride + n]
            b = ref.field(capi.ENUMS[f])[o * stride:o * stride + n]
            assert torch.equal(a, b), f"{f} of rank {o}"
    tot = ref.field(capi.MOE_PLAN_TOTALS).tolist()
    assert view("MOE_PLAN_TOTALS")[:6].tolist() == tot[:6]
    for f, n in [("MOE_PLAN_TILE_ROW", tot[0]), ("MOE_PLAN_TILE_EXPERT", tot[0]),
                 ("MOE_PLAN_SEG_ORDER", tot[1]), ("MOE_PLAN_PAIR", 4 * tot[5])]:
        assert torch.equal(view(f)[:n], ref.field(capi.ENUMS[f])[:n]), f


def _plan_buffer(layer):
    """A plan workspace holding garbage except a clear status word (an output of the call)."""
    buf = torch.full((layer.plan_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    off, cnt = capi.moe_field(layer.cfg, capi.MOE_PLAN_STATUS)
    buf[off:off + 4 * cnt] = 0
    return buf


@pytest.mark.parametrize("name", ["tiny", "qwen3_235b_like"])
def test_noalloc_plan_drives_the_combine_on_two_calls_in_a_row(name):
    """A plan workspace filled only by moe_plan_build_noalloc runs moe_expert_combine and
    moe_scale (on rank workspaces whose X a moe_plan_build of the same routing filled):
    the receive buffers and outputs equal the regular path's bit for bit and the
    oracle's within the parity tolerance, for two different routings in a row into the
    same buffer. The second call allocates no device memory."""
    plan2 = handle = None
    for call, seed in enumerate([0, 7]):
        wl = get_workload(name, seed=seed)
        inp = P.inputs_for(wl)
        torch.cuda.synchronize()
        ref = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb)
        sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
        ref.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                    producer=sp, consumer=sc)
        torch.cuda.synchronize()
        assert ref.status() == (0, 0)
        if plan2 is None:
            plan2 = _plan_buffer(ref)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        capi.moe_plan_build_noalloc(ref.cfg, ref.ids.data_ptr(), plan2.data_ptr(), ref.plan_bytes,
                                    sp.cuda_stream)
        torch.cuda.synchronize()
        if call > 0:
            assert torch.cuda.mem_get_info()[0] == free0, "the call allocated device memory"
        handle = capi.moe_plan_create(ref.cfg, plan2.data_ptr(), ref.plan_bytes,
                                      [t.data_ptr() for t in ref.rank_ws], ref.rank_bytes)
        recv2 = [torch.full_like(r, 7.0) for r in ref.recv]
        out2 = [torch.full_like(o, 7.0) for o in ref.out]
        capi.moe_expert_combine(handle, [t.data_ptr() for t in inp.w_gate],
                                [t.data_ptr() for t in inp.w_up],
                                [t.data_ptr() for t in inp.w_down],
                                [t.data_ptr() for t in recv2], sp.cuda_stream, sc.cuda_stream)
        capi.moe_scale(handle, ref.w.data_ptr(), [t.data_ptr() for t in recv2],
                       [t.data_ptr() for t in out2], sp.cuda_stream)
        assert capi.moe_status(handle, sp.cuda_stream) == (0, 0)
        torch.cuda.synchronize()
        capi.moe_plan_destroy(handle)
        rr = ref.field(capi.MOE_PLAN_RECV_ROWS).tolist()
        for s_ in range(wl.W):
            assert torch.equal(recv2[s_][:rr[s_]], ref.recv[s_][:rr[s_]]), f"call {call} recv {s_}"
            assert torch.equal(out2[s_], ref.out[s_]), f"call {call} out {s_}"
        orc = P.oracle_run(wl, inp)
        for s_ in range(wl.W):
            P.assert_close(P.f64(out2[s_]), orc.out[s_], f"call {call} out rank {s_}")
        ref.close()


def test_noalloc_rejects_what_it_cannot_hold():
    # 8 ranks x 128 experts x 4096 tokens: the token bitmaps alone exceed the 1 MiB scratch
    cfg = capi.moe_cfg(8, 128, 8, 4096, 128, 128, 128, 1, 4, 0)
    pb, _, _ = capi.moe_workspace_size(cfg)
    out = torch.zeros(pb, dtype=torch.uint8, device="cuda")
    ids = torch.zeros(8 * 4096 * 8, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.MoeError, match="MOE_ERR_UNSUPPORTED"):
        capi.moe_plan_build_noalloc(cfg, ids.data_ptr(), out.data_ptr(), pb, 0)
    with pytest.raises(capi.MoeError, match="MOE_ERR_WORKSPACE"):
        capi.moe_plan_build_noalloc(get_cfg_tiny(), ids.data_ptr(), out.data_ptr(), 256, 0)


def get_cfg_tiny():
    wl = get_workload("tiny")
    return capi.moe_cfg(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb, 4, 0)

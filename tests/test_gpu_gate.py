"""Parity of the two gate kernels (router scores fused with the softmax and the top
k: on tcgen05, or for E <= 16 with the token rows streamed into registers and the
scores on mma.sync) against the float64 oracle, through the C ABI.

Tolerance (derived from the arithmetic). Each score is a sum of D products of
bf16 values; every product is exact in fp32, and the kernel adds them (and the
K-split partials) in fp32. Whatever the order, with at most D + 8 additions of
relative error <= 2u each (u = 2^-24; 2u covers round-to-nearest and truncating
adders), |score - exact| <= 2u (D + 8) sum_c |x_c w_c| + 2u |exact|.

The routing decision is taken on the kernel's own scores, so where two of the
exact scores lie within their bounds of each other either order is correct.
The check is exact feasibility: the kernel's ids, in their order, must be the
top k (ties to the lower id aside) of some score vector inside the bounds; where
every comparison is wider than the bounds this forces the oracle's ids. The
weights are then the softmax of the exact scores at the kernel's ids, within
expm1(2 max bound) for the scores' error plus 2u (E + 16) for the fp32 softmax.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from tests import parity as P  # noqa: E402
from tile_signaled_grouped_gb300 import capi  # noqa: E402
from tile_signaled_grouped_gb300.runtime import ExpertCombine  # noqa: E402
from tile_signaled_grouped_gb300.workloads import (Workload, get_workload,  # noqa: E402
                                                   make_inputs, router_weights)

U = 2.0 ** -24


def score_bound(xs, wr, lg):
    return 2 * U * (xs.shape[-1] + 8) * (np.abs(xs) @ np.abs(wr).T) + 2 * U * np.abs(lg)


def feasible(row_ids, lo, hi):
    """Whether row_ids (in order) is the descending top-k of some v with lo <= v <= hi."""
    prev = np.inf
    for a in row_ids:
        cur = min(hi[a], prev)
        if cur < lo[a]:
            return False
        prev = cur
    rest = np.ones(len(lo), dtype=bool)
    rest[list(row_ids)] = False
    return not rest.any() or lo[rest].max() <= prev


def decided(order, lo, hi, k):
    """The oracle's first k ids are the only feasible answer (every gap wider than the bounds)."""
    last = min(k + 1, len(order))
    return all(lo[order[j]] > hi[order[j + 1]] for j in range(last - 1))


def check_gate(wl, xs, wr, ids_g, w_g, lg_g, forced=None):
    """Returns (tokens checked, tokens decided by the bounds)."""
    lg = O.gate_logits(xs, wr)
    bound = score_bound(xs, wr, lg)
    if lg_g is not None:
        err = np.abs(lg_g - lg)
        worst = np.unravel_index(np.argmax(err / bound), err.shape)
        assert (err <= bound).all(), (
            f"score {worst}: |err| {err[worst]:.3e} > bound {bound[worst]:.3e}")
    ids_o, _ = O.route(lg, wl.topk, forced)
    p = O.softmax(lg)
    lo, hi = lg - bound, lg + bound
    n_dec = 0
    for s in range(wl.W):
        for t in range(wl.T):
            got = ids_g[s, t].tolist()
            if forced is not None:
                assert got == forced[s, t].tolist(), (s, t)
            else:
                assert len(set(got)) == wl.topk and all(0 <= e < wl.E for e in got), (s, t, got)
                assert feasible(got, lo[s, t], hi[s, t]), (
                    f"token ({s},{t}): ids {got} not a top-{wl.topk} within the bounds; "
                    f"oracle {ids_o[s, t].tolist()}")
                order = np.argsort(-lg[s, t], kind="stable")
                if decided(order, lo[s, t], hi[s, t], wl.topk):
                    n_dec += 1
                    assert got == ids_o[s, t].tolist(), (s, t)
            tol = np.expm1(2 * bound[s, t].max()) + 2 * U * (wl.E + 16)
            want = p[s, t, got]
            assert np.all(np.abs(w_g[s, t] - want) <= tol * want), (s, t, w_g[s, t], want, tol)
    return wl.W * wl.T, n_dec


def run_gate(wl, splits=0, forced=True, with_logits=True):
    inp = make_inputs(wl, device="cuda", with_weights=False)
    wr = router_weights(wl, device="cuda")
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb)
    lg = torch.full((wl.W, wl.T, wl.E), float("nan"), device="cuda") if with_logits else None
    fid = inp.forced_ids if forced else None
    torch.cuda.synchronize()
    layer.gate(inp.x, wr, fid, logits_out=lg, splits=splits)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    xs = np.stack([P.f64(t) for t in inp.x])
    out = (layer.ids.cpu().numpy(), layer.w.cpu().numpy(),
           None if lg is None else P.f64(lg), xs, P.f64(wr),
           None if fid is None else fid.cpu().numpy())
    layer.close()
    return out


GATE_SHAPES = [
    # E = 8 (MMA N 32), two ragged token tiles per rank
    Workload("E8_T150", W=4, L=2, topk=2, T=150, d_model=256, d_ff=128, tb_M=64, routing="gate"),
    # E = 48 (N 64), one partial tile
    Workload("E48_T77", W=4, L=12, topk=4, T=77, d_model=512, d_ff=128, tb_M=64, routing="gate"),
    # E = 96 (N 96, 128 TMEM columns), full tiles
    Workload("E96_T256", W=8, L=12, topk=6, T=256, d_model=2048, d_ff=128, tb_M=128,
             routing="gate"),
    # E = 200 (N 224), one token per rank
    Workload("E200_T1", W=8, L=25, topk=8, T=1, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    # E = 256 (N 256), ragged, D not a multiple of 8 K blocks per CTA
    Workload("E256_T300", W=8, L=32, topk=8, T=300, d_model=1152, d_ff=128, tb_M=64,
             routing="gate"),
    # k = E: every expert, ordered
    Workload("k_equals_E", W=2, L=2, topk=4, T=40, d_model=128, d_ff=128, tb_M=64,
             routing="gate"),
    # E = 24 (a thread per token, 32 candidates), D of 10 K blocks: uneven K ranges
    Workload("E24_T200", W=4, L=6, topk=3, T=200, d_model=640, d_ff=128, tb_M=64,
             routing="gate"),
]


@pytest.mark.parametrize("splits", [0, 1, 2, 4, 8])
@pytest.mark.parametrize("wl", GATE_SHAPES, ids=lambda w: w.name)
def test_gate_parity(wl, splits):
    """splits 0 is the automatic choice: the kernel that streams the token rows into
    registers for E <= 16 (E8_T150, k_equals_E), the tcgen05 kernel above; 1-8 are the
    tcgen05 kernel's K splits."""
    ids_g, w_g, lg_g, xs, wr, _ = run_gate(wl, splits)
    check_gate(wl, xs, wr, ids_g, w_g, lg_g)


# Shapes for the kernel that streams the token rows into registers (E <= 16, taken
# with splits 0): one and two n-tiles of 8 experts with padded experts, a single
# expert, every expert chosen, one token per rank, tokens per CTA that are not a
# multiple of the 16-token group, and more CTAs than one wave.
ROWS_SHAPES = [
    Workload("rows_E1", W=1, L=1, topk=1, T=37, d_model=128, d_ff=128, tb_M=64, routing="gate"),
    Workload("rows_E9_T2500", W=3, L=3, topk=3, T=2500, d_model=384, d_ff=128, tb_M=64,
             routing="gate"),
    Workload("rows_E12_T333", W=4, L=3, topk=3, T=333, d_model=640, d_ff=128, tb_M=64,
             routing="gate"),
    Workload("rows_E16_k16_T1", W=8, L=2, topk=16, T=1, d_model=256, d_ff=128, tb_M=64,
             routing="gate"),
    Workload("rows_E8_waves", W=1, L=8, topk=2, T=20000, d_model=128, d_ff=128, tb_M=64,
             routing="gate"),
]


@pytest.mark.parametrize("splits", [0, capi.DEFINES["MOE_GATE_BESIDE"]], ids=["wave", "beside"])
@pytest.mark.parametrize("wl", ROWS_SHAPES, ids=lambda w: w.name)
def test_rows_gate_parity(wl, splits):
    """splits 0: the small CTAs where they fill every SM (rows_E9_T2500, rows_E8_waves),
    else CTAs that spread the tokens over one wave; MOE_GATE_BESIDE: always the small
    CTAs that fit beside a producer CTA (32 tokens, 8 warps; 16 tokens, 4 warps with
    two n-tiles)."""
    ids_g, w_g, lg_g, xs, wr, _ = run_gate(wl, splits)
    check_gate(wl, xs, wr, ids_g, w_g, lg_g)


@pytest.mark.parametrize("T", [1024, 4096])
def test_gate_small_and_wave_ctas(T):
    """A100-like layer (4 ranks, E = 8). T = 1024: 128 small CTAs would not fill the
    GPU, so splits 0 spreads the tokens over one wave of larger CTAs while
    MOE_GATE_BESIDE keeps the small ones; both pass the feasibility check against the
    oracle (their scores differ by summation order only). T = 4096: both take the
    small CTAs, and give the same scores, ids and weights bit for bit."""
    wl = get_workload("a100_like", routing="gate", T=T)
    a = run_gate(wl, 0)
    b = run_gate(wl, capi.DEFINES["MOE_GATE_BESIDE"])
    check_gate(wl, a[3], a[4], a[0], a[1], a[2])
    check_gate(wl, b[3], b[4], b[0], b[1], b[2])
    if T == 4096:
        for x, y in zip(a[:3], b[:3]):
            assert np.array_equal(x, y)


@pytest.mark.parametrize("name", ["a100_like", "qwen3_235b_like", "deepseek_v3_like",
                                  "stress_skew"])
def test_gate_full_size(name):
    """The gate at the workload shapes (its own routing, not the prescribed one), with
    the automatic K split."""
    wl = get_workload(name, routing="gate")
    ids_g, w_g, lg_g, xs, wr, _ = run_gate(wl)
    check_gate(wl, xs, wr, ids_g, w_g, lg_g)


def test_gate_prescribed_ids_keep_the_scores_probabilities():
    wl = get_workload("a100_like", T=512)  # balanced routing: the ids are prescribed
    ids_g, w_g, lg_g, xs, wr, forced = run_gate(wl, forced=True, with_logits=False)
    check_gate(wl, xs, wr, ids_g, w_g, None, forced)


@pytest.mark.parametrize("wl,splits", [(GATE_SHAPES[4], 4), (ROWS_SHAPES[2], 0)],
                         ids=["tcgen05_split4", "rows"])
def test_gate_is_deterministic_for_a_split(wl, splits):
    a = run_gate(wl, splits=splits)
    b = run_gate(wl, splits=splits)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)


def test_gate_rejects_what_it_cannot_run():
    wl = Workload("E512", W=8, L=64, topk=2, T=16, d_model=128, d_ff=128, tb_M=64,
                  routing="gate")
    inp = make_inputs(wl, device="cuda", with_weights=False)
    wr = router_weights(wl, device="cuda")
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M)
    with pytest.raises(capi.MoeError, match="UNSUPPORTED"):
        layer.gate(inp.x, wr)
    layer.close()
    wl = GATE_SHAPES[0]
    inp = make_inputs(wl, device="cuda", with_weights=False)
    wr = router_weights(wl, device="cuda")
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M)
    with pytest.raises(capi.MoeError, match="ARG"):
        layer.gate(inp.x, wr, splits=3)
    buf = torch.zeros(wl.E * wl.d_model + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(capi.MoeError, match="ARG"):  # router not 16-byte aligned
        layer.gate(inp.x, buf[1:1 + wl.E * wl.d_model])
    layer.close()


@pytest.mark.parametrize("mode", ["fused", "overlap"])
def test_forward_from_the_router(mode):
    """route -> plan -> FFN and combine -> scale with the routing taken by the gate
    kernel: where the bounds decide every token, the ids (and so the whole plan) are
    the oracle's, and the outputs match within the path's tolerance."""
    base = Workload("gate_e2e", W=4, L=2, topk=2, T=96, d_model=256, d_ff=256, tb_M=64,
                    routing="gate")
    inp = P.inputs_for(base)
    wr = router_weights(base, device="cuda")
    wr64 = P.f64(wr)

    def undecided():
        xs = np.stack([P.f64(t) for t in inp.x])
        lg = O.gate_logits(xs, wr64)
        bound = score_bound(xs, wr64, lg)
        lo, hi = lg - bound, lg + bound
        und = [(s, t) for s in range(base.W) for t in range(base.T)
               if not decided(np.argsort(-lg[s, t], kind="stable"), lo[s, t], hi[s, t],
                              base.topk)]
        return und, xs, bound

    # Tokens whose routing the bounds leave open take the row of a decided token, so
    # that the oracle's ids are the only correct ones everywhere.
    und, xs, bound = undecided()
    ok = sorted(set((s, t) for s in range(base.W) for t in range(base.T)) - set(und))
    for n, (s, t) in enumerate(und):
        s0, t0 = ok[n % len(ok)]
        inp.x[s][t] = inp.x[s0][t0]
    und, xs, bound = undecided()
    assert not und
    ids, w = O.gate(xs, wr64, base.topk)
    plan = O.build_plan(ids, base.W, base.L, base.tb_M, base.mgb)
    cc = -1 if mode == "fused" else 4
    layer = ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff,
                          base.tb_M, base.mgb, cc, 0, 1)
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    torch.cuda.synchronize()
    layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, w_router=wr, producer=sp,
                  consumer=sc)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    tol = float(np.expm1(2 * bound.max()) + 2 * U * (base.E + 16))
    P.check_plan(layer, base, plan, ids, w, w_rtol=tol)
    P.check_layout_and_outputs(layer, base, inp, P.oracle_run(base, inp, routing=(ids, w)))
    layer.close()


def test_captured_step_from_the_router_replays_bit_exactly():
    """A whole step routed by the gate kernel, captured into a CUDA graph: replaying it
    gives the eager step's outputs bit for bit (every kernel of the step, the gate's
    K-split sum included, adds in a fixed order)."""
    base = Workload("gate_graph", W=4, L=8, topk=4, T=160, d_model=512, d_ff=256, tb_M=64,
                    routing="gate")
    inp = P.inputs_for(base)
    wr = router_weights(base, device="cuda")
    layer = ExpertCombine(base.W, base.L, base.topk, base.T, base.d_model, base.d_ff,
                          base.tb_M, base.mgb)
    sp, sc = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    torch.cuda.synchronize()
    layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, w_router=wr, producer=sp,
                  consumer=sc)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    eager = [t.clone() for t in layer.out]
    ids = layer.ids.clone()
    for t in layer.out:
        t.zero_()
    graph = layer.capture(inp.x, inp.w_gate, inp.w_up, inp.w_down, w_router=wr, producer=sp,
                          consumer=sc)
    graph.replay()
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    assert torch.equal(layer.ids, ids)
    assert all(torch.equal(a, b) for a, b in zip(eager, layer.out))
    del graph
    layer.close()


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("wl", [GATE_SHAPES[0], GATE_SHAPES[2], GATE_SHAPES[4],
                                get_workload("qwen3_235b_like", routing="gate"),
                                get_workload("a100_like")], ids=lambda w: w.name)
def test_gate_writes_the_plan_counts(wl, splits):
    """The gate's routing tail sets the plan's token bitmaps: the plan built from them
    (moe_plan_build with NULL ids, no bitmap kernel) equals, array for array, the plan
    the plan kernels build from the same ids."""
    inp = make_inputs(wl, device="cuda", with_weights=False)
    wr = router_weights(wl, device="cuda")
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb)
    torch.cuda.synchronize()
    layer.gate(inp.x, wr, inp.forced_ids, splits=splits)
    layer.plan_build(inp.x, from_gate=True)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    names = [n for n in capi.ENUMS if n.startswith("MOE_PLAN_")
             and n not in ("MOE_PLAN_NFIELDS", "MOE_PLAN_FLAGS", "MOE_PLAN_GROUP_SIG")]
    from_gate = {n: layer.field(capi.ENUMS[n]).clone() for n in names}
    layer.plan_build(inp.x, ids=layer.ids)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    for n in names:
        assert torch.equal(from_gate[n], layer.field(capi.ENUMS[n])), n
    with pytest.raises(capi.MoeError, match="ARG"):  # no gate since the last build
        layer.plan_build(inp.x, from_gate=True)
    layer.close()


def test_gate_reports_bad_prescribed_ids():
    """Prescribed ids out of range or repeated: the gate's routing tail reports the
    first token (MOE_DEV_ROUTING), like the plan build does."""
    wl = GATE_SHAPES[0]
    inp = make_inputs(wl, device="cuda", with_weights=False)
    wr = router_weights(wl, device="cuda")
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb)
    forced = torch.stack([torch.arange(wl.T) % wl.E, (torch.arange(wl.T) + 1) % wl.E],
                         dim=-1).to(torch.int32).expand(wl.W, wl.T, 2).contiguous().cuda()
    forced[2, 17, 1] = forced[2, 17, 0]  # repeated within the token
    torch.cuda.synchronize()
    layer.gate(inp.x, wr, forced)
    torch.cuda.synchronize()
    assert layer.status() == (capi.MOE_DEV_ROUTING, 2 * wl.T + 17)
    layer.clear_status()
    layer.gate(inp.x, wr)
    torch.cuda.synchronize()
    assert layer.status() == (0, 0)
    layer.close()

"""Helpers shared by the GPU parity tests: run the CUDA path, build the oracle's
view of the same inputs, and compare element by element.

Tolerance for floating-point results, against the float64 oracle: relative L2
error <= 5e-3 and, per element, |got - want| <= max(2e-2, ulp_bf16(want)).
The results are bf16 tensors. Where |want| >= 4 the spacing of bf16 values
(one ulp) is >= 0.03125, so even the correctly rounded value can sit more than
2e-2 away, and the path's two bf16 roundings (hidden activation, then output)
can land one ulp away; there the bound is that one ulp. Below |want| = 2.56 the
bound is the plain 2e-2.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from tile_signaled_grouped_gb300 import capi
from tile_signaled_grouped_gb300.runtime import ExpertCombine
from tile_signaled_grouped_gb300.workloads import make_inputs

MAX_ABS = 2e-2
REL_L2 = 5e-3


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def assert_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.size == 0:
        return
    err = np.abs(got - want)
    bound = np.maximum(MAX_ABS, bf16_ulp(want))
    worst = int(np.argmax(err / bound))
    den = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want)) / den if den > 0 else float(np.linalg.norm(got))
    assert err.flat[worst] <= bound.flat[worst] and rel <= REL_L2, (
        f"{what}: max-abs {err.max():.3e}, worst {err.flat[worst]:.3e} at |want| "
        f"{abs(want.flat[worst]):.3f} (bound {bound.flat[worst]:.3e}), rel-L2 {rel:.3e}")


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy (bf16 and fp32 widen exactly; done on the tensor's device)."""
    return t.detach().double().cpu().numpy()


def run_gpu(wl, inp, mode="overlap", consumer_ctas=8, timeout_ns=0, pairs=0):
    """The whole path through the C ABI. mode: 'overlap' (two streams), 'serial', or
    'fused' (the copy inside the pair producer); pairs: 1 runs the CTA-pair producer
    (0, the default here, keeps the one-CTA producer under test)."""
    cc = {"overlap": consumer_ctas, "serial": 0, "fused": -1}[mode]
    layer = ExpertCombine(wl.W, wl.L, wl.topk, wl.T, wl.d_model, wl.d_ff, wl.tb_M, wl.mgb,
                          cc, timeout_ns, 1 if mode == "fused" else pairs)
    sp = torch.cuda.Stream()
    sc = torch.cuda.Stream(priority=-1)
    torch.cuda.synchronize()
    layer.forward(inp.x, inp.w_gate, inp.w_up, inp.w_down, inp.logits, inp.forced_ids,
                  producer=sp, consumer=None if mode == "serial" else sc)
    torch.cuda.synchronize()
    return layer


def oracle_plan(wl, inp):
    forced = None if inp.forced_ids is None else inp.forced_ids.cpu().numpy()
    ids, w = O.route(inp.logits.cpu().numpy(), wl.topk, forced)
    return ids, w, O.build_plan(ids, wl.W, wl.L, wl.tb_M, wl.mgb)


def check_plan(layer, wl, plan, ids, w, w_rtol=2e-6):
    """Every plan array bit-exact against the oracle; the gate weights within w_rtol."""
    W, L, E = wl.W, wl.L, wl.E
    g = lambda f: layer.field(f).cpu().numpy()
    assert np.array_equal(layer.ids.cpu().numpy(), ids), "routing ids"
    np.testing.assert_allclose(layer.w.cpu().numpy(), w, rtol=w_rtol, atol=1e-9)
    assert np.array_equal(g(capi.MOE_PLAN_CNT).reshape(E, W), plan.cnt), "cnt"
    assert np.array_equal(g(capi.MOE_PLAN_GROUP_START).reshape(E, W), plan.group_start)
    assert np.array_equal(g(capi.MOE_PLAN_RECV_OFF).reshape(E, W), plan.recv_off), "recv_off"
    assert np.array_equal(g(capi.MOE_PLAN_EXPERT_START), plan.expert_start), "expert_start"
    assert np.array_equal(g(capi.MOE_PLAN_ROWS_ALLOC), plan.rows_alloc)
    assert np.array_equal(g(capi.MOE_PLAN_NRB), plan.nrb)
    assert np.array_equal(g(capi.MOE_PLAN_RANK_ROWS), plan.rank_rows)
    assert np.array_equal(g(capi.MOE_PLAN_RANK_NREMOTE), plan.n_remote)
    assert np.array_equal(g(capi.MOE_PLAN_RECV_ROWS), plan.recv_rows)
    nseg = g(capi.MOE_PLAN_RANK_NSEG)
    assert nseg.tolist() == [len(s) for s in plan.segments], "segment counts"
    nbm = g(capi.MOE_PLAN_SCHEDULE).size // W
    rm = g(capi.MOE_PLAN_XSRC).size // W
    for o in range(W):
        nb = int(plan.rank_rows[o]) // wl.tb_M
        sl = slice(o * nbm, o * nbm + nb)
        assert np.array_equal(g(capi.MOE_PLAN_BAND_EXPERT)[sl], plan.band_expert[o]), o
        assert np.array_equal(g(capi.MOE_PLAN_BAND_DST)[sl], plan.band_dst[o]), o
        assert np.array_equal(g(capi.MOE_PLAN_BAND_VALID)[sl], plan.band_valid[o]), o
        assert np.array_equal(g(capi.MOE_PLAN_BAND_DST_ROW)[sl], plan.band_dst_row[o]), o
        assert np.array_equal(g(capi.MOE_PLAN_SCHEDULE)[sl], plan.S[o]), f"S of rank {o}"
        ns = len(plan.segments[o])
        segs = np.array(plan.segments[o], dtype=np.int64).reshape(-1, 2)
        assert np.array_equal(g(capi.MOE_PLAN_SEG_FIRST)[o * nbm:o * nbm + ns], segs[:, 0])
        assert np.array_equal(g(capi.MOE_PLAN_SEG_NBANDS)[o * nbm:o * nbm + ns], segs[:, 1])
        rows = int(plan.rank_rows[o])
        assert np.array_equal(g(capi.MOE_PLAN_XSRC)[o * rm:o * rm + rows], plan.xsrc[o]), o
    assert np.array_equal(g(capi.MOE_PLAN_SCALE_SRC).reshape(W, wl.T, wl.topk), plan.src)


def check_order(layer, wl, plan):
    """The producer's tile list and the consumer's segment order: unique where the
    method fixes them (every tile exactly once; each rank's tiles in its S order;
    remote tiles before local ones), valid otherwise."""
    g = lambda f: layer.field(f).cpu().numpy()
    tot = g(capi.MOE_PLAN_TOTALS)
    ntiles, nsegs = int(tot[0]), int(tot[1])
    tr = g(capi.MOE_PLAN_TILE_ROW)[:ntiles]
    ranks, rows = tr >> 24, tr & 0xFFFFFF
    tb = wl.tb_M
    want = set()
    for o in range(wl.W):
        for li in range(wl.L):
            e = o * wl.L + li
            lo, n = int(plan.expert_start[e]), int(plan.rows_alloc[e])
            step = 128
            want |= {(o, r) for r in range(lo, lo + n, step)}
    assert sorted(zip(ranks.tolist(), rows.tolist())) == sorted(want), "tile cover"
    seen_local = False
    for o_, r_ in zip(ranks.tolist(), rows.tolist()):
        b = r_ // tb
        remote = int(plan.band_dst[o_][b]) != o_
        assert not (remote and seen_local), "a remote tile after a local tile"
        seen_local |= not remote
    for o in range(wl.W):
        pos = {int(b): i for i, b in enumerate(plan.S[o])}
        seq = [pos[r // tb] for oo, r in zip(ranks.tolist(), rows.tolist()) if oo == o]
        assert seq == sorted(seq), f"rank {o} tiles out of S order"
    so = g(capi.MOE_PLAN_SEG_ORDER)[:nsegs]
    assert nsegs == sum(len(s) for s in plan.segments)
    nbm = g(capi.MOE_PLAN_SCHEDULE).size // wl.W
    assert sorted(so.tolist()) == sorted(o * nbm + j for o in range(wl.W)
                                         for j in range(len(plan.segments[o])))


def check_pairs(layer, wl, plan):
    """The CTA-pair list, which is unique: tiles j and j^1 of one expert's block
    (rows expert_start + 128 j) form a pair, listed at the earlier of the two tile
    positions, the earlier tile first; a tile whose partner lies past the block
    is alone (partner -1)."""
    g = lambda f: layer.field(f).cpu().numpy()
    tot = g(capi.MOE_PLAN_TOTALS)
    ntiles, npairs = int(tot[0]), int(tot[5])
    tr = g(capi.MOE_PLAN_TILE_ROW)[:ntiles]
    te = g(capi.MOE_PLAN_TILE_EXPERT)[:ntiles]
    groups = {}
    for pos in range(ntiles):
        o, row, e = int(tr[pos]) >> 24, int(tr[pos]) & 0xFFFFFF, int(te[pos])
        assert e // wl.L == o
        j = (row - int(plan.expert_start[e])) // 128
        groups.setdefault((e, j // 2), []).append(pos)
    want = sorted((sorted(v) + [-1])[:2] for v in groups.values())
    rec = g(capi.MOE_PLAN_PAIR)[:4 * npairs].reshape(-1, 4)
    assert npairs == len(want), (npairs, len(want))
    assert rec[:, :2].tolist() == want, "pair list"
    for first, second, trow, info in rec.tolist():
        assert trow == int(tr[first]), "pair record: rank and row"
        assert info & 0xFFFF == int(te[first]) % wl.L, "pair record: local expert"
        if second >= 0:
            above = (int(tr[second]) & 0xFFFFFF) < (trow & 0xFFFFFF)
            assert bool(info >> 16) == above, "pair record: partner side"


def check_layout_and_outputs(layer, wl, inp, plan, ids, w, sample=None, rng=None):
    """X bit-exact; Y of valid rows within tolerance and exactly 0 on padding rows;
    receive buffers an exact copy of Y rows; outputs within tolerance.
    sample: None for every row/token, else the number sampled per rank."""
    W, T, D = wl.W, wl.T, wl.d_model
    rng = rng or np.random.default_rng(0)
    wg = [_LazyExperts(t) for t in inp.w_gate]
    wu = [_LazyExperts(t) for t in inp.w_up]
    wd = [_LazyExperts(t) for t in inp.w_down]
    xs = [f64(t) for t in inp.x]
    ycache = {}
    for o in range(W):
        rows_n = int(plan.rank_rows[o])
        X = layer.rank_field(capi.MOE_RANK_X, o)[:rows_n]
        Y = layer.rank_field(capi.MOE_RANK_Y, o)[:rows_n]
        xsrc = plan.xsrc[o]
        valid = np.nonzero(xsrc >= 0)[0]
        pad = np.nonzero(xsrc < 0)[0]
        # X: copies of token rows, zero rows elsewhere (bit-exact)
        if sample is None:
            sel = valid
        else:
            sel = np.sort(rng.choice(valid, size=min(sample, len(valid)), replace=False))
        Xs = X[torch.as_tensor(sel, device=X.device)].cpu() if len(sel) else None
        for n, r in enumerate(sel):
            s, t = divmod(int(xsrc[r]), T)
            assert torch.equal(Xs[n], inp.x[s][t].cpu()), f"X row {r} of rank {o}"
        if len(pad):
            pt = torch.as_tensor(pad, device=X.device)
            assert not X[pt].any().item(), f"padding rows of X, rank {o}"
            assert not Y[pt].any().item(), f"padding rows of Y must be exactly 0, rank {o}"
        if len(sel):
            want = O.buffer_row_outputs(plan, xs, wg, wu, wd, o, sel)
            got = f64(Y[torch.as_tensor(sel, device=Y.device)])
            assert_close(got, want, f"Y rank {o}")
            for r, y in zip(sel.tolist(), want):
                ycache[(o, r)] = y
    # Combine: receive rows are exact copies of the owner's Y rows.
    for o in range(W):
        Y = layer.rank_field(capi.MOE_RANK_Y, o)
        for b in range(len(plan.band_expert[o])):
            dst = int(plan.band_dst[o][b])
            if dst == o:
                continue
            v, r0 = int(plan.band_valid[o][b]), int(plan.band_dst_row[o][b])
            assert torch.equal(layer.recv[dst][r0:r0 + v], Y[b * wl.tb_M:b * wl.tb_M + v]), \
                f"combine copy of band {b} of rank {o}"
    # Scale: per token sum over its k experts, evaluated expert by expert.
    picks = {}
    for s_ in range(W):
        toks = np.arange(T) if sample is None else np.sort(
            rng.choice(T, size=min(sample, T), replace=False))
        picks[s_] = toks
    need = {}
    for s_, toks in picks.items():
        for t in toks.tolist():
            for j in range(wl.topk):
                need.setdefault(int(ids[s_, t, j]), []).append((s_, t, j))
    yv = {}
    for e in sorted(need):
        o, li = divmod(e, wl.L)
        rows = np.stack([xs[s_][t] for s_, t, _ in need[e]])
        ys = O.expert_ffn(rows, wg[o][li], wu[o][li], wd[o][li])
        for key, y in zip(need[e], ys):
            yv[key] = y
    for s_, toks in picks.items():
        got = f64(layer.out[s_][torch.as_tensor(toks, device=layer.out[s_].device)])
        want = np.zeros_like(got)
        for n, t in enumerate(toks.tolist()):
            for j in range(wl.topk):
                want[n] += w[s_, t, j] * yv[(s_, t, j)]
        assert_close(got, want, f"out rank {s_}")


class _LazyExperts:
    """Per-expert float64 copies of one rank's weight tensor, made on first use."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.cache = {}

    def __getitem__(self, li):
        if li not in self.cache:
            if len(self.cache) > 2:
                self.cache.clear()
            self.cache[li] = f64(self.t[li])
        return self.cache[li]


def inputs_for(wl):
    return make_inputs(wl, device="cuda")

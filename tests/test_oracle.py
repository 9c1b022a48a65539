"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU is needed. Every check here is independent of the oracle's own code:
hand-derived values of the worked example (tests/golden), closed forms
printed on the pages, invariants the method guarantees, special cases that
reduce to textbook values, and brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def random_ids(rng, W, L, T, k, p=None):
    """k distinct experts per token; optional popularity p over the E experts."""
    E = W * L
    ids = np.zeros((W, T, k), dtype=np.int64)
    for s in range(W):
        for t in range(T):
            ids[s, t] = rng.choice(E, size=k, replace=False, p=p)
    return ids


# ---------------------------------------------------------------- gate

def test_route_closed_form_probabilities_and_ties():
    # logits (0, ln3, ln3, 0): partition sum 1+3+3+1 = 8.
    lg = np.array([[[0.0, math.log(3.0), math.log(3.0), 0.0]]], dtype=np.float32)
    ids, w = O.route(lg, 2)
    assert ids[0, 0].tolist() == [1, 2]          # equal logits: lower id first
    np.testing.assert_allclose(w[0, 0], [3 / 8, 3 / 8], rtol=1e-6)
    ids, w = O.route(lg, 3)
    assert ids[0, 0].tolist() == [1, 2, 0]        # 0 and 3 tie; 0 wins
    np.testing.assert_allclose(w[0, 0], [3 / 8, 3 / 8, 1 / 8], rtol=1e-6)
    # equal logits: uniform probabilities 1/E, ids in ascending order
    ids, w = O.route(np.zeros((1, 1, 5), np.float32), 5)
    assert ids[0, 0].tolist() == [0, 1, 2, 3, 4]
    np.testing.assert_allclose(w[0, 0], [0.2] * 5, rtol=1e-12)


def test_route_brute_force_and_forced_ids():
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((3, 7, 6)).astype(np.float32)
    lg[0, 0, 2] = lg[0, 0, 4]  # a tie
    ids, w = O.route(lg, 3)
    for s in range(3):
        for t in range(7):
            row = [float(v) for v in lg[s, t]]
            want = sorted(range(6), key=lambda e: (-row[e], e))[:3]
            assert ids[s, t].tolist() == want
            z = sum(math.exp(v) for v in row)
            assert abs(w[s, t].sum() - sum(math.exp(row[e]) for e in want) / z) < 1e-12
    assert (np.diff(w, axis=-1) <= 0).all()
    forced = np.array([[[5, 0]]])
    ids, w = O.route(lg[:1, :1], 2, forced_ids=forced)
    assert ids.tolist() == [[[5, 0]]]
    assert w[0, 0, 0] < 1 and w[0, 0, 1] < 1


def test_gate_logits_operand_roles_and_brute_force():
    rng = np.random.default_rng(7)
    # Square router, token c = unit vector e_c: score of expert e is w_router[e][c]
    # (a transposed router would give w_router[c][e]).
    wr = rng.standard_normal((6, 6))
    x = np.eye(6)[None]
    lg = O.gate_logits(x, wr)
    assert lg.shape == (1, 6, 6)
    for c in range(6):
        for e in range(6):
            assert lg[0, c, e] == wr[e, c]
    # Tiny non-square case against an exactly rounded sum.
    x = rng.standard_normal((2, 3, 5))
    wr = rng.standard_normal((4, 5))
    lg = O.gate_logits(x, wr)
    assert lg.shape == (2, 3, 4)
    for s in range(2):
        for t in range(3):
            for e in range(4):
                assert abs(lg[s, t, e] - math.fsum(x[s, t, c] * wr[e, c] for c in range(5))) < 1e-12


def test_gate_closed_form_routing():
    # One token (1, 0); router column 0 = (0, ln3, ln3, 0): the scores of the
    # closed-form routing case above, whatever column 1 holds.
    wr = np.array([[0.0, 5.0], [math.log(3.0), -2.0], [math.log(3.0), 7.0], [0.0, 1.0]])
    ids, w = O.gate(np.array([[[1.0, 0.0]]]), wr, 2)
    assert ids[0, 0].tolist() == [1, 2]
    np.testing.assert_allclose(w[0, 0], [3 / 8, 3 / 8], rtol=1e-12)
    # The identity router routes each token to its own largest entries.
    x = np.array([[[0.5, -1.0, 2.0, 0.25], [3.0, 3.0, -4.0, 1.0]]])
    ids, _ = O.gate(x, np.eye(4), 2)
    assert ids[0].tolist() == [[2, 0], [0, 1]]
    # Prescribed ids keep the probabilities of the computed scores.
    ids, w = O.gate(np.array([[[1.0, 0.0]]]), wr, 2, forced_ids=np.array([[[3, 1]]]))
    assert ids[0, 0].tolist() == [3, 1]
    np.testing.assert_allclose(w[0, 0], [1 / 8, 3 / 8], rtol=1e-12)


# ---------------------------------------------------------------- FFN

def test_silu_special_values():
    assert O.silu(0.0) == 0.0
    # sigma(ln 3) = 3/4, sigma(-ln 3) = 1/4
    np.testing.assert_allclose(O.silu(math.log(3)), 0.75 * math.log(3), rtol=1e-14)
    np.testing.assert_allclose(O.silu(-math.log(3)), -0.25 * math.log(3), rtol=1e-14)
    z = np.linspace(-8, 8, 33)
    np.testing.assert_allclose(O.silu(z) - O.silu(-z), z, atol=1e-12)  # odd part is z/2 * 2
    assert O.silu(40.0) == pytest.approx(40.0) and abs(O.silu(-40.0)) < 1e-15


def test_ffn_closed_form_and_operand_roles():
    l3 = math.log(3)
    x = np.array([[l3]])
    one, two = np.array([[1.0]]), np.array([[2.0]])
    # gate = x, up = 2x:  SiLU(ln3) * 2 ln3 = 1.5 (ln3)^2
    ffn = lambda *a: O.expert_ffn(*a, round_hidden=False)
    np.testing.assert_allclose(ffn(x, one, two, one), [[1.5 * l3 * l3]], rtol=1e-14)
    # gate and up swapped: SiLU(2 ln3) * ln3 = 2 ln3 * (9/10) * ln3 = 1.8 (ln3)^2
    np.testing.assert_allclose(ffn(x, two, one, one), [[1.8 * l3 * l3]], rtol=1e-14)
    # rectangular operands in nn.Linear layout: D=2, F=3
    x = np.array([[l3, 0.0]])
    wg = np.array([[1.0, 5.0], [0.0, 1.0], [-1.0, 7.0]])  # g = (ln3, 0, -ln3)
    wu = np.array([[1.0, 9.0], [1.0, 0.0], [1.0, 2.0]])   # u = (ln3, ln3, ln3)
    wd = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])     # y = (a0, a2)
    a0 = 0.75 * l3 * l3
    a2 = -0.25 * l3 * l3
    np.testing.assert_allclose(ffn(x, wg, wu, wd), [[a0, a2]], rtol=1e-14)
    # zero input gives zero output; output is linear in W_down
    assert not O.expert_ffn(np.zeros((2, 2)), wg, wu, wd).any()
    rng = np.random.default_rng(0)
    xr = rng.standard_normal((4, 2))
    np.testing.assert_allclose(O.expert_ffn(xr, wg, wu, 3 * wd), 3 * O.expert_ffn(xr, wg, wu, wd))


def test_round_bf16_matches_the_library_conversion():
    """round_bf16 against torch's float32 -> bfloat16 conversion (round to nearest even)."""
    import torch
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                        [0.0, -0.0, 1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9,
                         3.0 * 2.0 ** 100, -65504.0]])
    want = torch.tensor(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_bf16(v.astype(np.float32)), want)
    assert O.round_bf16(1.0 + 2.0 ** -8) == 1.0            # tie -> even (mantissa 0)
    assert O.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie -> even (up)


def test_ffn_rounds_the_hidden_activation():
    # x = 2, all weights 1: g = u = 2, h = 2 * 2 * sigma(2) = 3.5232..., bf16 -> 3.515625
    x = np.array([[2.0]])
    one = np.array([[1.0]])
    h = 4.0 / (1.0 + np.exp(-2.0))
    assert abs(h - 3.52318831) < 1e-8
    assert O.expert_ffn(x, one, one, one)[0, 0] == 3.515625
    assert O.expert_ffn(x, one, one, 2 * one)[0, 0] == 7.03125
    np.testing.assert_allclose(O.expert_ffn(x, one, one, one, round_hidden=False), [[h]], rtol=1e-15)


def test_ffn_both_roundings_from_one_hidden_activation():
    """expert_ffn_both gives the two readings of the hidden activation: the hand value
    above (h = 3.5232 rounds to 3.515625) and the unrounded h, and on random rectangular
    operands the same rows as expert_ffn with and without the rounding."""
    x, one = np.array([[2.0]]), np.array([[1.0]])
    r, u = O.expert_ffn_both(x, one, one, 2 * one)
    assert r[0, 0] == 7.03125
    np.testing.assert_allclose(u, [[8.0 / (1.0 + np.exp(-2.0))]], rtol=1e-15)
    rng = np.random.default_rng(4)
    xr = rng.standard_normal((5, 3))
    wg, wu, wd = (rng.standard_normal(s) for s in ((4, 3), (4, 3), (3, 4)))
    r, u = O.expert_ffn_both(xr, wg, wu, wd)
    np.testing.assert_allclose(r, O.expert_ffn(xr, wg, wu, wd), rtol=0, atol=1e-13)
    np.testing.assert_allclose(u, O.expert_ffn(xr, wg, wu, wd, round_hidden=False), rtol=0,
                               atol=1e-13)
    assert np.abs(r - u).max() > 0  # the rounding is applied to one of them only


# ---------------------------------------------------------------- layout / schedule / plan

def test_worked_example_figure2():
    g = _load("fig2_worked_example.json")
    p = O.build_plan(np.array(g["ids"]), g["W"], g["L"], g["tb"], g["mgb"])
    r = g["rank"]
    T = g["T"]

    def as_pairs(xs):
        return [None if v < 0 else [int(v) // T, int(v) % T] for v in xs]

    xs = p.xsrc[r]
    assert as_pairs(xs[0:24]) == g["expert2_xsrc_as_rank_token"]
    assert as_pairs(xs[24:48]) == g["expert3_xsrc_as_rank_token"]
    for e in ("2", "3"):
        assert p.expert_start[int(e)] == g["expert_start"][e]
        assert p.pad[int(e)] == g["pad"][e]
        assert p.nrb[int(e)] == g["nrb"][e]
    assert p.band_expert[r].tolist() == g["band_expert"]
    assert p.band_dst[r].tolist() == g["band_dst"]
    assert p.band_valid[r].tolist() == g["band_valid"]
    assert p.band_dst_row[r].tolist() == g["band_dst_row"]
    assert p.S[r].tolist() == g["S"]
    assert p.n_remote[r] == g["n_remote"]
    assert [list(x) for x in p.segments[r]] == g["segments"]
    assert p.recv_rows.tolist() == g["recv_rows"]


def test_rule_ii_tie_keeps_the_lower_local_index_first():
    """Rule (ii) with equal remote loads (the pages leave the order of a tie open; the
    reading taken is the lower local index first, as in the balanced A100-like layer).
    Hand-derived: W = 2, L = 2, tb_M = 2; every rank sends token 0 to experts 0 and 2
    and token 1 to experts 1 and 3. On rank 0, expert 0 holds one remote row (rank 1's
    token 0) padded to a 2-row band, then its one local row: bands 0 (remote, to rank
    1) and 1 (local); expert 1 likewise at rows 4..7: bands 2 and 3. Both experts have
    one remote band, so S = [0, 2, 1, 3]: both remote bands, expert 0's first, then the
    local bands in local-index order."""
    ids = np.array([[[0, 2], [1, 3]], [[0, 2], [1, 3]]])
    p = O.build_plan(ids, 2, 2, 2, 1)
    for r in range(2):
        assert p.nrb[2 * r:2 * r + 2].tolist() == [1, 1]
        assert p.band_dst[r].tolist() == [1 - r, r, 1 - r, r]
        assert p.S[r].tolist() == [0, 2, 1, 3]
        assert p.n_remote[r] == 2


def test_padding_bound_closed_forms():
    g = _load("padding_bounds.json")
    for c in g["cases"]:
        W, tb = c["W"], c["tb"]
        assert O.padding_bound(W, tb) == c["bound"]
        # Worst case: every remote rank sends exactly one row to expert 0.
        ids = np.zeros((W, 1, 1), dtype=np.int64)
        p = O.build_plan(ids, W, 1, tb)
        assert p.pad[0] == c["bound"]
        assert p.nrb[0] == W - 1
        if "rows" in c:
            assert round(100.0 * c["bound"] / c["rows"], 2) == c["percent"]


CASES = [
    # W, L, T, k, tb, mgb, skew
    (2, 1, 5, 1, 4, 1, None),
    (3, 2, 9, 2, 4, 2, None),
    (4, 2, 16, 2, 8, 1, None),
    (4, 2, 33, 3, 4, 3, None),
    (4, 3, 20, 12, 4, 2, None),      # k = E: every token to every expert
    (5, 2, 1, 2, 2, 1, None),        # T = 1
    (4, 4, 64, 1, 16, 2, "zipf"),    # skew, many empty experts
    (8, 2, 12, 4, 4, 4, None),
    (2, 3, 40, 2, 8, 2, "zipf"),
]


def _check_invariants(ids, p):
    W, L, T, k, tb = p.W, p.L, p.T, p.k, p.tb
    E = W * L
    bound = O.padding_bound(W, tb)
    remote_assign = 0
    for s in range(W):
        for t in range(T):
            for j in range(k):
                if ids[s, t, j] // L != s:
                    remote_assign += 1
    sent = 0
    for o in range(W):
        xs = p.xsrc[o]
        nbands = len(xs) // tb
        assert len(xs) % tb == 0
        assert len(p.S[o]) == nbands and sorted(p.S[o].tolist()) == list(range(nbands))
        for b in range(nbands):
            rows = xs[b * tb:(b + 1) * tb]
            e = int(p.band_expert[o][b])
            assert e // L == o
            v = int(p.band_valid[o][b])
            # valid rows are a prefix of the band; the rest are zero rows
            assert 1 <= v <= tb
            assert (rows[:v] >= 0).all() and (rows[v:] < 0).all()
            # exactly one owner rank per band: every valid row comes from band_dst
            srcs = {int(x) // T for x in rows[:v]}
            assert srcs == {int(p.band_dst[o][b])}
            # the band's tokens really route to its expert, in ascending token order
            toks = [int(x) % T for x in rows[:v]]
            assert toks == sorted(toks)
            for t in toks:
                assert e in ids[int(p.band_dst[o][b]), t].tolist()
            if p.band_dst[o][b] != o:
                sent += v
        # per expert: pad bound, zero rows = pad + tail
        for li in range(L):
            e = o * L + li
            lo, n = int(p.expert_start[e]), int(p.rows_alloc[e])
            assert p.pad[e] <= bound
            zero = int((xs[lo:lo + n] < 0).sum())
            assert zero == p.pad[e] + (p.rows_alloc[e] - p.rows[e])
            assert p.rows_alloc[e] - p.rows[e] < tb
            assert p.cnt[e].sum() == n - zero
        # S: remote bands first; experts in non-increasing remote-band order
        R = int(p.n_remote[o])
        dst = p.band_dst[o][p.S[o]]
        assert (dst[:R] != o).all() and (dst[R:] == o).all()
        exps = p.band_expert[o][p.S[o][:R]].tolist()
        runs = [exps[0]] if exps else []
        for a, b_ in zip(exps, exps[1:]):
            if b_ != a:
                assert b_ not in runs
                runs.append(b_)
        nr = [int(p.nrb[e]) for e in runs]
        assert nr == sorted(nr, reverse=True)
        # segments tile the remote prefix, in order
        segs = p.segments[o]
        pos = 0
        for i, (first, nbs) in enumerate(segs):
            assert first == pos and nbs >= 1
            if i == 0 or i == len(segs) - 1:
                assert nbs == 1
            assert nbs <= max(1, p.mgb)
            bands = p.S[o][first:first + nbs].tolist()
            assert bands == list(range(bands[0], bands[0] + nbs))
            keys = {(int(p.band_expert[o][b]), int(p.band_dst[o][b])) for b in bands}
            assert len(keys) == 1
            pos += nbs
        assert pos == R
    assert sent == remote_assign
    # receive buffers: exact disjoint cover; scale map is a bijection
    for s in range(W):
        cover = np.zeros(int(p.recv_rows[s]), dtype=np.int64)
        owner_row = {}
        for o in range(W):
            for b in range(len(p.band_expert[o])):
                if p.band_dst[o][b] == s and o != s:
                    r0, v = int(p.band_dst_row[o][b]), int(p.band_valid[o][b])
                    cover[r0:r0 + v] += 1
                    for i in range(v):
                        owner_row[r0 + i] = (o, b * tb + i)
        assert (cover == 1).all()
        seen = set()
        for t in range(T):
            for j in range(k):
                e = int(ids[s, t, j])
                src = int(p.src[s, t, j])
                if e // L != s:
                    assert src >= 0 and src not in seen
                    seen.add(src)
                    o, row = owner_row[src]
                    assert o == e // L and int(p.xsrc[o][row]) == s * T + t
                    li = int(np.searchsorted([p.expert_start[o * L + q] for q in range(L)], row, "right")) - 1
                    assert o * L + li == e
                else:
                    row = -src - 1
                    assert int(p.xsrc[s][row]) == s * T + t
                    li = int(np.searchsorted([p.expert_start[s * L + q] for q in range(L)], row, "right")) - 1
                    assert s * L + li == e
        assert len(seen) == p.recv_rows[s]
    assert p.cnt.sum() == W * T * k and E == p.E


@pytest.mark.parametrize("case", CASES)
def test_plan_invariants_random(case):
    W, L, T, k, tb, mgb, skew = case
    rng = np.random.default_rng(hash(case) % 2**32)
    p_e = None
    if skew == "zipf":
        w = np.arange(1, W * L + 1, dtype=np.float64) ** -1.2
        p_e = w / w.sum()
    for _ in range(3):
        ids = random_ids(rng, W, L, T, k, p_e)
        _check_invariants(ids, O.build_plan(ids, W, L, tb, mgb))


def test_plan_degenerate_routings():
    W, L, T, tb = 4, 2, 10, 4
    # all local: every token goes to its own rank's experts -> nothing is sent
    ids = np.array([[[2 * s, 2 * s + 1]] * T for s in range(W)])
    p = O.build_plan(ids, W, L, tb)
    assert p.recv_rows.tolist() == [0] * W and (p.n_remote == 0).all()
    assert all(len(s) == 0 for s in p.segments) and p.pad.sum() == 0
    _check_invariants(ids, p)
    # all remote, groups exactly one band: no padding at all
    ids = np.array([[[(2 * ((s + 1) % W)), (2 * ((s + 1) % W)) + 1]] * 8 for s in range(W)])
    p = O.build_plan(ids, W, L, tb)
    assert p.pad.sum() == 0 and (p.rows == p.rows_alloc).all()
    _check_invariants(ids, p)
    # rejected routings
    with pytest.raises(ValueError):
        O.build_plan(np.array([[[0, 0]]]), 1, 2, 4)
    with pytest.raises(ValueError):
        O.build_plan(np.array([[[0, 9]]]), 1, 2, 4)


# ---------------------------------------------------------------- end to end, brute force

def _direct(x, ids, w, wg, wu, wd, L):
    """sum_j w_j FFN_{e_j}(x) per token, with plain loops and no layout at all."""
    W, T, k = ids.shape
    D = x[0].shape[1]
    out = [np.zeros((T, D)) for _ in range(W)]
    for s in range(W):
        for t in range(T):
            for j in range(k):
                o, li = divmod(int(ids[s, t, j]), L)
                xv = x[s][t].astype(np.float64)
                g = wg[o][li].astype(np.float64) @ xv
                u = wu[o][li].astype(np.float64) @ xv
                a = np.array([gi / (1.0 + math.exp(-gi)) for gi in g]) * u
                a = O.round_bf16(a)  # the second GEMM's operand is bf16
                out[s][t] += w[s, t, j] * (wd[o][li].astype(np.float64) @ a)
    return out


def _rand_weights(rng, W, L, D, F):
    wg = [rng.standard_normal((L, F, D)) * 0.3 for _ in range(W)]
    wu = [rng.standard_normal((L, F, D)) * 0.3 for _ in range(W)]
    wd = [rng.standard_normal((L, D, F)) * 0.3 for _ in range(W)]
    return wg, wu, wd


@pytest.mark.parametrize("W,L,T,k,tb,mgb", [(4, 2, 12, 2, 4, 2), (3, 3, 7, 3, 2, 1), (2, 2, 9, 4, 8, 3)])
def test_forward_matches_direct_sum(W, L, T, k, tb, mgb):
    rng = np.random.default_rng(7)
    D, F = 6, 5
    x = [rng.standard_normal((T, D)) for _ in range(W)]
    wg, wu, wd = _rand_weights(rng, W, L, D, F)
    lg = rng.standard_normal((W, T, W * L)).astype(np.float32)
    r = O.forward(x, wg, wu, wd, lg, k, L, tb, mgb)
    want = _direct(x, r["ids"], r["w"], wg, wu, wd, L)
    for s in range(W):
        np.testing.assert_allclose(r["out"][s], want[s], atol=1e-10, rtol=0)
    # padding rows of every buffer produce exact zeros
    for o in range(W):
        assert not r["Y"][o][r["plan"].xsrc[o] < 0].any()


def test_special_cases_reduce_to_plain_ffn():
    rng = np.random.default_rng(3)
    W, L, T, D, F, tb = 3, 2, 5, 4, 3, 4
    x = [rng.standard_normal((T, D)) for _ in range(W)]
    wg, wu, wd = _rand_weights(rng, W, L, D, F)
    # k = 1 with weight 1: out is one expert's plain FFN
    ids = rng.integers(0, W * L, size=(W, T, 1))
    p = O.build_plan(ids, W, L, tb)
    Y = [O.rank_outputs(p, x, wg, wu, wd, o) for o in range(W)]
    out = O.scale(p, np.ones((W, T, 1)), O.combine(p, Y), Y)
    for s in range(W):
        for t in range(T):
            o, li = divmod(int(ids[s, t, 0]), L)
            want = O.expert_ffn(x[s][t][None], wg[o][li], wu[o][li], wd[o][li])[0]
            np.testing.assert_allclose(out[s][t], want, atol=1e-12)
    # one-hot weights select a slot; weights enter linearly
    ids2 = np.stack([ids[..., 0], (ids[..., 0] + 1) % (W * L)], axis=-1)
    p2 = O.build_plan(ids2, W, L, tb)
    Y2 = [O.rank_outputs(p2, x, wg, wu, wd, o) for o in range(W)]
    R2 = O.combine(p2, Y2)
    a = O.scale(p2, np.stack([np.ones((W, T)), np.zeros((W, T))], -1), R2, Y2)
    b = O.scale(p2, np.stack([np.zeros((W, T)), np.ones((W, T))], -1), R2, Y2)
    ab = O.scale(p2, np.full((W, T, 2), 0.5), R2, Y2)
    for s in range(W):
        np.testing.assert_allclose(a[s], out[s], atol=1e-12)
        np.testing.assert_allclose(ab[s], 0.5 * (a[s] + b[s]), atol=1e-12)


def test_buffer_row_outputs_matches_whole_buffer():
    rng = np.random.default_rng(5)
    W, L, T, D, F, tb = 3, 2, 8, 4, 3, 4
    x = [rng.standard_normal((T, D)) for _ in range(W)]
    wg, wu, wd = _rand_weights(rng, W, L, D, F)
    ids = random_ids(rng, W, L, T, 2)
    p = O.build_plan(ids, W, L, tb)
    for o in range(W):
        Y = O.rank_outputs(p, x, wg, wu, wd, o)
        rows = list(range(0, int(p.rank_rows[o]), 3))
        np.testing.assert_allclose(O.buffer_row_outputs(p, x, wg, wu, wd, o, rows), Y[rows], atol=1e-12)


def test_receive_order_example():
    g = _load("recv_order_example.json")
    p = O.build_plan(np.array(g["ids"]), g["W"], g["L"], g["tb"], g["mgb"])
    for e, off in g["recv_off_rank0"].items():
        assert p.recv_off[int(e), 0] == off
    assert p.recv_rows.tolist() == g["recv_rows"]
    assert p.src[0].tolist() == g["scale_map_rank0"]
    _check_invariants(np.array(g["ids"]), p)


def test_bf16_ulp_helper_used_by_the_gpu_tolerance():
    """The element bound of the GPU parity tests: bf16 spacing at a few exact points."""
    from tests.parity import bf16_ulp
    assert bf16_ulp(1.0) == 2.0 ** -7 and bf16_ulp(1.99) == 2.0 ** -7
    assert bf16_ulp(4.0) == 2.0 ** -5 and bf16_ulp(-8.5) == 2.0 ** -4
    assert bf16_ulp(2.56) == 2.0 ** -6 < 2e-2 < bf16_ulp(4.0)

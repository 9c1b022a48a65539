"""CPU oracle of the tile-signalled MoE expert-combine path.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg (and its reference arm) import this module. The product path
(the CUDA library and its Python binding) never calls it, and this module
imports nothing from the product.

It is deliberately plain: numpy, float64, Python loops over small index sets.
No blocking, no fusion, no reordering beyond what the method's definition states.

Sources, cited by page title and section:
  [TileMoE] zhongzhuzhou.org notes "MoE 计算-通信细粒度重叠：用 Tile 级信号把
            All-to-All 藏在 GEMM 背后" on "Fine-grained Computation-Communication
            Overlap via Tile-level Signaling and Scheduling for Mixture-of-Experts".
            The sections are the notes' own: 2.1 (MoE layer), 2.2 (five-step
            distributed forward), 4.2 (remote-owner-aligned row layout), 4.4
            (remote-first schedule and Algorithm 1), 4.5 (combine plan), 4.3/6
            (padding bound), 5.2 (row bands and segments, Figure 3b).
  [Perseus] papercache.org summary of "Eliminating Hidden Serialization in
            Multi-Node Megakernel Communication", section 4.1 and Algorithm 1
            (decoupled signalling: one fence per destination group).

Readings where the pages are silent or ambiguous (each is also listed in the
design notes of the repository):
  R1  Expert e is owned by rank e // L. Figure 2b of [TileMoE] puts expert 2 on
      rank 1 with W=4, L=2, which fixes this contiguous placement.
  R2  Inside one group, rows keep ascending source-token order. A token reaches
      an expert at most once, so this is a total order.
  R3  Only remote groups are zero-padded to a multiple of tb_M ([TileMoE]
      Algorithm 1 pads r' != r_self only). The local group is not padded. The
      expert's block is then rounded up to a multiple of tb_M; those tail rows
      are an allocation detail and are not counted as padding.
  R4  Expert blocks sit in local-index order inside the owner's buffer.
  R5  Rule (ii) sorts by remote row-band count, descending; ties keep the lower
      local index first.
  R6  The receive buffer of rank s is ordered by sender rank o (ascending,
      o != s), then local expert index, then the group's row order.
  R7  Segments ([TileMoE] 5.2) are cut per rank over the remote prefix of S.
      The first and the last remote band are single-band segments. Middle bands
      merge greedily, up to mgb consecutive entries of S, and never cross an
      (expert, destination) group. Each segment is then one contiguous copy.
  R8  Gate weights are the softmax probabilities over all E experts at the
      chosen ids. They are not renormalised over the top-k. Top-k compares the
      fp32 logits; equal logits go to the lower expert id, and the output is
      in descending order.
  R9  The expert FFN is SiLU-gated: y = W_down (SiLU(W_gate x) * (W_up x)), with
      SiLU(z) = z / (1 + exp(-z)). Padding rows are defined to produce 0.
  R10 The padding bound (W-1)(tb_M-1) of [TileMoE] 4.3/6 holds per (rank, local
      expert). The worked example of 11.10 applies it to one expert's tokens.
  R11 Both expert GEMMs take half-precision operands ([TileMoE] 7.1: CUTLASS
      GEMMs; 7.6: outputs agree with the serial baseline up to FP16 rounding).
      Here the operands are bf16, so the hidden activation h = SiLU(g) * u, being
      the second GEMM's input, is rounded to bf16 (to nearest, ties to even)
      before W_down is applied. Everything else is float64.
  R14 The gate ([TileMoE] 2.1: a small gating network; 2.2 step 1: every rank
      gates its own tokens) is one bias-free linear layer whose weights
      w_router [E, D] every rank holds alike: logits_s[t] = w_router x_s[t]. Its
      operands are half precision like the expert GEMMs' (R11); the scores are
      float64 sums of the bf16 values here.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "softmax", "silu", "round_bf16", "route", "gate_logits", "gate", "Plan", "build_plan",
    "expert_ffn", "expert_ffn_both", "layout_rows", "rank_outputs", "buffer_row_outputs",
    "combine", "scale", "forward", "padding_bound",
]


# --------------------------------------------------------------------------
# Gate ([TileMoE] 2.1; 2.2 step 1)
# --------------------------------------------------------------------------

def softmax(logits) -> np.ndarray:
    """Softmax over the last axis, in float64."""
    z = np.asarray(logits, dtype=np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=-1, keepdims=True)


def route(logits, k: int, forced_ids=None):
    """Gate: softmax over the E experts, then the k most probable ones.

    logits: [W, T, E] (fp32 values). forced_ids: optional [W, T, k] prescribed
    routing (balanced or skewed workloads); the weights are then the gate
    probabilities at those ids. Returns (ids int64 [W,T,k], w float64 [W,T,k]).
    Reading R8: the decision compares logits (softmax is strictly increasing),
    equal logits go to the lower expert id, and the weights are not renormalised.
    """
    lg = np.asarray(logits, dtype=np.float64)
    p = softmax(lg)
    if forced_ids is None:
        # Stable sort of the negated logits: descending value, ties by ascending id.
        order = np.argsort(-lg, axis=-1, kind="stable")
        ids = order[..., :k]
    else:
        ids = np.asarray(forced_ids, dtype=np.int64)
    w = np.take_along_axis(p, ids, axis=-1)
    return ids.astype(np.int64), w


def gate_logits(x, w_router) -> np.ndarray:
    """Gate scores of every token: logits[s][t][e] = sum_c x[s][t][c] * w_router[e][c].

    x: [W, T, D] token rows; w_router: [E, D] (nn.Linear layout), shared by the
    ranks (reading R14). float64 sums of the given values.
    """
    xs = np.asarray(x, dtype=np.float64)
    wr = np.asarray(w_router, dtype=np.float64)
    return xs @ wr.T


def gate(x, w_router, k: int, forced_ids=None):
    """Routing from the token rows: the gate scores (gate_logits), then route()."""
    return route(gate_logits(x, w_router), k, forced_ids)


# --------------------------------------------------------------------------
# Layout, schedule and combine plan ([TileMoE] 4.2, 4.4 Algorithm 1, 4.5, 5.2)
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Plan:
    W: int
    L: int
    k: int
    T: int
    tb: int
    mgb: int
    members: list        # members[e][s]: source tokens t (ascending) of group (e, s)
    cnt: np.ndarray      # [E, W] group sizes |G_s| for expert e
    group_start: np.ndarray  # [E, W] first row of group (e, s) inside expert e's block
    group_rows: np.ndarray   # [E, W] padded group size
    rows: np.ndarray         # [E] sum of padded group sizes
    rows_alloc: np.ndarray   # [E] rows rounded up to tb
    expert_start: np.ndarray  # [E] first row of expert e's block in its owner's buffer
    rank_rows: np.ndarray     # [W] rows of each owner's buffer
    nb: np.ndarray            # [E] row bands of expert e
    nrb: np.ndarray           # [E] remote row bands of expert e
    pad: np.ndarray           # [E] zero rows added to remote groups of expert e
    band_expert: list         # [W] arrays over rank-local band ids
    band_dst: list
    band_valid: list
    band_dst_row: list        # row in the destination's receive buffer, -1 for local
    S: list                   # [W] schedule: rank-local band ids
    n_remote: np.ndarray      # [W] length of the remote prefix of S
    segments: list            # [W] list of (first S index, number of bands)
    recv_off: np.ndarray      # [E, W] first receive row of (e, s) at rank s, -1 if local
    recv_rows: np.ndarray     # [W] rows received by each rank
    xsrc: list                # [W] per buffer row: source token s*T+t, or -1 for a zero row
    src: np.ndarray           # [W, T, k] scale map (see scale())

    @property
    def E(self) -> int:
        return self.W * self.L

    def owner(self, e: int) -> int:
        return e // self.L  # reading R1

    def group_order(self, e: int) -> list:
        o = self.owner(e)
        return [s for s in range(self.W) if s != o] + [o]


def _ceil_to(n: int, m: int) -> int:
    return -(-n // m) * m


def build_plan(ids, W: int, L: int, tb: int, mgb: int = 1) -> Plan:
    """Expert problem construction and combine plan for every logical rank.

    ids: [W, T, k] expert ids per token (distinct within a token).
    """
    ids = np.asarray(ids, dtype=np.int64)
    if ids.ndim != 3 or ids.shape[0] != W:
        raise ValueError("ids must be [W, T, k]")
    _, T, k = ids.shape
    E = W * L
    if tb <= 0 or mgb <= 0:
        raise ValueError("tb and mgb must be positive")
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    for s in range(W):
        for t in range(T):
            if len(set(ids[s, t].tolist())) != k:
                raise ValueError(f"token ({s},{t}) repeats an expert")

    # Groups G_s of every expert, rows in ascending token order (reading R2).
    members = [[[] for _ in range(W)] for _ in range(E)]
    for s in range(W):
        for t in range(T):
            for j in range(k):
                members[ids[s, t, j]][s].append(t)
    cnt = np.array([[len(members[e][s]) for s in range(W)] for e in range(E)], dtype=np.int64)

    def owner(e):
        return e // L

    def order(e):
        o = owner(e)
        return [s for s in range(W) if s != o] + [o]

    # Remote-owner-aligned layout X_e ([TileMoE] 4.2, Algorithm 1 first half).
    group_start = np.zeros((E, W), dtype=np.int64)
    group_rows = np.zeros((E, W), dtype=np.int64)
    rows = np.zeros(E, dtype=np.int64)
    rows_alloc = np.zeros(E, dtype=np.int64)
    pad = np.zeros(E, dtype=np.int64)
    for e in range(E):
        off = 0
        for s in order(e):
            c = int(cnt[e, s])
            padded = c if s == owner(e) else _ceil_to(c, tb)  # reading R3
            group_start[e, s] = off
            group_rows[e, s] = padded
            pad[e] += padded - c
            off += padded
        rows[e] = off
        rows_alloc[e] = _ceil_to(off, tb)

    expert_start = np.zeros(E, dtype=np.int64)
    rank_rows = np.zeros(W, dtype=np.int64)
    for o in range(W):
        off = 0
        for li in range(L):  # reading R4
            e = o * L + li
            expert_start[e] = off
            off += rows_alloc[e]
        rank_rows[o] = off

    nb = rows_alloc // tb
    nrb = np.array([sum(int(group_rows[e, s]) for s in range(W) if s != owner(e)) // tb
                    for e in range(E)], dtype=np.int64)

    # Receive offsets (reading R6).
    recv_off = np.full((E, W), -1, dtype=np.int64)
    recv_rows = np.zeros(W, dtype=np.int64)
    for s in range(W):
        off = 0
        for o in range(W):
            if o == s:
                continue
            for li in range(L):
                e = o * L + li
                recv_off[e, s] = off
                off += cnt[e, s]
        recv_rows[s] = off

    # Combine plan per row band ([TileMoE] 4.5): destination, remote row, valid rows.
    band_expert, band_dst, band_valid, band_dst_row = [], [], [], []
    for o in range(W):
        n = int(rank_rows[o]) // tb
        be = np.full(n, -1, dtype=np.int64)
        bd = np.full(n, -1, dtype=np.int64)
        bv = np.zeros(n, dtype=np.int64)
        br = np.full(n, -1, dtype=np.int64)
        for li in range(L):
            e = o * L + li
            for b in range(int(nb[e])):
                r = b * tb  # first row of the band inside expert e's block
                dst = None
                for s in order(e):
                    lo = int(group_start[e, s])
                    if lo <= r < lo + int(group_rows[e, s]):
                        dst = s
                        break
                if dst is None:
                    raise AssertionError("band starts outside every group")
                gb = (int(expert_start[e]) + r) // tb
                be[gb] = e
                bd[gb] = dst
                bv[gb] = min(tb, int(group_start[e, dst]) + int(cnt[e, dst]) - r)
                if dst != o:
                    br[gb] = int(recv_off[e, dst]) + (r - int(group_start[e, dst]))
        band_expert.append(be)
        band_dst.append(bd)
        band_valid.append(bv)
        band_dst_row.append(br)

    # Remote-first schedule S ([TileMoE] 4.4 rules (i), (ii); Algorithm 1 second half).
    S, n_remote = [], np.zeros(W, dtype=np.int64)
    for o in range(W):
        local = [o * L + li for li in range(L)]
        by_remote = sorted(local, key=lambda e: (-int(nrb[e]), e))  # reading R5
        seq = []
        for e in by_remote:
            b0 = int(expert_start[e]) // tb
            seq += [b0 + b for b in range(int(nrb[e]))]
        n_remote[o] = len(seq)
        for e in local:
            b0 = int(expert_start[e]) // tb
            seq += [b0 + b for b in range(int(nrb[e]), int(nb[e]))]
        S.append(np.array(seq, dtype=np.int64))

    # Segments over the remote prefix of S ([TileMoE] 5.2, Figure 3b; reading R7).
    segments = []
    for o in range(W):
        R = int(n_remote[o])
        segs = []
        if R >= 1:
            segs.append([0, 1])
        prev_key = None
        for i in range(1, R - 1):
            b = int(S[o][i])
            key = (int(band_expert[o][b]), int(band_dst[o][b]))
            cur = segs[-1]
            if i > 1 and key == prev_key and cur[1] < mgb:
                cur[1] += 1
            else:
                segs.append([i, 1])
            prev_key = key
        if R >= 2:
            segs.append([R - 1, 1])
        segments.append([tuple(x) for x in segs])

    # Source of every row of each owner's buffer: token id s*T+t, or -1 (zero row).
    xsrc = []
    for o in range(W):
        xs = np.full(int(rank_rows[o]), -1, dtype=np.int64)
        for li in range(L):
            e = o * L + li
            for s in range(W):
                base = int(expert_start[e]) + int(group_start[e, s])
                for i, t in enumerate(members[e][s]):
                    xs[base + i] = s * T + t
        xsrc.append(xs)

    # Scale map: for token (s, t) slot j, src >= 0 is a row of rank s's receive
    # buffer (remote expert); src < 0 encodes row -src-1 of rank s's own expert
    # output buffer (local expert).
    pos = [[{t: i for i, t in enumerate(members[e][s])} for s in range(W)] for e in range(E)]
    src = np.zeros((W, T, k), dtype=np.int64)
    for s in range(W):
        for t in range(T):
            for j in range(k):
                e = int(ids[s, t, j])
                i = pos[e][s][t]
                if owner(e) != s:
                    src[s, t, j] = int(recv_off[e, s]) + i
                else:
                    src[s, t, j] = -(int(expert_start[e]) + int(group_start[e, s]) + i) - 1

    return Plan(W, L, k, T, tb, mgb, members, cnt, group_start, group_rows, rows, rows_alloc,
                expert_start, rank_rows, nb, nrb, pad, band_expert, band_dst, band_valid,
                band_dst_row, S, n_remote, segments, recv_off, recv_rows, xsrc, src)


# --------------------------------------------------------------------------
# Expert FFN ([TileMoE] 2.1, 2.3; reading R9)
# --------------------------------------------------------------------------

def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def round_bf16(v) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even (returned as float64).

    bf16 keeps the top 16 bits of an IEEE float32: round the float64 value to
    float32 first (exact for every bf16 value), then round the low 16 bits of the
    float32 pattern to nearest with ties to even. Inf and NaN are not expected.
    """
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    bits = (bits + 0x7FFF + lsb) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def _hidden(xrows, w_gate, w_up) -> np.ndarray:
    """h = SiLU(W_gate x) * (W_up x) for each row x, float64, not rounded."""
    x = np.asarray(xrows, dtype=np.float64)
    g = x @ np.asarray(w_gate, dtype=np.float64).T
    u = x @ np.asarray(w_up, dtype=np.float64).T
    return silu(g) * u


def expert_ffn(xrows, w_gate, w_up, w_down, round_hidden: bool = True) -> np.ndarray:
    """y = W_down h, h = SiLU(W_gate x) * (W_up x), for each row x.

    xrows [n, D]; w_gate, w_up [F, D]; w_down [D, F] (nn.Linear layout).
    float64 throughout; h is rounded to bf16 before the second GEMM (reading R11)
    unless round_hidden is False.
    """
    a = _hidden(xrows, w_gate, w_up)
    if round_hidden:
        a = round_bf16(a)
    return a @ np.asarray(w_down, dtype=np.float64).T


def expert_ffn_both(xrows, w_gate, w_up, w_down):
    """(expert_ffn with h rounded to bf16, expert_ffn with h unrounded) of the same
    rows, computing h once: the half-precision reading R11 and the plain
    float64 FFN side by side."""
    a = _hidden(xrows, w_gate, w_up)
    wd = np.asarray(w_down, dtype=np.float64).T
    return round_bf16(a) @ wd, a @ wd


def layout_rows(plan: Plan, x, o: int) -> np.ndarray:
    """Owner o's input buffer X (all experts' blocks): token rows, zero elsewhere.

    x: list of W arrays [T, D].
    """
    D = np.asarray(x[0]).shape[1]
    out = np.zeros((int(plan.rank_rows[o]), D), dtype=np.float64)
    xs = plan.xsrc[o]
    for r in np.nonzero(xs >= 0)[0]:
        s, t = divmod(int(xs[r]), plan.T)
        out[r] = np.asarray(x[s][t], dtype=np.float64)
    return out


def rank_outputs(plan: Plan, x, w_gate, w_up, w_down, o: int) -> np.ndarray:
    """Expert outputs Y of owner o's whole buffer; padding and tail rows are 0."""
    X = layout_rows(plan, x, o)
    Y = np.zeros_like(X)
    xs = plan.xsrc[o]
    for li in range(plan.L):
        e = o * plan.L + li
        lo = int(plan.expert_start[e])
        hi = lo + int(plan.rows_alloc[e])
        r = np.arange(lo, hi)[xs[lo:hi] >= 0]
        if len(r):
            Y[r] = expert_ffn(X[r], w_gate[o][li], w_up[o][li], w_down[o][li])
    return Y


def buffer_row_outputs(plan: Plan, x, w_gate, w_up, w_down, o: int, rows) -> np.ndarray:
    """Expert outputs for selected rows of owner o's buffer (0 for zero rows).

    Evaluates only the requested rows, so full-size workloads can be sampled.
    w_gate/w_up/w_down[o] may be any indexable of per-expert [F, D] / [D, F]
    arrays (for example a lazy view that copies one expert at a time).
    """
    rows = np.asarray(list(rows), dtype=np.int64)
    D = np.asarray(x[0]).shape[1]
    out = np.zeros((len(rows), D), dtype=np.float64)
    xs = plan.xsrc[o]
    starts = np.array([int(plan.expert_start[o * plan.L + li]) for li in range(plan.L)])
    for n, r in enumerate(rows):
        if xs[r] < 0:
            continue
        li = int(np.searchsorted(starts, r, side="right")) - 1
        s, t = divmod(int(xs[r]), plan.T)
        xr = np.asarray(x[s][t], dtype=np.float64)[None, :]
        out[n] = expert_ffn(xr, w_gate[o][li], w_up[o][li], w_down[o][li])[0]
    return out


# --------------------------------------------------------------------------
# Combine ([TileMoE] 2.2 step 4, 4.5, 5.2) and scale ([TileMoE] 2.2 step 5)
# --------------------------------------------------------------------------

def combine(plan: Plan, Y: list) -> list:
    """Receive buffers: every remote band's valid rows land at its planned offset."""
    D = Y[0].shape[1]
    recv = [np.zeros((int(plan.recv_rows[s]), D), dtype=np.float64) for s in range(plan.W)]
    for o in range(plan.W):
        for b in range(len(plan.band_expert[o])):
            dst = int(plan.band_dst[o][b])
            if dst == o or plan.band_expert[o][b] < 0:
                continue
            v = int(plan.band_valid[o][b])
            r0 = int(plan.band_dst_row[o][b])
            recv[dst][r0:r0 + v] = Y[o][b * plan.tb:b * plan.tb + v]
    return recv


def scale(plan: Plan, w, recv: list, Y: list) -> list:
    """out_s[t] = sum_j w[s,t,j] * (expert e_j's output for token (s,t))."""
    w = np.asarray(w, dtype=np.float64)
    D = Y[0].shape[1]
    out = []
    for s in range(plan.W):
        o_s = np.zeros((plan.T, D), dtype=np.float64)
        for t in range(plan.T):
            for j in range(plan.k):
                src = int(plan.src[s, t, j])
                row = recv[s][src] if src >= 0 else Y[s][-src - 1]
                o_s[t] += w[s, t, j] * row
        out.append(o_s)
    return out


def forward(x, w_gate, w_up, w_down, logits, k: int, L: int, tb: int, mgb: int = 1,
            forced_ids=None):
    """The whole path for small cases: route, plan, FFN, combine, scale."""
    W = len(x)
    ids, w = route(logits, k, forced_ids)
    plan = build_plan(ids, W, L, tb, mgb)
    Y = [rank_outputs(plan, x, w_gate, w_up, w_down, o) for o in range(W)]
    recv = combine(plan, Y)
    out = scale(plan, w, recv, Y)
    return dict(ids=ids, w=w, plan=plan, Y=Y, recv=recv, out=out)


def padding_bound(W: int, tb: int) -> int:
    """Worst-case zero rows per (rank, local expert): (W-1)(tb_M-1) ([TileMoE] 4.3, 6, 11.10)."""
    return (W - 1) * (tb - 1)

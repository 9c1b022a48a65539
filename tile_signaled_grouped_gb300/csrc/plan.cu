// Expert problem construction and combine plan on the GPU.
//
// TileMoE notes (zhongzhuzhou.org, "Fine-grained Computation-Communication
// Overlap via Tile-level Signaling and Scheduling for Mixture-of-Experts"):
//   section 4.2  remote-owner-aligned row layout X_e (rows grouped by the rank
//                that owns the token, remote groups first, each zero-padded to
//                a multiple of tb_M, the local group last),
//   section 4.4  remote-first schedule S (rule i: remote bands first; rule ii:
//                experts with more remote row bands first) - Algorithm 1,
//   section 4.5  combine plan (per band: destination, remote row, valid rows),
//   section 5.2  segments (first and last one band, middle ones merge mgb bands).
//
// Stable order inside a group (ascending source token) comes from one bit per
// (expert, source rank, token) and a popcount prefix, so every array is
// bit-exact and independent of thread timing. No size ever travels to the
// host: later kernels read the totals from device memory.
#include "moe_common.cuh"

namespace moe {
namespace {

// The two per-rank / single-CTA plan kernels run with 256 threads and size their
// shared arrays to the layer (L experts per rank, W ranks), so that they fit on an SM
// beside a running producer CTA (which leaves about 26K registers and 4 KB of
// shared memory): the plan of one batch can then overlap the FFN of another.
constexpr int kPlanThreads = 256;

__device__ __forceinline__ int roundup(int a, int m) { return (a + m - 1) / m * m; }

__device__ __forceinline__ bool slot_valid(const int32_t* row, int j, int E) {
  const int e = row[j];
  if (e < 0 || e >= E) return false;
  for (int q = 0; q < j; ++q)
    if (row[q] == e) return false;
  return true;
}

// One bit per (expert, source rank, token).
__global__ void plan_bitmap_kernel(DevPlan p, const int32_t* __restrict__ ids) {
  const Dims d = p.d;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(p.a[PA_BITMAP]);
  uint32_t* status = reinterpret_cast<uint32_t*>(p.a[PA_STATUS]);
  const int ntok = d.W * d.T;
  for (int tok = blockIdx.x * blockDim.x + threadIdx.x; tok < ntok;
       tok += gridDim.x * blockDim.x) {
    const int s = tok / d.T, t = tok % d.T;
    const int32_t* row = ids + (size_t)tok * d.k;
    for (int j = 0; j < d.k; ++j) {
      if (!slot_valid(row, j, d.E)) {
        report_error(status, MOE_DEV_ROUTING, (uint32_t)tok);
        continue;
      }
      const int e = row[j];
      atomicOr(&bitmap[((size_t)e * d.W + s) * d.TW + (t >> 5)], 1u << (t & 31));
    }
  }
}

// One warp per (expert, source rank): group size and the popcount prefix of every word.
__global__ void plan_count_kernel(DevPlan p) {
  const Dims d = p.d;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= d.E * d.W) return;
  const uint32_t* bitmap = reinterpret_cast<const uint32_t*>(p.a[PA_BITMAP]);
  int32_t* wpre = p.a[PA_WPRE];
  const size_t base = (size_t)gw * d.TW;
  int carry = 0;
  for (int w0 = 0; w0 < d.TW; w0 += 32) {
    const int wi = w0 + lane;
    const int c = wi < d.TW ? __popc(bitmap[base + wi]) : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (wi < d.TW) wpre[base + wi] = carry + x - c;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) p.a[PA_CNT][gw] = carry;  // [E][W]
}

__device__ __forceinline__ int block_incl_max_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max(x, y);
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < nw ? scratch[lane] : INT_MIN;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s = max(s, y);
    }
    if (lane < nw) scratch[lane] = s;
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  const int r = wid > 0 ? max(scratch[wid - 1], x) : x;
  *total = scratch[32];
  __syncthreads();
  return r;
}

// Largest index q in [0, n) with a[q] <= v (a non-decreasing, a[0] <= v).
__device__ __forceinline__ int last_le(const int* a, int n, int v) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Dynamic shared memory of plan_rank_kernel: 7 arrays of L ints, 2 of L * W.
__host__ __device__ inline size_t rank_smem_bytes(int L, int W) {
  return (size_t)(7 * L + 2 * L * W) * sizeof(int);
}

// One CTA per owner rank o: layout X_e, schedule S, combine plan, segments.
__global__ void __launch_bounds__(kPlanThreads) plan_rank_kernel(DevPlan p) {
  const Dims d = p.d;
  const int o = blockIdx.x;
  const int tid = threadIdx.x, nt = blockDim.x;
  extern __shared__ int s_dyn[];
  int* s_rows_alloc = s_dyn;
  int* s_nb = s_rows_alloc + d.L;
  int* s_nrb = s_nb + d.L;
  int* s_estart = s_nrb + d.L;
  int* s_order = s_estart + d.L;
  int* s_rpre = s_order + d.L;
  int* s_lpre = s_rpre + d.L;
  int* s_gs = s_lpre + d.L;         // [L][W]
  int* s_cnt = s_gs + d.L * d.W;    // [L][W]
  __shared__ int scratch[33];
  __shared__ int s_NB, s_R;

  const int32_t* cnt = p.a[PA_CNT];
  int32_t* group_start = p.a[PA_GROUP_START];
  int32_t* recv_off = p.a[PA_RECV_OFF];

  // 1. Per local expert: groups in the order (remote ranks ascending, then o).
  for (int li = tid; li < d.L; li += nt) {
    const int e = o * d.L + li;
    int off = 0, remote_rows = 0;
    for (int q = 0; q < d.W; ++q) {
      const int s = q < d.W - 1 ? (q < o ? q : q + 1) : o;
      const int c = cnt[e * d.W + s];
      const int padded = s == o ? c : roundup(c, d.tb);
      group_start[e * d.W + s] = off;
      s_gs[li * d.W + s] = off;
      s_cnt[li * d.W + s] = c;
      off += padded;
      if (s != o) remote_rows += padded;
    }
    const int ra = roundup(off, d.tb);
    s_rows_alloc[li] = ra;
    s_nb[li] = ra / d.tb;
    s_nrb[li] = remote_rows / d.tb;
    p.a[PA_ROWS_ALLOC][e] = ra;
    p.a[PA_NB][e] = ra / d.tb;
    p.a[PA_NRB][e] = remote_rows / d.tb;
    // Receive offsets: sender rank ascending, then local expert, then row order.
    for (int s = 0; s < d.W; ++s) {
      if (s == o) {
        recv_off[e * d.W + s] = -1;
        continue;
      }
      int base = 0;
      for (int o2 = 0; o2 < o; ++o2) {
        if (o2 == s) continue;
        for (int l2 = 0; l2 < d.L; ++l2) base += cnt[(o2 * d.L + l2) * d.W + s];
      }
      for (int l2 = 0; l2 < li; ++l2) base += cnt[(o * d.L + l2) * d.W + s];
      recv_off[e * d.W + s] = base;
    }
  }
  __syncthreads();

  // 2. Expert placement, rank totals, rule (ii) order.
  if (tid == 0) {
    int acc = 0, R = 0;
    for (int li = 0; li < d.L; ++li) {
      s_estart[li] = acc;
      p.a[PA_EXPERT_START][o * d.L + li] = acc;
      acc += s_rows_alloc[li];
      R += s_nrb[li];
    }
    s_NB = acc / d.tb;
    s_R = R;
    p.a[PA_RANK_ROWS][o] = acc;
    p.a[PA_RANK_NB][o] = acc / d.tb;
    p.a[PA_RANK_NREMOTE][o] = R;
    int recv = 0;
    for (int o2 = 0; o2 < d.W; ++o2) {
      if (o2 == o) continue;
      for (int l2 = 0; l2 < d.L; ++l2) recv += cnt[(o2 * d.L + l2) * d.W + o];
    }
    p.a[PA_RECV_ROWS][o] = recv;
  }
  for (int li = tid; li < d.L; li += nt) {
    int pos = 0;
    for (int l2 = 0; l2 < d.L; ++l2)
      pos += (s_nrb[l2] > s_nrb[li]) || (s_nrb[l2] == s_nrb[li] && l2 < li);
    s_order[pos] = li;
  }
  __syncthreads();
  if (tid == 0) {
    int rp = 0;
    for (int q = 0; q < d.L; ++q) {
      s_rpre[q] = rp;
      rp += s_nrb[s_order[q]];
    }
    int lp = rp;
    for (int li = 0; li < d.L; ++li) {
      s_lpre[li] = lp;
      lp += s_nb[li] - s_nrb[li];
    }
  }
  __syncthreads();
  const int NB = s_NB, R = s_R;
  int32_t* S = p.a[PA_SCHED] + (size_t)o * d.NBM;

  // 3. Schedule S: remote bands by rule (ii), then local bands by local index.
  for (int i = tid; i < NB; i += nt) {
    int b;
    if (i < R) {
      const int q = last_le(s_rpre, d.L, i);
      const int li = s_order[q];
      b = s_estart[li] / d.tb + (i - s_rpre[q]);
    } else {
      const int li = last_le(s_lpre, d.L, i);
      b = s_estart[li] / d.tb + s_nrb[li] + (i - s_lpre[li]);
    }
    S[i] = b;
  }

  // 4. Combine plan per band.
  int32_t* b_exp = p.a[PA_BAND_EXPERT] + (size_t)o * d.NBM;
  int32_t* b_dst = p.a[PA_BAND_DST] + (size_t)o * d.NBM;
  int32_t* b_val = p.a[PA_BAND_VALID] + (size_t)o * d.NBM;
  int32_t* b_row = p.a[PA_BAND_DST_ROW] + (size_t)o * d.NBM;
  for (int b = tid; b < NB; b += nt) {
    const int li = last_le(s_estart, d.L, b * d.tb);
    const int e = o * d.L + li;
    const int r = b * d.tb - s_estart[li];
    int dst = o, gs = 0, c = 0;
    for (int q = 0; q < d.W; ++q) {
      const int s = q < d.W - 1 ? (q < o ? q : q + 1) : o;
      const int g0 = s_gs[li * d.W + s], cc = s_cnt[li * d.W + s];
      const int padded = s == o ? cc : roundup(cc, d.tb);
      if (r >= g0 && r < g0 + padded) {
        dst = s;
        gs = g0;
        c = cc;
        break;
      }
    }
    b_exp[b] = e;
    b_dst[b] = dst;
    b_val[b] = min(d.tb, gs + c - r);
    b_row[b] = dst != o ? recv_off[e * d.W + dst] + (r - gs) : -1;
  }
  // X rows start as zero rows; the scatter kernel marks the token rows.
  int32_t* xsrc = p.a[PA_XSRC] + (size_t)o * d.RM;
  for (int r = tid; r < d.RM; r += nt) xsrc[r] = -1;
  __syncthreads();

  // 5. Segments over the remote prefix of S.
  int32_t* seg_first = p.a[PA_SEG_FIRST] + (size_t)o * d.NBM;
  int32_t* seg_nb = p.a[PA_SEG_NB] + (size_t)o * d.NBM;
  int32_t* seg_gidx = p.a[PA_SEG_GIDX] + (size_t)o * d.NBM;
  int run_carry = -1, seg_carry = 0;
  for (int base = 0; base < R; base += nt) {
    const int i = base + tid;
    const bool in = i < R;
    const bool middle = in && i >= 1 && i <= R - 2;
    bool head = false;
    if (middle) {
      if (i == 1) {
        head = true;
      } else {
        const int b1 = S[i], b0 = S[i - 1];
        head = (b_exp[b1] != b_exp[b0]) || (b_dst[b1] != b_dst[b0]);
      }
    }
    int tmax;
    int runstart = block_incl_max_scan(head ? i : -1, scratch, &tmax);
    runstart = max(runstart, run_carry);
    run_carry = max(run_carry, tmax);
    const bool start = in && (i == 0 || i == R - 1 || (middle && (i - runstart) % d.mgb == 0));
    int tot;
    const int idx = seg_carry + block_excl_scan(start ? 1 : 0, scratch, &tot);
    if (start) seg_first[idx] = i;
    seg_carry += tot;
  }
  const int nseg = seg_carry;
  __syncthreads();
  for (int j = tid; j < nseg; j += nt)
    seg_nb[j] = (j + 1 < nseg ? seg_first[j + 1] : R) - seg_first[j];
  // Index of each segment inside its (sender o, destination) group, in S order.
  for (int dst = 0; dst < d.W; ++dst) {
    int carry = 0;
    for (int base = 0; base < nseg; base += nt) {
      const int j = base + tid;
      const bool mine = j < nseg && b_dst[S[seg_first[j]]] == dst;
      int tot;
      const int idx = carry + block_excl_scan(mine ? 1 : 0, scratch, &tot);
      if (mine) seg_gidx[j] = idx;
      carry += tot;
    }
    if (tid == 0) p.a[PA_GROUP_NSEG][o * d.W + dst] = carry;
  }
  if (tid == 0) p.a[PA_RANK_NSEG][o] = nseg;
}

// One thread per (token, slot): row of the token inside its owner's X and the scale map.
__global__ void plan_scatter_kernel(DevPlan p, const int32_t* __restrict__ ids) {
  const Dims d = p.d;
  const uint32_t* bitmap = reinterpret_cast<const uint32_t*>(p.a[PA_BITMAP]);
  const int n = d.W * d.T * d.k;
  for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < n; a += gridDim.x * blockDim.x) {
    const int tok = a / d.k, j = a % d.k;
    const int s = tok / d.T, t = tok % d.T;
    const int32_t* row = ids + (size_t)tok * d.k;
    if (!slot_valid(row, j, d.E)) {
      p.a[PA_SCALE_SRC][a] = INT_MIN;
      continue;
    }
    const int e = row[j];
    const int o = e / d.L;
    const size_t wi = ((size_t)e * d.W + s) * d.TW + (t >> 5);
    const int pos = p.a[PA_WPRE][wi] + __popc(bitmap[wi] & ((1u << (t & 31)) - 1u));
    const int xr = p.a[PA_EXPERT_START][e] + p.a[PA_GROUP_START][e * d.W + s] + pos;
    p.a[PA_XSRC][(size_t)o * d.RM + xr] = s * d.T + t;
    p.a[PA_SCALE_SRC][a] = o != s ? p.a[PA_RECV_OFF][e * d.W + s] + pos : -xr - 1;
  }
}

// Single CTA: the producer's tile order and its scheduling units, and the consumer's
// segment order (following the tile order). Each rank's remote tiles, then its local
// tiles (its S order), are cut into scheduling units of at most kTileGroup tiles
// that keep each expert's run of tiles (S keeps an expert's remote tiles, and its
// local tiles, contiguous) inside one unit wherever it fits: the runs are packed in
// order, a new unit opened when the next run does not fit, and a run longer than
// kTileGroup cut into near-equal parts of even length (CTA pairs stay together). A
// unit's GEMM1 reads each weight tile of its experts once (its tasks are hidden-
// column-major), so a run split over two units would read its expert's weights
// twice. The units of the remote phase come first, round-robin over the ranks (unit
// 0 of every rank, then unit 1, ...), then those of the local phase.
__global__ void __launch_bounds__(kPlanThreads) plan_order_kernel(DevPlan p) {
  const Dims d = p.d;
  const int tid = threadIdx.x, nt = blockDim.x;
  __shared__ int scratch[33];
  __shared__ int s_nt[MOE_MAX_RANKS], s_rt[MOE_MAX_RANKS], s_lt[MOE_MAX_RANKS];
  __shared__ int s_rem[MOE_MAX_RANKS], s_nb[MOE_MAX_RANKS], s_nseg[MOE_MAX_RANKS];
  __shared__ int s_nu[MOE_MAX_RANKS][2], s_NU;
  __shared__ int s_ecnt[2 * 1024];  // tiles of each (expert, phase); E <= 1024
  const int W = d.W, tb = d.tb;
  const int P = tb >= kTileM ? tb / kTileM : 1;
  int32_t* rank_tiles = p.a[PA_RANK_TILES];  // [W][NMM] rank-local row of each tile, S order

  if (tid < W) {
    s_rem[tid] = p.a[PA_RANK_NREMOTE][tid];
    s_nb[tid] = p.a[PA_RANK_NB][tid];
    s_nseg[tid] = p.a[PA_RANK_NSEG][tid];
  }
  __syncthreads();

  // 1. Each rank's tile sequence in S order.
  for (int o = 0; o < W; ++o) {
    const int32_t* S = p.a[PA_SCHED] + (size_t)o * d.NBM;
    const int32_t* estart = p.a[PA_EXPERT_START] + o * d.L;
    const int32_t* bexp = p.a[PA_BAND_EXPERT] + (size_t)o * d.NBM;
    int32_t* rt = rank_tiles + (size_t)o * d.NMM;
    const int NB = s_nb[o], R = s_rem[o];
    if (tb >= kTileM) {
      for (int q = tid; q < NB * P; q += nt) rt[q] = S[q / P] * tb + (q % P) * kTileM;
      if (tid == 0) {
        s_nt[o] = NB * P;
        s_rt[o] = R * P;
      }
    } else {
      // tb = 64: one tile per pair of bands (2i, 2i+1) of an expert, placed where
      // the pair's first band sits in S (it always comes first).
      int carry = 0, carry_r = 0;
      for (int base = 0; base < NB; base += nt) {
        const int i = base + tid;
        bool emit = false;
        int b = 0;
        if (i < NB) {
          b = S[i];
          const int e = bexp[b];
          const int bl = b - estart[e - o * d.L] / tb;
          emit = (bl & 1) == 0;
        }
        int tot;
        const int q = carry + block_excl_scan(emit ? 1 : 0, scratch, &tot);
        if (emit) rt[q] = b * tb;
        int totr;
        block_excl_scan((emit && i < R) ? 1 : 0, scratch, &totr);
        carry += tot;
        carry_r += totr;
      }
      if (tid == 0) {
        s_nt[o] = carry;
        s_rt[o] = carry_r;
      }
    }
    __syncthreads();
  }
  if (tid < W) s_lt[tid] = s_nt[tid] - s_rt[tid];
  __syncthreads();

  int NM = 0;
  for (int o = 0; o < W; ++o) NM += s_nt[o];

  // 2. Scheduling units. Tiles of each (expert, phase), then one thread per (rank,
  // phase) walks its expert runs and records where each unit starts.
  const int cap = unit_cap(d);
  int32_t* ustart = p.a[PA_UNIT_TMP];       // [W][2][cap] first tile of each unit in its phase
  int32_t* ugpos = ustart + 2 * W * cap;    // [W][2][cap] its position in the tile order
  for (int i = tid; i < 2 * d.E; i += nt) s_ecnt[i] = 0;
  __syncthreads();
  for (int o = 0; o < W; ++o) {
    const int32_t* rt = rank_tiles + (size_t)o * d.NMM;
    const int32_t* bexp = p.a[PA_BAND_EXPERT] + (size_t)o * d.NBM;
    for (int q = tid; q < s_nt[o]; q += nt)
      atomicAdd(&s_ecnt[2 * bexp[rt[q] / tb] + (q < s_rt[o] ? 0 : 1)], 1);
  }
  __syncthreads();
  if (tid < 2 * W) {
    const int o = tid >> 1, ph = tid & 1;
    const int q0 = ph ? s_rt[o] : 0, q1 = ph ? s_nt[o] : s_rt[o];
    const int32_t* rt = rank_tiles + (size_t)o * d.NMM;
    const int32_t* bexp = p.a[PA_BAND_EXPERT] + (size_t)o * d.NBM;
    int32_t* us = ustart + (size_t)(o * 2 + ph) * cap;
    int nu = 0, open = -1;  // phase-local first tile of the open unit (-1: none)
    for (int q = q0; q < q1;) {
      const int len = s_ecnt[2 * bexp[rt[q] / tb] + ph];  // this expert's run (>= 1)
      const int qq = q - q0;
      if (len > kTileGroup) {
        const int n = (len + kTileGroup - 1) / kTileGroup;
        const int part = 2 * ((len + 2 * n - 1) / (2 * n));  // even, at most kTileGroup
        for (int i = 0; i < n && i * part < len; ++i) us[nu++] = qq + i * part;
        open = -1;
      } else if (open < 0 || qq + len - open > kTileGroup) {
        us[nu++] = qq;
        open = qq;
      }
      q += len;
    }
    s_nu[o][ph] = nu;
  }
  __syncthreads();
  // Positions: the remote units round-robin over the ranks, then the local ones.
  if (tid == 0) {
    int u = 0, pos = 0;
    for (int ph = 0; ph < 2; ++ph) {
      int maxnu = 0;
      for (int o = 0; o < W; ++o) maxnu = max(maxnu, s_nu[o][ph]);
      for (int j = 0; j < maxnu; ++j)
        for (int o = 0; o < W; ++o) {
          const int nuo = s_nu[o][ph];
          if (j >= nuo) continue;
          const int32_t* us = ustart + (size_t)(o * 2 + ph) * cap;
          const int tiles = ph ? s_lt[o] : s_rt[o];
          ugpos[(size_t)(o * 2 + ph) * cap + j] = pos;
          p.a[PA_UNIT_BEGIN][u++] = pos;
          pos += (j + 1 < nuo ? us[j + 1] : tiles) - us[j];
        }
    }
    p.a[PA_UNIT_BEGIN][u] = NM;
    p.a[PA_TOTALS][0] = NM;
    p.a[PA_TOTALS][2] = u;
    s_NU = u;
  }
  __syncthreads();
  const int NU = s_NU;

  // 2a. Global tile order and the tile of every band: a tile's unit is the last one
  // starting at or before it in its phase.
  for (int o = 0; o < W; ++o) {
    const int32_t* rt = rank_tiles + (size_t)o * d.NMM;
    const int32_t* bexp = p.a[PA_BAND_EXPERT] + (size_t)o * d.NBM;
    const int32_t* estart = p.a[PA_EXPERT_START] + o * d.L;
    const int32_t* ralloc = p.a[PA_ROWS_ALLOC] + o * d.L;
    int32_t* btile = p.a[PA_BAND_TILE] + (size_t)o * d.NBM;
    for (int q = tid; q < s_nt[o]; q += nt) {
      const int ph = q < s_rt[o] ? 0 : 1;
      const int qq = ph ? q - s_rt[o] : q;
      const int32_t* us = ustart + (size_t)(o * 2 + ph) * cap;
      int lo = 0, hi = s_nu[o][ph] - 1;  // us[0] == 0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (us[mid] <= qq) lo = mid; else hi = mid - 1;
      }
      const int pos = ugpos[(size_t)(o * 2 + ph) * cap + lo] + (qq - us[lo]);
      const int row = rt[q];
      const int b = row / tb;
      const int e = bexp[b];
      p.a[PA_TILE_ROW][pos] = (o << 24) | row;
      p.a[PA_TILE_EXPERT][pos] = e;
      if (tb >= kTileM) {
        if (row % tb == 0) btile[b] = pos;
      } else {
        btile[b] = pos;
        const int li = e - o * d.L;
        if ((b + 1) * tb < estart[li] + ralloc[li]) btile[b + 1] = pos;
      }
    }
  }
  __syncthreads();

  // 2b. CTA pairs of the pair producer: tiles j and j^1 of one expert (rows
  // estart + 128 j of its block) form a pair, listed where the earlier of the
  // two sits in the tile order, as one 16-byte record. The pair units are the
  // tile units: unit u holds the pairs whose earlier tile lies in tile unit u.
  {
    int32_t* heads_before = rank_tiles;  // reuse: pairs listed before each tile position
    int carry_p = 0;
    for (int base = 0; base < NM; base += nt) {
      const int pos = base + tid;
      int partner = -1;
      bool head = false;
      int4 rec;
      if (pos < NM) {
        const int tr = p.a[PA_TILE_ROW][pos];
        const int o = tr >> 24, row = tr & 0xFFFFFF;
        const int e = p.a[PA_TILE_EXPERT][pos];
        const int es = p.a[PA_EXPERT_START][e], ra = p.a[PA_ROWS_ALLOC][e];
        const int prow = es + (((row - es) / kTileM) ^ 1) * kTileM;
        if (prow < es + ra)
          partner = p.a[PA_BAND_TILE][(size_t)o * d.NBM + prow / tb] +
                    (tb > kTileM ? (prow % tb) / kTileM : 0);
        head = partner < 0 || pos < partner;
        // Record of the pair: first tile, partner, first tile's (rank, row), and
        // the local expert with one bit saying whether the partner's rows lie
        // 128 above (else 128 below) the first tile's.
        rec = make_int4(pos, partner, tr, (e - o * d.L) | (partner >= 0 && prow < row ? 1 << 16 : 0));
      }
      int tot;
      const int idx = carry_p + block_excl_scan(head ? 1 : 0, scratch, &tot);
      if (pos < NM) {
        heads_before[pos] = idx;
        if (head) reinterpret_cast<int4*>(p.a[PA_PAIR])[idx] = rec;
      }
      carry_p += tot;
    }
    __syncthreads();
    for (int u = tid; u <= NU; u += nt) {
      const int b = p.a[PA_UNIT_BEGIN][u];
      p.a[PA_PAIR_UNIT_BEGIN][u] = b < NM ? heads_before[b] : carry_p;
    }
    if (tid == 0) p.a[PA_TOTALS][5] = carry_p;
    __syncthreads();
    // Runs of one expert inside each pair unit (a unit's pairs keep its tiles' expert
    // runs in order): the producer takes a unit's GEMM1 tasks run by run.
    const int4* prec = reinterpret_cast<const int4*>(p.a[PA_PAIR]);
    for (int u = tid; u < NU; u += nt) {
      const int ub = p.a[PA_PAIR_UNIT_BEGIN][u], ue = p.a[PA_PAIR_UNIT_BEGIN][u + 1];
      int rs = ub;
      for (int q = ub; q <= ue; ++q) {
        if (q == ue || (q > rs && (prec[q].w & 0xFFFF) != (prec[rs].w & 0xFFFF))) {
          for (int i = rs; i < q; ++i) p.a[PA_PAIR_RUN][i] = (rs - ub) | ((q - rs) << 16);
          rs = q;
        }
      }
    }
    __syncthreads();
  }

  // 3. Consumer order: segments sorted by the tile of their first band.
  int32_t* slot = p.a[PA_RANK_TILES];  // reuse: [2 * NM] slots, -1 = empty
  __syncthreads();
  for (int i = tid; i < 2 * NM; i += nt) slot[i] = -1;
  __syncthreads();
  for (int o = 0; o < W; ++o) {
    const int32_t* S = p.a[PA_SCHED] + (size_t)o * d.NBM;
    const int32_t* sf = p.a[PA_SEG_FIRST] + (size_t)o * d.NBM;
    const int32_t* btile = p.a[PA_BAND_TILE] + (size_t)o * d.NBM;
    for (int j = tid; j < s_nseg[o]; j += nt) {
      const int b = S[sf[j]];
      const int pos = btile[b];
      const int row = p.a[PA_TILE_ROW][pos] & 0xFFFFFF;
      slot[2 * pos + (b * tb != row ? 1 : 0)] = o * d.NBM + j;
    }
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < 2 * NM; base += nt) {
    const int i = base + tid;
    const int v = i < 2 * NM ? slot[i] : -1;
    int tot;
    const int idx = carry + block_excl_scan(v >= 0 ? 1 : 0, scratch, &tot);
    if (v >= 0) p.a[PA_SEG_ORDER][idx] = v;
    carry += tot;
  }
  const int nsegs = carry;
  for (int g = tid; g < W * W; g += nt) p.a[PA_GROUP_NCHUNK][g] = 0;
  __syncthreads();

  // 4. One record per segment in consumer order: source band, destination, rows,
  // and its range of copy chunks (rpc rows each) in the global chunk sequence; and
  // the record of every chunk.
  int chunk_carry = 0;
  for (int base = 0; base < nsegs; base += nt) {
    const int idx = base + tid;
    int nch = 0;
    int rec[kSegRec] = {};
    if (idx < nsegs) {
      const int code = p.a[PA_SEG_ORDER][idx];
      const int o = code / d.NBM, j = code % d.NBM;
      const size_t rb = (size_t)o * d.NBM;
      const int nb = p.a[PA_SEG_NB][rb + j];
      const int b0 = p.a[PA_SCHED][rb + p.a[PA_SEG_FIRST][rb + j]];
      const int dst = p.a[PA_BAND_DST][rb + b0];
      const int vrows = (nb - 1) * tb + p.a[PA_BAND_VALID][rb + b0 + nb - 1];
      nch = (vrows + d.rpc - 1) / d.rpc;
      rec[0] = o;
      rec[1] = dst;
      rec[2] = b0;
      rec[3] = nb;
      rec[4] = vrows;
      rec[5] = p.a[PA_BAND_DST_ROW][rb + b0];
      rec[7] = nch;
      atomicAdd(&p.a[PA_GROUP_NCHUNK][o * W + dst], nch);
    }
    int tot;
    const int cb = chunk_carry + block_excl_scan(nch, scratch, &tot);
    if (idx < nsegs) {
      rec[6] = cb;
      int32_t* out = p.a[PA_SEG_REC] + (size_t)idx * kSegRec;
#pragma unroll
      for (int q = 0; q < kSegRec; ++q) out[q] = rec[q];
      for (int k = 0; k < nch; ++k) p.a[PA_CHUNK_REC][cb + k] = idx;
    }
    chunk_carry += tot;
  }
  if (tid == 0) {
    p.a[PA_TOTALS][1] = nsegs;
    p.a[PA_TOTALS][4] = chunk_carry;
    int bands = 0;
    for (int o = 0; o < W; ++o) bands += s_nb[o];
    p.a[PA_TOTALS][3] = bands;
  }
}

// Layout gather: X rows of every owner from its tokens' rows, zero rows elsewhere
// (padding, block tails, and up to the next 128-row boundary). One warp per row,
// over the rows that exist (their count is read on the device); a warp reads the
// plan entries of 32 of its rows at once, and each lane keeps up to 8 independent
// 16-byte loads of a row in flight. A row that is to be zero and was
// already zero after the previous gather (PA_XPREV) is left alone: padding-heavy
// layouts keep most of their zero rows from one step to the next.
struct GatherPtrs {
  const __nv_bfloat16* x[MOE_MAX_RANKS];
  __nv_bfloat16* xb[MOE_MAX_RANKS];
};

__global__ void layout_gather_kernel(DevPlan p, const __grid_constant__ GatherPtrs g) {
  const Dims d = p.d;
  const int lane = threadIdx.x & 31;
  int end[MOE_MAX_RANKS];  // cumulative rows to write, per owner
  int total = 0;
#pragma unroll
  for (int o = 0; o < MOE_MAX_RANKS; ++o) {
    if (o < d.W) total += min(d.RM, roundup(p.a[PA_RANK_ROWS][o], kTileM));
    end[o] = total;
  }
  const int n16 = d.D / 8;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  if (threadIdx.x == 0) span_begin(p.span, kSpanGatherStart);
  // A warp takes rows gw, gw + warps, ... in batches of 32: lane j reads the plan
  // entries of the batch's j-th row (one round trip for 32 rows), and the warp then
  // copies or zeroes, one row at a time, only the rows that need it.
  for (int base = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; base < total;
       base += 32 * warps) {
    const int gw = base + lane * warps;
    int o = 0, r = 0, src = -1;
    bool work = false;
    if (gw < total) {
#pragma unroll
      for (int q = 0; q < MOE_MAX_RANKS - 1; ++q) o += (q < d.W - 1 && gw >= end[q]) ? 1 : 0;
      r = gw - (o > 0 ? end[o - 1] : 0);
      const int rows = p.a[PA_RANK_ROWS][o];
      src = r < rows ? p.a[PA_XSRC][(size_t)o * d.RM + r] : -1;
      int32_t* prev = p.a[PA_XPREV] + (size_t)o * d.RM + r;
      const int before = *prev;
      work = !(src < 0 && before == -1);  // else still a zero row
      if (before != src) *prev = src;
    }
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, work);
    while (todo) {
      const int j = __ffs(todo) - 1;
      todo &= todo - 1;
      const int jo = __shfl_sync(0xFFFFFFFFu, o, j);
      const int jr = __shfl_sync(0xFFFFFFFFu, r, j);
      const int jsrc = __shfl_sync(0xFFFFFFFFu, src, j);
      uint4* dst = reinterpret_cast<uint4*>(g.xb[jo] + (size_t)jr * d.D);
      if (jsrc >= 0) {
        const int s = jsrc / d.T, t = jsrc % d.T;
        const uint4* sp = reinterpret_cast<const uint4*>(g.x[s] + (size_t)t * d.D);
        for (int c0 = 0; c0 < n16; c0 += 8 * 32) {
          uint4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < n16) v[u] = __ldg(sp + c);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < n16) dst[c] = v[u];
          }
        }
      } else {
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int c = lane; c < n16; c += 32) dst[c] = z;
      }
    }
  }
  if (p.span != nullptr) {  // the same for the whole grid
    __syncthreads();
    if (threadIdx.x == 0) span_end(p.span, kSpanGatherEnd);
  }
}

}  // namespace

cudaError_t preload_plan() {
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, plan_bitmap_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, plan_count_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, plan_rank_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, plan_scatter_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, plan_order_kernel)) != cudaSuccess) return e;
  return cudaFuncGetAttributes(&fa, layout_gather_kernel);
}

cudaError_t launch_plan(const DevPlan& p, const int32_t* ids, cudaStream_t s, bool marked) {
  const Dims& d = p.d;
  if (!marked) {
    const int ntok = d.W * d.T;
    plan_bitmap_kernel<<<(ntok + 255) / 256, 256, 0, s>>>(p, ids);
  }
  const int warps = d.E * d.W;
  plan_count_kernel<<<(warps * 32 + 255) / 256, 256, 0, s>>>(p);
  plan_rank_kernel<<<d.W, kPlanThreads, rank_smem_bytes(d.L, d.W), s>>>(p);
  const int na = d.W * d.T * d.k;
  plan_scatter_kernel<<<(na + 255) / 256, 256, 0, s>>>(p, ids);
  plan_order_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const DevPlan& p, const __nv_bfloat16* const* x,
                          __nv_bfloat16* const* xbuf, int num_sms, cudaStream_t s) {
  GatherPtrs g{};
  for (int r = 0; r < p.d.W; ++r) {
    g.x[r] = x[r];
    g.xb[r] = xbuf[r];
  }
  layout_gather_kernel<<<num_sms * 16, 256, 0, s>>>(p, g);
  return cudaGetLastError();
}

}  // namespace moe

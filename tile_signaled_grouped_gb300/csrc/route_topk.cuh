// Routing of one token by a warp, by a group of lanes or by one thread: softmax over
// its E gate scores and the top k.
//
// TileMoE notes (zhongzhuzhou.org), section 2.1 and 2.2 step 1: the router turns a
// token's scores into a probability distribution over the E experts and keeps the
// k most probable ones; the gate weights are those probabilities (not renormalised
// over the k). Used by the routing kernel (a warp per token, scores read from
// memory) and by the two gate kernels (scores summed from their K-split partials),
// which also mark each routed token in the plan's bitmap (TokenMark, mark_token).
#pragma once

#include "moe_common.cuh"

namespace moe {

#if defined(__CUDACC__)

// Order-preserving map of a float to an unsigned key (larger float, larger key);
// -0 is taken as +0, so equal values have equal keys.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Compare-exchange of two (score, expert) candidates: afterwards slot i holds the
// one that comes first (larger score, then lower id).
template <int PER>
__device__ __forceinline__ void route_cswap(float (&v)[PER], int (&e)[PER], int i, int j) {
  const bool sw = (v[j] > v[i]) | ((v[j] == v[i]) & (e[j] < e[i]));
  const float vi = v[i], vj = v[j];
  const int ei = e[i], ej = e[j];
  v[i] = sw ? vj : vi;
  v[j] = sw ? vi : vj;
  e[i] = sw ? ej : ei;
  e[j] = sw ? ei : ej;
}

// Sorts a lane's candidates, first one first: Batcher's odd-even merge networks for
// 2, 4 and 8 inputs (1, 5 and 19 compare-exchanges; every key (score, id) is
// distinct, so any sorting network gives the same order).
template <int PER>
__device__ __forceinline__ void route_sort(float (&v)[PER], int (&e)[PER]) {
  if constexpr (PER == 2) {
    route_cswap<PER>(v, e, 0, 1);
  } else if constexpr (PER == 4) {
    constexpr int kNet[5][2] = {{0, 1}, {2, 3}, {0, 2}, {1, 3}, {1, 2}};
#pragma unroll
    for (int c = 0; c < 5; ++c) route_cswap<PER>(v, e, kNet[c][0], kNet[c][1]);
  } else if constexpr (PER == 8) {
    constexpr int kNet[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6},
                                 {5, 7}, {1, 2}, {5, 6}, {0, 4}, {1, 5}, {2, 6}, {3, 7},
                                 {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int c = 0; c < 19; ++c) route_cswap<PER>(v, e, kNet[c][0], kNet[c][1]);
  } else {
#pragma unroll
    for (int r = 0; r < PER; ++r)
#pragma unroll
      for (int i = r & 1; i + 1 < PER; i += 2) route_cswap<PER>(v, e, i, i + 1);
  }
}

// Where a routed token's bits go in the plan's token bitmap (see mark_token): the
// word of expert e is bitmap[e * per_expert + word], the token's bit in it `bit`.
struct TokenMark {
  uint32_t* bitmap;
  size_t per_expert;
  size_t word;
  uint32_t bit;
};

// One token, routed by G = 32 lanes (a whole warp, converged) or by G = 1 thread.
// Lane lig of the group holds the scores of experts lig, lig + G, ... (PER of them;
// -inf past E). Writes ids_row[0..k) and w_row[0..k) (from lig == 0). The decision
// compares scores, larger first, equal scores to the lower expert id: the order of
// the probabilities without their rounding ties. With forced_row, the ids are
// those and the weights the probabilities at them (0 for an id out of range, which
// the plan build reports). With `mark` (a gate's own top k, not prescribed ids), the
// thread that writes slot j also sets the token's bit of that expert in the plan's
// token bitmap, from the id it holds (no read back of the row it wrote).
//
// Cost. Every step is branch-free: padded candidates hold -inf, so exp adds an
// exact 0 for them and they never win. A warp's reductions are redux.sync over all
// 32 lanes (one instruction each; a reduction over part of a warp runs once per
// distinct lane mask, so groups of 2 to 16 lanes would be slower). With PER <= 8 a
// lane sorts its candidates once (route_sort) and each of the k rounds is two
// reductions and a shift of the winner's list; with more candidates per lane each
// round rescans them (the first strict maximum in ascending id order). A warp keeps
// round j's winner in lane j and computes the k weights after the rounds, one exp
// per lane, so no exp sits on the rounds' chain of reductions.
template <int G, int PER>
__device__ __forceinline__ void route_group(const float (&vin)[PER], int E, int k,
                                            const int32_t* forced_row, int32_t* ids_row,
                                            float* w_row, int lig,
                                            const TokenMark* mark = nullptr) {
  static_assert(G == 1 || G == 32, "a thread or a whole warp per token");
  static_assert(PER <= 32, "candidates per lane");
  constexpr uint32_t kAll = 0xFFFFFFFFu;
  // A warp's prescribed ids: lane j loads id j now, so that load overlaps the softmax
  // instead of adding one memory round trip per round (k <= 32).
  const int forced_mine =
      (G > 1 && forced_row != nullptr && lig < k) ? __ldg(forced_row + lig) : -1;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < PER; ++i) mx = fmaxf(mx, vin[i]);
  if (G > 1) mx = key_float(__reduce_max_sync(kAll, float_key(mx)));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) sum += expf(vin[i] - mx);
#pragma unroll
  for (int o = G / 2; o; o >>= 1) sum += __shfl_xor_sync(kAll, sum, o);
  const float inv = 1.0f / sum;

  if (forced_row != nullptr) {
    for (int j = 0; j < k; ++j) {
      const int e = G > 1 ? __shfl_sync(kAll, forced_mine, j) : __ldg(forced_row + j);
      const bool in = e >= 0 && e < E;
      float ve = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) ve = (in && e == lig + G * i) ? vin[i] : ve;
      if (G > 1) ve = __shfl_sync(kAll, ve, in ? e % G : 0);
      const float wj = in ? expf(ve - mx) * inv : 0.f;
      if (lig == 0) {
        ids_row[j] = e;
        w_row[j] = wj;
      }
    }
    return;
  }
  if (PER <= 8) {
    float v[PER];
    int e[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      v[i] = vin[i];
      e[i] = lig + G * i;
    }
    route_sort<PER>(v, e);
    uint32_t my_key = 0, my_id = 0;  // G = 32: round lig's winner
    for (int j = 0; j < k; ++j) {
      // The group's best head: the largest key, then the lowest id holding it.
      const uint32_t key = float_key(v[0]);
      const uint32_t kmax = G > 1 ? __reduce_max_sync(kAll, key) : key;
      const uint32_t cand = key == kmax ? (uint32_t)e[0] : 0xFFFFFFFFu;
      const uint32_t emin = G > 1 ? __reduce_min_sync(kAll, cand) : cand;
      const bool win = (uint32_t)e[0] == emin;
#pragma unroll
      for (int i = 0; i + 1 < PER; ++i) {
        v[i] = win ? v[i + 1] : v[i];
        e[i] = win ? e[i + 1] : e[i];
      }
      v[PER - 1] = win ? -INFINITY : v[PER - 1];
      e[PER - 1] = win ? 0x7FFFFFFF : e[PER - 1];
      if (G > 1) {
        my_key = lig == j ? kmax : my_key;
        my_id = lig == j ? emin : my_id;
      } else {
        ids_row[j] = (int32_t)emin;
        w_row[j] = expf(key_float(kmax) - mx) * inv;
        if (mark != nullptr) atomicOr(mark->bitmap + emin * mark->per_expert + mark->word, mark->bit);
      }
    }
    if (G > 1 && lig < k) {
      ids_row[lig] = (int32_t)my_id;
      w_row[lig] = expf(key_float(my_key) - mx) * inv;
      if (mark != nullptr) atomicOr(mark->bitmap + my_id * mark->per_expert + mark->word, mark->bit);
    }
  } else {
    uint32_t taken = 0;  // bit i: this lane's candidate i already chosen
    uint32_t my_key = 0, my_id = 0;  // G = 32: round lig's winner
    for (int j = 0; j < k; ++j) {
      // This lane's best candidate not yet taken: the first strict maximum in
      // ascending id order, so equal scores keep the lower id (a score of -inf
      // still counts once nothing else is left).
      float bv = -INFINITY;
      int bi = -1;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const bool better =
            !((taken >> i) & 1u) & (lig + G * i < E) & ((vin[i] > bv) | (bi < 0));
        bv = better ? vin[i] : bv;
        bi = better ? i : bi;
      }
      const uint32_t be = bi >= 0 ? (uint32_t)(lig + G * bi) : 0xFFFFFFFFu;
      const uint32_t key = float_key(bv);
      const uint32_t kmax = G > 1 ? __reduce_max_sync(kAll, key) : key;
      const uint32_t cand = key == kmax ? be : 0xFFFFFFFFu;
      const uint32_t emin = G > 1 ? __reduce_min_sync(kAll, cand) : cand;
      taken |= (bi >= 0 && be == emin) ? 1u << bi : 0u;
      if (G > 1) {
        my_key = lig == j ? kmax : my_key;
        my_id = lig == j ? emin : my_id;
      } else {
        ids_row[j] = (int32_t)emin;
        w_row[j] = expf(key_float(kmax) - mx) * inv;
        if (mark != nullptr) atomicOr(mark->bitmap + emin * mark->per_expert + mark->word, mark->bit);
      }
    }
    if (G > 1 && lig < k) {
      ids_row[lig] = (int32_t)my_id;
      w_row[lig] = expf(key_float(my_key) - mx) * inv;
      if (mark != nullptr) atomicOr(mark->bitmap + my_id * mark->per_expert + mark->word, mark->bit);
    }
  }
}

// One token routed by a group of G lanes (G = 2, 4, 8, 16 or 32 consecutive lanes of a
// converged warp, aligned to G; the warp's 32 / G groups route as many tokens at once).
// Lane lig of the group holds the scores of experts lig + G i (PER <= 8 of them, -inf
// past E), k <= E. The decision and the weights are route_group's: larger score first,
// equal scores to the lower id; weight = the softmax probability at the chosen id.
// The maximum, the sum of the exponentials and each round's winner are butterflies
// over the group (xor G/2, ..., 1); fp32 addition and the (score, id) order are
// commutative, so every lane of the group ends with the same values. Each lane sorts
// its candidates once (route_sort), so a round compares the groups' heads and the
// winner's lane shifts its list: where a thread per token runs a chain of some
// hundred dependent steps, or a warp per token a chain of redux.sync rounds for one
// token at a time, a group runs log2 G shuffles per round for 32 / G tokens at once.
// Lane 0 of an active group writes slot j (and, with `mark`, the token's bit of that
// expert).
template <int G, int PER>
__device__ __forceinline__ void route_lanes(const float (&vin)[PER], int k, int32_t* ids_row,
                                            float* w_row, int lig, bool active,
                                            const TokenMark* mark) {
  static_assert(G == 2 || G == 4 || G == 8 || G == 16 || G == 32, "lanes per token");
  static_assert(PER >= 1 && PER <= 8, "candidates per lane");
  constexpr uint32_t kAll = 0xFFFFFFFFu;
  float mx = vin[0];
#pragma unroll
  for (int i = 1; i < PER; ++i) mx = fmaxf(mx, vin[i]);
#pragma unroll
  for (int o = G / 2; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) sum += expf(vin[i] - mx);
#pragma unroll
  for (int o = G / 2; o; o >>= 1) sum += __shfl_xor_sync(kAll, sum, o);
  const float inv = 1.0f / sum;
  float v[PER];
  int e[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    v[i] = vin[i];
    e[i] = lig + G * i;
  }
  route_sort<PER>(v, e);
  int left = PER;  // candidates not yet taken, at the head of the sorted list
  for (int j = 0; j < k; ++j) {
    // This lane's head (key 0: none left; every score has a key > 0), then the group's.
    uint32_t bk = left > 0 ? float_key(v[0]) : 0u;
    uint32_t be = left > 0 ? (uint32_t)e[0] : 0xFFFFFFFFu;
#pragma unroll
    for (int o = G / 2; o; o >>= 1) {
      const uint32_t ok = __shfl_xor_sync(kAll, bk, o), oe = __shfl_xor_sync(kAll, be, o);
      const bool take = (ok > bk) | ((ok == bk) & (oe < be));
      bk = take ? ok : bk;
      be = take ? oe : be;
    }
    const bool win = left > 0 && (uint32_t)e[0] == be;
#pragma unroll
    for (int i = 0; i + 1 < PER; ++i) {
      v[i] = win ? v[i + 1] : v[i];
      e[i] = win ? e[i + 1] : e[i];
    }
    left -= win ? 1 : 0;
    if (active && lig == 0) {
      ids_row[j] = (int32_t)be;
      w_row[j] = expf(key_float(bk) - mx) * inv;
      if (mark != nullptr) atomicOr(mark->bitmap + be * mark->per_expert + mark->word, mark->bit);
    }
  }
}

// The plan's token bitmap (TileMoE notes section 4.2: rows are grouped by expert and
// source rank, in source-token order): one bit per (expert, source rank, token), set
// for every routing slot of token t of rank s, so that the plan build after a gate
// skips its bitmap kernel (the group counts stay in the plan's count kernel, which,
// unlike the gate kernels, fits beside a running producer CTA). A gate's own top k
// (k distinct ids in range) is marked inside route_group (TokenMark); this function
// marks prescribed ids, checked like the plan build checks them (out of range or
// repeated within the token: MOE_DEV_ROUTING, the slot skipped). G = 1: this thread
// routed the token; G = 32: lane j < k wrote slot j.
template <int G>
__device__ __forceinline__ void mark_token(const DevPlan& p, const int32_t* ids,
                                           const int32_t* forced, size_t tok, int s, int t,
                                           int lig, uint32_t* status) {
  const Dims& d = p.d;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(p.a[PA_BITMAP]);
  const int32_t* row = ids + tok * d.k;
  const bool check = forced != nullptr;
  if (G > 1 && check) __syncwarp();  // the ids the other lanes wrote
  for (int j = G > 1 ? lig : 0; j < d.k; j += G) {
    const int e = row[j];
    if (check) {
      bool ok = e >= 0 && e < d.E;
      for (int q = 0; q < j && ok; ++q) ok = row[q] != e;
      if (!ok) {
        report_error(status, MOE_DEV_ROUTING, (uint32_t)tok);
        continue;
      }
    }
    atomicOr(&bitmap[((size_t)e * d.W + s) * d.TW + (t >> 5)], 1u << (t & 31));
  }
}

#endif  // __CUDACC__

}  // namespace moe

// Combine copy: the body of the flag-polling consumer, shared by the standalone
// consumer kernel (its own SMs, beside or after the producer) and the copy warp of
// the fused pair producer. One warp runs it; see consumer.cu for the method.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kMaxGroups = MOE_MAX_RANKS * MOE_MAX_RANKS;

// Shared memory of one copying warp: SLOTS chunk slots live elsewhere.
template <int SLOTS>
struct CopySmem {
  uint64_t full[SLOTS];
  int stored[kMaxGroups];  // chunks of each group stored since the last release
  int rec[32][kSegRec];    // the segment record of each lane's chunk of the current round
  int cidx[32];            // that chunk's index inside its segment
};

// Copies every chunk i (of all segments, in the producer's tile order) with
// i % G == c: waits for its ready flags, moves it Y -> receive buffer through
// SLOTS shared-memory slots of kChunkBytes (at most INFLIGHT loads outstanding),
// and releases the stored chunks per group at each wait and at the end. Called by
// all 32 lanes of one warp.
template <int SLOTS, int INFLIGHT>
__device__ __forceinline__ void combine_copy(const DevPlan& p, const __nv_bfloat16* const* y,
                                             __nv_bfloat16* const* recv, uint8_t* slots,
                                             CopySmem<SLOTS>& sm, int c, int G) {
  static_assert(INFLIGHT >= 1 && INFLIGHT <= SLOTS, "copy ring");
  constexpr int kChunkSlots = SLOTS;
  constexpr int kLoadsInFlight = INFLIGHT;
  const Dims d = p.d;
  uint32_t* status = reinterpret_cast<uint32_t*>(p.a[PA_STATUS]);
  const uint32_t* flags = reinterpret_cast<const uint32_t*>(p.a[PA_FLAGS]);
  uint32_t* group_done = reinterpret_cast<uint32_t*>(p.a[PA_GROUP_DONE]);
  uint32_t* group_sig = reinterpret_cast<uint32_t*>(p.a[PA_GROUP_SIG]);
  const int32_t* recs = p.a[PA_SEG_REC];
  const int32_t* chunk_rec = p.a[PA_CHUNK_REC];
  const int32_t* gchunks = p.a[PA_GROUP_NCHUNK];
  const int nch = p.a[PA_TOTALS][4];
  const int lane = threadIdx.x & 31;
  const size_t row_bytes = (size_t)d.D * 2;

  for (int g = lane; g < kMaxGroups; g += 32) sm.stored[g] = 0;
  if (lane == 0) {
    for (int i = 0; i < kChunkSlots; ++i) mbar_init(&sm.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // Copy pipeline, driven by lane 0. Chunk i (in this CTA's order) uses slot i % S
  // and completes phase (i / S) & 1 of that slot's barrier. A chunk is stored as
  // soon as its load has landed; at most kLoadsInFlight loads are outstanding, so
  // when a slot is refilled at least S - kLoadsInFlight newer stores follow the
  // store that last used it, and waiting until only that many may still be reading
  // frees the slot without waiting for recent stores.
  struct Pend {
    uint8_t* dst;
    uint32_t bytes;
    int group;
  };
  Pend pend[kChunkSlots] = {};
  int n = 0, stored = 0;
  int released = 0;         // lane 0: chunks released (their landing stamped) so far
  bool unreleased = false;  // lane 0: chunks stored since the last release
  bool ok = true;
  const long long itimeout = p.timeout_ns + 4000000000LL;

  auto store_one = [&]() {  // lane 0: store chunk `stored` (bounded wait for its load)
    const int slot = stored % kChunkSlots;
    volatile int never = 0;
    if (!mbar_wait_bounded(&sm.full[slot], (stored / kChunkSlots) & 1, &never, itimeout, status,
                           0x60000000u))
      ok = false;
    bulk_store(pend[slot].dst, slots + (size_t)slot * kChunkBytes, pend[slot].bytes);
    bulk_commit();
    ++stored;
    ++sm.stored[pend[slot].group];
    unreleased = true;
  };
  auto store_landed = [&]() {  // lane 0: store every leading chunk whose load has landed
    while (stored < n && mbar_test_wait(&sm.full[stored % kChunkSlots], (stored / kChunkSlots) & 1))
      store_one();
  };
  // Every lane, at a warp-uniform point: lane 0 waits for its stores and fences
  // once; then each lane adds the stored chunks of its groups (g = lane, lane + 32)
  // to their counts with a release increment; the increment that completes a
  // group stores its signal.
  auto release_stored = [&]() {
    if (__shfl_sync(0xffffffffu, unreleased ? 1 : 0, 0) == 0) return;
    if (lane == 0) {
      bulk_wait_all();
      fence_proxy_async_global();
      fence_acq_rel_gpu();
      unreleased = false;
      if (p.chunk_t != nullptr) {
        // Timing on: every chunk stored since the last release has landed by now.
        // This CTA's m-th chunk is chunk c + m * G of the global sequence.
        const unsigned long long now = globaltimer();
        for (int m = released; m < stored; ++m) p.chunk_t[c + (size_t)m * G] = now;
      }
      released = stored;
    }
    __syncwarp();
    for (int g = lane; g < kMaxGroups; g += 32) {
      const uint32_t mine = (uint32_t)sm.stored[g];
      if (mine == 0) continue;
      sm.stored[g] = 0;
      fence_acq_rel_gpu();
      const uint32_t done = atomicAdd(group_done + g, mine) + mine;
      if (done == (uint32_t)gchunks[g]) {
        fence_acq_rel_gpu();
        st_release_u32(group_sig + g, 1u);
      }
    }
    __syncwarp();
  };

  // Rows [r0, r1) of the segment that round entry q (a lane's chunk) copies.
  auto chunk_rows = [&](int q, int& r0, int& r1) {
    r0 = sm.cidx[q] * d.rpc;
    r1 = min(sm.rec[q][4], r0 + d.rpc);
  };
  // Relaxed reads of the ready flags of one chunk (a subset of them per lane), all
  // in flight together; a caller that found them set issues one acquire fence per
  // lane (fence.acq_rel after the reads that observed the producer's release
  // increments) before the copies that read the chunk.
  auto flags_ready = [&](int q, int r0, int r1, int lane_lo, int lane_step) {
    const int b0 = sm.rec[q][2];
    const size_t rb = (size_t)sm.rec[q][0] * d.NBM;
    const int bl = b0 + r0 / d.tb, bh = b0 + (r1 - 1) / d.tb;
    const uint32_t* f = flags + (rb + bl) * d.nt2;
    const int nflags = (bh - bl + 1) * d.nt2;
    bool ready = true;
    for (int i = lane_lo; i < nflags; i += lane_step) ready &= ld_relaxed_u32(f + i) >= (uint32_t)d.parts;
    return ready;
  };

  // This warp's chunks are c, c + G, c + 2G, ... of the global sequence, and the plan
  // maps every chunk to its segment record. A round takes the next 32 of them, one
  // per lane: each lane reads its chunk's record and the chunk's ready flags (all
  // lanes' reads in flight together); then lane 0 moves the round's chunks in order,
  // waiting (bounded, all lanes) where a chunk is not produced yet.
  for (long long m0 = 0; ok; m0 += 32) {
    const long long i = (long long)c + (m0 + lane) * G;
    const bool have = i < nch;
    const int m = __popc(__ballot_sync(0xffffffffu, have));  // lanes 0 .. m-1
    if (m == 0) break;
    __syncwarp();  // lane 0 no longer reads the previous round's records
    bool rdy = true;
    if (have) {
      const int q = __ldg(chunk_rec + i);
      const int4* r = reinterpret_cast<const int4*>(recs + (size_t)q * kSegRec);
      const int4 lo = __ldg(r), hi = __ldg(r + 1);
      sm.rec[lane][0] = lo.x; sm.rec[lane][1] = lo.y; sm.rec[lane][2] = lo.z; sm.rec[lane][3] = lo.w;
      sm.rec[lane][4] = hi.x; sm.rec[lane][5] = hi.y; sm.rec[lane][6] = hi.z; sm.rec[lane][7] = hi.w;
      sm.cidx[lane] = (int)(i - hi.z);
      int r0, r1;
      chunk_rows(lane, r0, r1);
      rdy = flags_ready(lane, r0, r1, 0, 1);
    }
    unsigned ready = __ballot_sync(0xffffffffu, rdy);
    fence_acq_rel_gpu();  // each lane: its flag reads become acquires
    __syncwarp();         // orders lane 0's copies after every lane's acquire (and records)
    // The flags were acquired (generic proxy); the bulk loads read Y (async proxy).
    if (lane == 0) fence_proxy_async_global();
    for (int j = 0; j < m && ok; ++j) {
      int r0, r1;
      chunk_rows(j, r0, r1);
      if (!(ready >> j & 1u)) {
        // Not produced yet: store everything loaded, release the stored chunks,
        // then wait (bounded, all lanes).
        if (lane == 0)
          while (stored < n) store_one();
        release_stored();
        const unsigned long long t0 = globaltimer();
        bool done = false, stop = false;
        while (!done && !stop) {
          done = __all_sync(0xffffffffu, flags_ready(j, r0, r1, lane, 32));
          if (!done) {
            __nanosleep(64);
            if (lane == 0) {
              if (ld_relaxed_u32(status) != 0) {
                stop = true;
              } else if ((long long)(globaltimer() - t0) > p.timeout_ns) {
                const int bl = sm.rec[j][2] + r0 / d.tb;
                report_error(status, MOE_DEV_TIMEOUT,
                             0x50000000u | (uint32_t)((size_t)sm.rec[j][0] * d.NBM + bl));
                stop = true;
              }
            }
            stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
          }
        }
        if (stop) {
          ok = false;
          break;
        }
        // Chunks after this one may have become ready meanwhile.
        bool again = true;
        if (lane > j && lane < m) {
          int b0, b1;
          chunk_rows(lane, b0, b1);
          again = flags_ready(lane, b0, b1, 0, 1);
        }
        ready = __ballot_sync(0xffffffffu, again) | (j == 31 ? 0xffffffffu : (2u << j) - 1u);
        fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0) fence_proxy_async_global();
      }
      if (lane == 0) {
        store_landed();
        while (n - stored >= kLoadsInFlight) store_one();
        if (n >= kChunkSlots) bulk_wait_read<kChunkSlots - kLoadsInFlight>();
        const int o = sm.rec[j][0], dst = sm.rec[j][1], b0 = sm.rec[j][2];
        const int slot = n % kChunkSlots;
        const uint32_t bytes = (uint32_t)((size_t)(r1 - r0) * row_bytes);
        const uint8_t* src =
            reinterpret_cast<const uint8_t*>(y[o]) + ((size_t)b0 * d.tb + r0) * row_bytes;
        pend[slot].dst =
            reinterpret_cast<uint8_t*>(recv[dst]) + ((size_t)sm.rec[j][5] + r0) * row_bytes;
        pend[slot].bytes = bytes;
        pend[slot].group = o * d.W + dst;
        mbar_arrive_expect_tx(&sm.full[slot], bytes);
        bulk_load(slots + (size_t)slot * kChunkBytes, src, bytes, &sm.full[slot]);
        ++n;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
  }
  // Drain: store what was loaded (even after an error, so no copy outlives the
  // CTA's shared memory), release the stored chunks, wait for every store.
  if (lane == 0)
    while (stored < n) store_one();
  release_stored();
  if (lane == 0) bulk_wait_all();
}

}  // namespace moe

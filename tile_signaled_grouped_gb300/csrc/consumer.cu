// Combine consumer: polls the producer's per-tile ready flags and copies every
// finished segment's valid rows into its destination rank's receive buffer.
//
// TileMoE notes (zhongzhuzhou.org), section 5.2: the transfer unit is a row
// band (tb_M rows x the full output width: one owner, contiguous), merged into
// segments; section 5.3: a persistent consumer on its own SMs, coordinated with
// the producer only through device memory; section 4.5: destination, offset and
// valid-row count come from the precomputed combine plan (padding is never sent).
// Perseus summary (papercache.org), section 4.1, Algorithm 1: data moves without
// signals; one fence then precedes the signals of a whole destination group.
//
// GB300 form: each segment is cut into chunks of rpc rows (up to 40 KB); the
// chunks of all segments, in the producer's tile order, are dealt round-robin to
// the consumer CTAs, so every CTA follows production and the last segment is
// copied by all of them. A CTA is one warp: the lanes poll the flags of a chunk's
// bands together, and lane 0 moves the chunk with TMA bulk copies through a
// six-slot shared-memory ring (global -> shared completes on an mbarrier,
// shared -> global as a bulk group). A group is (sender o, destination s). When a
// CTA has stored the last of its chunks of a group, the group joins a release
// batch: at the CTA's next wait (or its end) it waits for its stores, issues one
// fence for the whole batch and one release increment of each group's chunk
// count; the increment that completes a group stores the group signal.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kMaxGroups = MOE_MAX_RANKS * MOE_MAX_RANKS;

constexpr int kListCap = kMaxSegChunks;  // owned chunks listed per batch of records

struct ConsumerSmem {
  uint64_t full[kChunkSlots];
  int owned[kMaxGroups];  // this CTA's chunks of each group not yet stored
  int total[kMaxGroups];  // this CTA's chunks of each group
  int rec[32][kSegRec];   // a batch of segment records
  int list[kListCap];     // owned chunks of the batch: (record << 24) | chunk index
};

static_assert(sizeof(ConsumerSmem) <= kConsumerSmemTail, "consumer shared memory layout");

// Chunks i in [cb, cb + n) with i % G == c.
__device__ __forceinline__ int owned_count(int cb, int n, int c, int G) {
  const int i0 = cb + ((c - cb) % G + G) % G;
  return i0 >= cb + n ? 0 : (cb + n - 1 - i0) / G + 1;
}

__global__ void __launch_bounds__(kConsumerThreads, 1)
    consumer_kernel(const __grid_constant__ ConsumerArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* slots = smem_raw;
  ConsumerSmem& sm = *reinterpret_cast<ConsumerSmem*>(smem_raw + (size_t)kChunkSlots * kChunkBytes);
  const Dims d = a.p.d;
  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  const uint32_t* flags = reinterpret_cast<const uint32_t*>(a.p.a[PA_FLAGS]);
  uint32_t* group_done = reinterpret_cast<uint32_t*>(a.p.a[PA_GROUP_DONE]);
  uint32_t* group_sig = reinterpret_cast<uint32_t*>(a.p.a[PA_GROUP_SIG]);
  const int32_t* recs = a.p.a[PA_SEG_REC];
  const int32_t* gchunks = a.p.a[PA_GROUP_NCHUNK];
  const int nseg = a.p.a[PA_TOTALS][1];
  const int lane = threadIdx.x;
  const int c = blockIdx.x, G = gridDim.x;
  const size_t row_bytes = (size_t)d.D * 2;

  for (int g = lane; g < kMaxGroups; g += 32) sm.owned[g] = 0;
  if (lane == 0) {
    for (int i = 0; i < kChunkSlots; ++i) mbar_init(&sm.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  // Pre-pass: how many chunks of each group this CTA copies.
  for (int idx = lane; idx < nseg; idx += 32) {
    const int32_t* r = recs + (size_t)idx * kSegRec;
    const int n = owned_count(r[6], r[7], c, G);
    if (n) atomicAdd(&sm.owned[r[0] * d.W + r[1]], n);
  }
  __syncwarp();
  for (int g = lane; g < kMaxGroups; g += 32) sm.total[g] = sm.owned[g];
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
  unsigned long long finished = 0;  // groups whose chunks (of this CTA) are all stored
  bool ok = true;
  const long long itimeout = a.p.timeout_ns + 4000000000LL;

  auto store_one = [&]() {  // lane 0: store chunk `stored` (bounded wait for its load)
    const int slot = stored % kChunkSlots;
    volatile int never = 0;
    if (!mbar_wait_bounded(&sm.full[slot], (stored / kChunkSlots) & 1, &never, itimeout, status,
                           0x60000000u))
      ok = false;
    bulk_store(pend[slot].dst, slots + (size_t)slot * kChunkBytes, pend[slot].bytes);
    bulk_commit();
    ++stored;
    const int g = pend[slot].group;
    if (--sm.owned[g] == 0) finished |= 1ull << g;
  };
  auto store_landed = [&]() {  // lane 0: store every leading chunk whose load has landed
    while (stored < n && mbar_try_wait(&sm.full[stored % kChunkSlots], (stored / kChunkSlots) & 1))
      store_one();
  };
  // One fence for every group this CTA has finished since the last release, then
  // one count increment per group; the increment that completes a group signals it.
  auto release_finished = [&]() {
    if (finished == 0) return;
    bulk_wait_all();
    fence_proxy_async_global();
    fence_acq_rel_gpu();
    while (finished) {
      const int g = __ffsll((long long)finished) - 1;
      finished &= finished - 1;
      const uint32_t mine = (uint32_t)sm.total[g];
      const uint32_t done = atomicAdd(group_done + g, mine) + mine;
      if (done == (uint32_t)gchunks[g]) st_release_u32(group_sig + g, 1u);
    }
  };

  // Rows and flags of listed chunk `e` (a packed list entry).
  auto chunk_of = [&](int e, int& q, int& r0, int& r1) {
    q = e >> 24;
    const int k = e & 0xFFFFFF;
    r0 = k * d.rpc;
    r1 = min(sm.rec[q][4], r0 + d.rpc);
  };
  auto flags_ready = [&](int q, int r0, int r1, int lane_lo, int lane_step) {
    const int b0 = sm.rec[q][2];
    const size_t rb = (size_t)sm.rec[q][0] * d.NBM;
    const int bl = b0 + r0 / d.tb, bh = b0 + (r1 - 1) / d.tb;
    const uint32_t* f = flags + (rb + bl) * d.nt2;
    const int nflags = (bh - bl + 1) * d.nt2;
    bool ready = true;
    for (int i = lane_lo; i < nflags; i += lane_step) ready &= ld_acquire_u32(f + i) >= (uint32_t)d.parts;
    return ready;
  };

  // Records are read a batch of 32 ahead: each lane keeps the record it will
  // publish for the next batch in registers, so that load's latency overlaps the
  // copies of the current batch.
  int nextrec[kSegRec];
  auto fetch = [&](int b) {
    if (b + lane < nseg) {
      const int32_t* r = recs + (size_t)(b + lane) * kSegRec;
#pragma unroll
      for (int q = 0; q < kSegRec; ++q) nextrec[q] = r[q];
    }
  };
  fetch(0);
  int base = 0, fetched = 0;
  while (base < nseg && ok) {
    // Publish up to 32 records (the prefetched ones when they start at `base`).
    const int nb = min(32, nseg - base);
    __syncwarp();
    if (fetched != base) fetch(base);
    if (lane < nb) {
#pragma unroll
      for (int q = 0; q < kSegRec; ++q) sm.rec[lane][q] = nextrec[q];
    }
    __syncwarp();
    int cnt = 0;
    if (lane < nb) cnt = owned_count(sm.rec[lane][6], sm.rec[lane][7], c, G);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    // Records taken: every lane whose inclusive count fits (the first always fits,
    // because a segment has at most kListCap chunks).
    const unsigned fit = __ballot_sync(0xffffffffu, lane < nb && incl <= kListCap);
    const int take = max(1, __popc(fit));
    const int nlist = __shfl_sync(0xffffffffu, incl, take - 1);
    fetch(base + take);
    fetched = base + take;
    if (lane < take && cnt > 0) {
      const int cb = sm.rec[lane][6];
      int k = ((c - cb) % G + G) % G;
      for (int j = 0, pos = incl - cnt; j < cnt; ++j, ++pos, k += G) sm.list[pos] = (lane << 24) | k;
    }
    __syncwarp();

    // Walk the listed chunks 32 at a time: every lane checks one chunk's flags, so
    // the flag latency is paid once per 32 chunks while copies are in flight.
    for (int s0 = 0; s0 < nlist && ok; s0 += 32) {
      const int m = min(32, nlist - s0);
      bool mine = true;
      if (lane < m) {
        int q, r0, r1;
        chunk_of(sm.list[s0 + lane], q, r0, r1);
        mine = flags_ready(q, r0, r1, 0, 1);
      }
      unsigned ready = __ballot_sync(0xffffffffu, mine);
      for (int j = 0; j < m && ok; ++j) {
        int q, r0, r1;
        chunk_of(sm.list[s0 + j], q, r0, r1);
        if (!(ready >> j & 1u)) {
          // Not produced yet: store everything loaded, then wait (bounded, all lanes).
          if (lane == 0) {
            while (stored < n) store_one();
            release_finished();
          }
          const unsigned long long t0 = globaltimer();
          bool done = false, stop = false;
          while (!done && !stop) {
            done = __all_sync(0xffffffffu, flags_ready(q, r0, r1, lane, 32));
            if (!done) {
              __nanosleep(64);
              if (lane == 0) {
                if (ld_relaxed_u32(status) != 0) {
                  stop = true;
                } else if ((long long)(globaltimer() - t0) > a.p.timeout_ns) {
                  const int bl = sm.rec[q][2] + r0 / d.tb;
                  report_error(status, MOE_DEV_TIMEOUT,
                               0x50000000u | (uint32_t)((size_t)sm.rec[q][0] * d.NBM + bl));
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
            int q2, a0, a1;
            chunk_of(sm.list[s0 + lane], q2, a0, a1);
            again = flags_ready(q2, a0, a1, 0, 1);
          }
          ready = __ballot_sync(0xffffffffu, again) | ((1u << j) << 1) - 1u;
        }
        if (lane == 0) {
          fence_proxy_async_global();  // the flags were acquired; the bulk load reads Y
          store_landed();
          while (n - stored >= kLoadsInFlight) store_one();
          if (n >= kChunkSlots) bulk_wait_read<kChunkSlots - kLoadsInFlight>();
          const int o = sm.rec[q][0], dst = sm.rec[q][1], b0 = sm.rec[q][2];
          const int slot = n % kChunkSlots;
          const uint32_t bytes = (uint32_t)((size_t)(r1 - r0) * row_bytes);
          const uint8_t* src =
              reinterpret_cast<const uint8_t*>(a.y[o]) + ((size_t)b0 * d.tb + r0) * row_bytes;
          pend[slot].dst =
              reinterpret_cast<uint8_t*>(a.recv[dst]) + ((size_t)sm.rec[q][5] + r0) * row_bytes;
          pend[slot].bytes = bytes;
          pend[slot].group = o * d.W + dst;
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          bulk_load(slots + (size_t)slot * kChunkBytes, src, bytes, &sm.full[slot]);
          ++n;
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    base += take;
  }
  if (lane == 0) {
    // Drain: store what was loaded (even after an error, so no copy outlives the
    // CTA's shared memory), then wait for every store.
    while (stored < n) store_one();
    release_finished();
    bulk_wait_all();
  }
}

}  // namespace

cudaError_t preload_consumer() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, consumer_kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(consumer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kConsumerSmem);
}

cudaError_t launch_consumer(const ConsumerArgs& a, int grid, cudaStream_t s) {
  // 120 KB of shared memory per CTA also keeps a consumer CTA from sharing an SM
  // with a producer CTA or another consumer CTA: the kernels run on disjoint SMs.
  consumer_kernel<<<grid, kConsumerThreads, kConsumerSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

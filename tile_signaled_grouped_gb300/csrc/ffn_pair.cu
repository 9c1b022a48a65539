// Persistent grouped expert-FFN producer on CTA pairs (sm_103a: clusters of two
// CTAs, TMA + tcgen05 with cta_group::2 + TMEM).
//
// Computes what the one-CTA producer computes (TileMoE notes, zhongzhuzhou.org,
// section 5.1: one persistent kernel over all local experts, tiles taken in the
// remote-first order, and the epilogue of every finished output tile makes it
// visible and sets its ready flag, section 2.3), with one change of granularity:
// a task covers two 128-row tiles of the same expert, rows estart + 256 i and
// estart + 256 i + 128 of its block (the plan's pair list; the second tile may be
// missing). One tcgen05.mma of M = 256 multiplies both: each CTA of the pair
// stages its own 128 rows of A and half of the B rows, and the accumulator rows
// of each CTA land in its own TMEM. Per 256 x 256 x 64 step the pair reads
// 2 x 16 KB of A and 32 KB of weights (instead of 2 x 48 KB for two one-CTA
// tiles), so a stage is 32 KB and seven stages fit beside the task state.
//
// Roles. In each CTA a scheduler thread (warp 10) takes the tasks: cluster rank
// 0 (the leader) takes tickets from the atomic counter and hands each ticket to
// rank 1 through a ring in rank 1's shared memory; both decode the same ticket
// and post it to the CTA's task ring. In both CTAs warp 0 lane 0 issues the TMA loads
// of its own half (signalling the leader's full barrier: .cta_group::2 copies may
// complete on the peer's barrier), and warps 2-9 drain the CTA's own accumulator
// rows (two groups of four warps, one column half each), write h or Y and
// publish the tile's signal. Only the leader's warp 1 lane 0 issues MMAs; its
// commits arrive on both CTAs' barriers (multicast).
// The accumulator is freed for reuse when both CTAs' epilogues have arrived on
// the leader's tempty barrier.
//
// Fused variant (consumer_ctas = MOE_CONSUMER_FUSED): every CTA also runs the
// combine copy in one more warp (the standalone consumer's body with one chunk
// slot), so no SM is set aside for the consumer; the pipeline keeps six stages.
//
// Waits. The scheduler posts a GEMM2 task once its rows' GEMM1 tiles are counted
// (a wait bounded by timeout_ns); on expiry it records MOE_DEV_TIMEOUT and posts the
// task anyway (its result is void), so the two CTAs never disagree on the task
// sequence; the leader stops taking tickets as soon as the status word is set.
// Every other wait depends only on the pair's own progress and is bounded by
// timeout_ns + 4 s.
// The CTAs meet in a cluster barrier only at the start (barriers and TMEM ready
// in both) and at the end (every MMA drained, every copy landed), then free TMEM.
#include "combine_copy.cuh"

namespace moe {
namespace {

constexpr int kPMaxStages = 7;  // pipeline depth (the fused variant uses one stage less)
// Warp roles: warp 0 TMA, warp 1 MMA (rank 0 only), warps 2-9 epilogue, warp 10
// scheduler (lane 0 of each single-thread role works; its other lanes idle).
constexpr int kEpiWarp0 = 2, kEpiWarps = 8;
constexpr int kSchedWarp = kEpiWarp0 + kEpiWarps;
constexpr int kCopyWarp = kSchedWarp + 1;  // fused variant: the combine copy
static_assert(kEpiWarps % 4 == 0, "each epilogue group covers all four TMEM lane quarters");
constexpr int kPRing = 2;  // posted tasks in flight inside one CTA (more widens the L2 working set)
constexpr int kHRing = 4;  // tickets in flight from rank 0 to rank 1
constexpr int kPABytes = kTileM * kBlockK * 2;  // 16 KB: this CTA's 128 rows of A
constexpr int kPBBytes = 128 * kBlockK * 2;     // 16 KB: at most 128 B rows per CTA
constexpr int kPUnitCache = 256;  // scheduling units kept in shared memory; later ones are read from the plan
constexpr int kPAccCols = 256;

enum PTaskKind : int { kPEnd = -1, kPG1 = 0, kPG2 = 1 };

struct PTask {
  int kind;
  int own;   // this CTA's tile (global tile index), -1 if the pair has no second tile
  int nt;    // tile along F (GEMM1) or D (GEMM2)
  int o;     // owner rank
  int row0;  // first X / h row this CTA loads (its own tile, else the pair's first)
  int li;    // local expert index
  int ld;    // tile whose rows this CTA loads
  int pad;
};

struct PSmem {
  uint64_t full[kPMaxStages], empty[kPMaxStages];
  uint64_t tfull[2], tempty[2];
  uint64_t qfull[kPRing], qempty[kPRing];
  uint64_t hfull[kHRing], hempty[kHRing];  // ticket hand-off: hfull in rank 1, hempty in rank 0
  uint64_t drain;
  long long hticket[kHRing];  // written by rank 0 into rank 1
  PTask task[kPRing];
  PTask etask;
  int eok;
  uint32_t tmem_base;
  int abort;
  int nunits;
  int unit_begin[kPUnitCache + 1];
};

// The fused variant also runs the combine copy in warp kCopyWarp: one chunk slot
// and the copy state, paid for with one pipeline stage.
using PairCopySmem = CopySmem<1>;
template <bool FUSED>
struct PairCfg {
  static constexpr int kStages = FUSED ? kPMaxStages - 1 : kPMaxStages;
  static constexpr int kThreads = 32 * (kSchedWarp + 1 + (FUSED ? 1 : 0));
  static constexpr size_t kStageBytes = (size_t)kStages * (kPABytes + kPBBytes);
  static constexpr size_t kSmem = 1024 /*alignment slack*/ + kStageBytes + sizeof(PSmem) +
                                  (FUSED ? (size_t)kChunkBytes + sizeof(PairCopySmem) + 16 : 0);
};
static_assert(PairCfg<false>::kSmem <= 227 * 1024, "pair producer shared memory");
static_assert(PairCfg<true>::kSmem <= 227 * 1024, "fused pair producer shared memory");

// --- cluster and cta_group::2 forms ------------------------------------------
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
               : "memory");
}
__device__ __forceinline__ void st_cluster_s64(uint32_t cl_addr, long long v) {
  asm volatile("st.shared::cluster.s64 [%0], %1;" ::"r"(cl_addr), "l"(v) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals may come from the other CTA).
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                      long long timeout_ns, uint32_t* status, uint32_t detail) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cl(bar, parity)) return true;
    if (*abort) return false;
    if ((long long)(globaltimer() - t0) > timeout_ns) {
      report_error(status, MOE_DEV_TIMEOUT, detail);
      *abort = 1;
      return false;
    }
  }
}
// TMA tile load into this CTA's shared memory that completes on a barrier of
// either CTA of the pair (cl_bar: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t cl_bar,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cl_bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the barrier at the same offset in every CTA of `mask` when all
// MMAs this thread issued so far have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Named barrier 1: the epilogue warps only.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

__device__ __forceinline__ int unit_at(const PSmem& sm, const int32_t* gub, int u) {
  return u <= kPUnitCache ? sm.unit_begin[u] : gub[u];
}

// Tasks before unit u: GEMM1 tasks of units < u, GEMM2 tasks of units < u - lag.
__device__ __forceinline__ long long tasks_before(const PSmem& sm, const int32_t* gub, int u,
                                                  int NU, int lag, int nt1, int nt2) {
  const int u1 = min(u, NU);
  const int u2 = max(0, min(u - lag, NU));
  return (long long)nt1 * unit_at(sm, gub, u1) + (long long)nt2 * unit_at(sm, gub, u2);
}

// Ticket -> (kind, pair, N-tile), the ticket order of the one-CTA producer over
// pairs instead of tiles; then this CTA's tile of the pair.
__device__ PTask decode_ticket(const PSmem& sm, const ProducerArgs& a, long long ticket,
                               uint32_t crank) {
  const Dims& d = a.p.d;
  const int32_t* gub = a.p.a[PA_PAIR_UNIT_BEGIN];
  const int NU = sm.nunits;
  const int NP = unit_at(sm, gub, NU);
  PTask tk{};
  tk.kind = kPEnd;
  const long long total = (long long)NP * (d.nt1 + d.nt2);
  if (ticket < 0 || ticket >= total || NU == 0) return tk;
  int lo = 0, hi = NU + a.lag - 1;  // largest u with tasks_before(u) <= ticket
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tasks_before(sm, gub, mid, NU, a.lag, d.nt1, d.nt2) <= ticket) lo = mid; else hi = mid - 1;
  }
  const int u = lo;
  long long r = ticket - tasks_before(sm, gub, u, NU, a.lag, d.nt1, d.nt2);
  const int sz1 = u < NU ? unit_at(sm, gub, u + 1) - unit_at(sm, gub, u) : 0;
  int pm;
  if (r < (long long)d.nt1 * sz1) {
    // A unit's GEMM1 tasks run by run of one expert, hidden-column-major inside a run:
    // a run's X tiles stay in L2 across its hidden blocks, and consecutive tasks share
    // a weight tile. Run i's tasks are [nt1 b_i, nt1 b_(i+1)) (b: its first pair's
    // offset in the unit), so the pair at offset r / nt1 lies in task r's run.
    tk.kind = kPG1;
    const int ub = unit_at(sm, gub, u);
    const int run = __ldg(a.p.a[PA_PAIR_RUN] + ub + (int)(r / d.nt1));
    const int rs = run & 0xFFFF, rl = run >> 16;
    const int local = (int)r - d.nt1 * rs;
    pm = ub + rs + local % rl;
    tk.nt = local / rl;
  } else {
    // GEMM2 tasks pair-major, except inside a run whose pairs' h fits in 8 MB
    // (rl * 256 rows * F * 2 bytes): there N-tile-major, so that the run's pairs take
    // each W_down slice back to back while their h stays in L2.
    r -= (long long)d.nt1 * sz1;
    tk.kind = kPG2;
    const int ub = unit_at(sm, gub, u - a.lag);
    const int run = __ldg(a.p.a[PA_PAIR_RUN] + ub + (int)(r / d.nt2));
    const int rs = run & 0xFFFF, rl = run >> 16;
    if ((long long)rl * d.F <= 16384) {
      const int local = (int)r - d.nt2 * rs;
      pm = ub + rs + local % rl;
      tk.nt = local / rl;
    } else {
      pm = ub + (int)(r / d.nt2);
      tk.nt = (int)(r % d.nt2);
    }
  }
  // One 16-byte record per pair (written by the plan, read-only here).
  const int4 rec = __ldg(reinterpret_cast<const int4*>(a.p.a[PA_PAIR]) + pm);
  tk.own = crank == 0 ? rec.x : rec.y;
  tk.ld = tk.own >= 0 ? tk.own : rec.x;
  tk.o = rec.z >> 24;
  tk.row0 = rec.z & 0xFFFFFF;
  if (crank != 0 && rec.y >= 0) tk.row0 += (rec.w >> 16) ? -kTileM : kTileM;
  tk.li = rec.w & 0xFFFF;
  return tk;
}

template <bool FUSED>
// At most 104 registers a thread (384 threads: 39,936 of the SM's 65,536), so that a
// 256-thread CTA of up to 96 registers (the scale, the gather, the plan kernels of the
// other batch in flight) fits beside a producer CTA; without the cap the compiler took
// 118, and the scale then waited for the whole next producer to finish.
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(104)
    ffn_pair_kernel(const __grid_constant__ ProducerArgs a) {
  constexpr int kPStages = PairCfg<FUSED>::kStages;
  extern __shared__ uint8_t smem_raw[];
  allow_dependent_launch();  // a scale launched behind this kernel may start beside it
  const Dims d = a.p.d;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* stage_base = smem_raw + pad;
  uint8_t* a_tiles = stage_base;                                // kPStages x 16 KB
  uint8_t* b_tiles = stage_base + (size_t)kPStages * kPABytes;  // kPStages x 16 KB
  PSmem& sm = *reinterpret_cast<PSmem*>(stage_base + (size_t)kPStages * (kPABytes + kPBBytes));
  // Fused variant: the copy slot (16-byte aligned) and the copy state follow.
  uint8_t* copy_slot = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(&sm + 1) + 15) & ~static_cast<uintptr_t>(15));
  PairCopySmem& csm = *reinterpret_cast<PairCopySmem*>(copy_slot + kChunkBytes);

  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  uint32_t* queue = reinterpret_cast<uint32_t*>(a.p.a[PA_QUEUE]);
  uint32_t* g1cnt = reinterpret_cast<uint32_t*>(a.p.a[PA_G1CNT]);
  uint32_t* flags = reinterpret_cast<uint32_t*>(a.p.a[PA_FLAGS]);
  const long long timeout = a.p.timeout_ns;
  const long long itimeout = a.p.timeout_ns + 4000000000LL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool lead = crank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&sm.full[i], 1);   // rank 0: its arrive.expect_tx (bytes of both CTAs)
      mbar_init(&sm.empty[i], 1);  // the leader's commit (multicast)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tfull[i], 1);   // the leader's commit (multicast)
      mbar_init(&sm.tempty[i], 2);  // rank 0: both CTAs' epilogue leaders
    }
    for (int i = 0; i < kPRing; ++i) {
      mbar_init(&sm.qfull[i], 1);
      mbar_init(&sm.qempty[i], lead ? 3 : 2);  // TMA thread, MMA thread (rank 0), epilogue leader
    }
    for (int i = 0; i < kHRing; ++i) {
      mbar_init(&sm.hfull[i], 1);
      mbar_init(&sm.hempty[i], 1);
    }
    mbar_init(&sm.drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sm.abort = 0;
    sm.nunits = a.p.a[PA_TOTALS][2];
  }
  if (warp == 0) tmem_alloc_pair(&sm.tmem_base, 2 * kPAccCols);
  __syncthreads();
  {
    const int NU = sm.nunits;
    const int32_t* gub = a.p.a[PA_PAIR_UNIT_BEGIN];
    for (int u = threadIdx.x; u <= min(NU, kPUnitCache); u += blockDim.x) sm.unit_begin[u] = gub[u];
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync_all();  // both CTAs: barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;
  if (threadIdx.x == 0) span_begin(a.p.span);

  if (FUSED && warp == kCopyWarp) {
    // ------------------------------------------------------------ combine copy
    // Every CTA of the grid copies its share of the finished segments (chunk i
    // when i % grid == CTA index), polling the ready flags, exactly as the
    // standalone consumer does on its own SMs.
    combine_copy<1, 1>(a.p, a.y, a.recv, copy_slot, csm, blockIdx.x, gridDim.x);
  } else if (warp == kSchedWarp && lane == 0) {
    // ------------------------------------------------------------ scheduler
    // Takes every ticket (rank 0 from the counter, handing it to rank 1), decodes
    // it, makes sure a GEMM2 task's h rows are complete, and posts the task to the
    // ring that the TMA, MMA and epilogue roles read. All global round trips of
    // the scheduling sit here, off the path of the loads. Rank 0 fetches each
    // ticket one task ahead and reads the status word right after a hand-off.
    const long long total =
        (long long)unit_at(sm, a.p.a[PA_PAIR_UNIT_BEGIN], sm.nunits) * (d.nt1 + d.nt2);
    long long next = lead ? (long long)atomicAdd(queue, 1u) : 0;
    uint32_t status_seen = lead ? ld_relaxed_u32(status) : 0u;
    for (int it = 0;; ++it) {
      const int hs = it % kHRing;
      const uint32_t hph = (it / kHRing) & 1;
      long long ticket = -1;
      if (lead) {
        ticket = next < total && status_seen == 0 ? next : -1;
        if (!pwait(&sm.hempty[hs], hph ^ 1, &sm.abort, itimeout, status, 0x13000000u)) break;
        st_cluster_s64(map_shared(&sm.hticket[hs], 1), ticket);
        mbar_arrive_cluster(map_shared(&sm.hfull[hs], 1));
        if (ticket >= 0) next = atomicAdd(queue, 1u);
        status_seen = ld_relaxed_u32(status);
      } else {
        if (!pwait(&sm.hfull[hs], hph, &sm.abort, itimeout, status, 0x14000000u)) break;
        ticket = sm.hticket[hs];
        mbar_arrive_cluster(map_shared(&sm.hempty[hs], 0));
      }
      const PTask tk = decode_ticket(sm, a, ticket, crank);
      if (tk.kind == kPG2) {
        // Every GEMM1 tile of the rows this CTA loads must be counted (bounded
        // wait). On expiry, or once another CTA has set the status word, the task
        // still runs: its result is void, and rank 0 takes no further ticket.
        const uint32_t* c = g1cnt + tk.ld;
        if (ld_acquire_u32(c) < (uint32_t)d.nt1) {
          const unsigned long long t0 = globaltimer();
          while (ld_acquire_u32(c) < (uint32_t)d.nt1) {
            if (ld_relaxed_u32(status) != 0) break;
            if ((long long)(globaltimer() - t0) > timeout) {
              report_error(status, MOE_DEV_TIMEOUT, 0x40000000u | (uint32_t)tk.ld);
              break;
            }
            __nanosleep(64);
          }
        }
      }
      const int slot = it % kPRing;
      if (!pwait(&sm.qempty[slot], ((it / kPRing) & 1) ^ 1, &sm.abort, itimeout, status,
                 0x10000000u))
        break;
      sm.task[slot] = tk;
      mbar_arrive(&sm.qfull[slot]);
      if (tk.kind == kPEnd) break;
    }
  } else if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    for (int r = 0; r < d.W; ++r) {
      tma_prefetch_desc(&a.tm_x[r]);
      tma_prefetch_desc(&a.tm_h[r]);
      tma_prefetch_desc(&a.tm_wg[r]);
      tma_prefetch_desc(&a.tm_wu[r]);
      tma_prefetch_desc(&a.tm_wd[r]);
    }
    const uint32_t half_b2 = (uint32_t)(d.N2 / 2);
    uint32_t kit = 0;
    for (int it = 0;; ++it) {
      const int slot = it % kPRing;
      if (!pwait(&sm.qfull[slot], (it / kPRing) & 1, &sm.abort, itimeout, status, 0x15000000u))
        break;
      const PTask cur = sm.task[slot];
      mbar_arrive(&sm.qempty[slot]);
      if (cur.kind == kPEnd) break;
      // h rows were found complete by the scheduler (acquire); order this
      // thread's view of them before its asynchronous-proxy reads.
      if (cur.kind == kPG2) fence_proxy_async_global();
      const bool g1 = cur.kind == kPG1;
      const int nk = (g1 ? d.D : d.F) / kBlockK;
      const uint32_t bytes = 2 * kPABytes + (g1 ? 2 * kN1 : d.N2) * kBlockK * 2;  // both CTAs
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++kit) {
        const int st = kit % kPStages;
        const uint32_t ph = (kit / kPStages) & 1;
        if (!pwait(&sm.empty[st], ph ^ 1, &sm.abort, itimeout, status, 0x11000000u)) {
          ok = false;
          break;
        }
        uint8_t* As = a_tiles + (size_t)st * kPABytes;
        uint8_t* Bs = b_tiles + (size_t)st * kPBBytes;
        if (lead) mbar_arrive_expect_tx(&sm.full[st], bytes);
        const uint32_t fb = map_shared(&sm.full[st], 0);
        const int kx = kb * kBlockK;
        if (g1) {
          tma_load_2d_pair(As, &a.tm_x[cur.o], fb, kx, cur.row0);
          const int wrow = cur.li * d.F + cur.nt * kN1;
          tma_load_2d_pair(Bs, lead ? &a.tm_wg[cur.o] : &a.tm_wu[cur.o], fb, kx, wrow);
        } else {
          tma_load_2d_pair(As, &a.tm_h[cur.o], fb, kx, cur.row0);
          tma_load_2d_pair(Bs, &a.tm_wd[cur.o], fb, kx,
                           cur.li * d.D + cur.nt * d.N2 + (int)(crank * half_b2));
        }
      }
      if (!ok) break;
    }
    // Every copy this CTA issued has landed once the MMAs that read its stage
    // completed (the leader's commit arrives on both CTAs' empty barriers).
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = kit > (uint32_t)kPStages ? kit - kPStages : 0; i < kit; ++i) {
      volatile int never = 0;
      const long long left = itimeout - (long long)(globaltimer() - t0);
      pwait(&sm.empty[i % kPStages], (i / kPStages) & 1, &never, left > 0 ? left : 0, status,
            0x12000000u);
    }
  } else if (warp == 1 && lane == 0 && lead) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    uint32_t kit = 0;
    for (int it = 0;; ++it) {
      const int slot = it % kPRing;
      if (!pwait(&sm.qfull[slot], (it / kPRing) & 1, &sm.abort, itimeout, status, 0x20000000u))
        break;
      const PTask tk = sm.task[slot];
      mbar_arrive(&sm.qempty[slot]);
      if (tk.kind == kPEnd) break;
      const int acc = it & 1;
      if (!pwait(&sm.tempty[acc], ((it >> 1) & 1) ^ 1, &sm.abort, itimeout, status, 0x21000000u))
        break;
      tc_fence_after();
      const bool g1 = tk.kind == kPG1;
      const int nk = (g1 ? d.D : d.F) / kBlockK;
      const uint32_t idesc = idesc_bf16_f32(2 * kTileM, g1 ? 2 * kN1 : d.N2);
      const uint32_t dt = tmem_base + (uint32_t)(acc * kPAccCols);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++kit) {
        const int st = kit % kPStages;
        if (!pwait(&sm.full[st], (kit / kPStages) & 1, &sm.abort, itimeout, status, 0x22000000u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(a_tiles + (size_t)st * kPABytes);
        const uint32_t b0 = smem_u32(b_tiles + (size_t)st * kPBBytes);
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k)
          tc_mma_pair(dt, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                      (kb | k) != 0 ? 1u : 0u);
        tc_commit_pair(&sm.empty[st], 0x3);
      }
      if (!ok) break;
      tc_commit_pair(&sm.tfull[acc], 0x3);
    }
    // Every MMA issued completes before either CTA can release TMEM or exit.
    tc_commit_pair(&sm.drain, 0x1);
    volatile int never = 0;
    pwait(&sm.drain, 0, &never, itimeout, status, 0x23000000u);
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // Eight warps in two groups of four; each group holds all four TMEM lane
    // quarters and drains half of the accumulator's columns. One leader thread
    // performs every bounded wait and broadcasts the outcome through shared
    // memory, so all 256 threads take the same path through the named barrier.
    const bool leader = threadIdx.x == 32 * kEpiWarp0;
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int grp = (warp - kEpiWarp0) >> 2;  // column half
    const int r = q * 32 + lane;
    const uint32_t tempty_rank0[2] = {map_shared(&sm.tempty[0], 0), map_shared(&sm.tempty[1], 0)};
    for (int it = 0;; ++it) {
      const int slot = it % kPRing;
      if (leader) {
        const bool ok = pwait(&sm.qfull[slot], (it / kPRing) & 1, &sm.abort, itimeout, status,
                              0x30000000u);
        if (ok) {
          sm.etask = sm.task[slot];
          mbar_arrive(&sm.qempty[slot]);
        }
        sm.eok = ok;
      }
      epi_sync();
      if (!sm.eok) break;
      const PTask tk = sm.etask;
      if (tk.kind == kPEnd) break;
      const int e = tk.o * d.L + tk.li;
      const int rows_lim = __ldg(a.p.a[PA_EXPERT_START] + e) + __ldg(a.p.a[PA_ROWS_ALLOC] + e);
      const int acc = it & 1;
      if (leader)
        sm.eok = pwait(&sm.tfull[acc], (it >> 1) & 1, &sm.abort, itimeout, status, 0x31000000u);
      epi_sync();
      if (!sm.eok) break;
      tc_fence_after();
      const int grow = tk.row0 + r;
      const bool valid = tk.own >= 0 && grow < rows_lim;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kPAccCols);
      // Row offsets and column offsets are multiples of 64 bytes (D, F multiples of 128), so
      // the output's base alignment decides whether 32-byte stores are aligned.
      const bool v8ok = ((reinterpret_cast<uintptr_t>(tk.kind == kPG1 ? (const void*)a.h[tk.o]
                                                                     : (const void*)a.y[tk.o])) &
                         31) == 0;
      if (tk.kind == kPG1) {
        uint4* out = reinterpret_cast<uint4*>(a.h[tk.o] + (size_t)grow * d.F + tk.nt * kN1);
#pragma unroll 1
        for (int c = 2 * grp; c < 2 * grp + 2; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c * 32, g);
          tmem_ld32(tbase + kN1 + c * 32, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1v = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            // SiLU(g) u = g / (1 + e^-g) u. The fast division (an approximate reciprocal)
            // is far cheaper than the IEEE one, which made this loop the epilogue's cost,
            // and h is rounded to bf16 right after.
            const float a0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float a1 = __fdividef(g1v, 1.0f + __expf(-g1v)) * u1;
            packed[i] = pack_bf16x2(a0, a1);
          }
          if (valid && v8ok) {
            st_global_v8(out + c * 4, packed);
            st_global_v8(out + c * 4 + 2, packed + 8);
          } else if (valid) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              out[c * 4 + i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                          packed[4 * i + 3]);
          }
        }
      } else {
        uint4* out = reinterpret_cast<uint4*>(a.y[tk.o] + (size_t)grow * d.D + tk.nt * d.N2);
        const int nc = d.N2 / 64;  // 32-column chunks per group
#pragma unroll 1
        for (int c = grp * nc; c < (grp + 1) * nc; c += 2) {
          uint32_t v[32], w[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_ld32(tbase + (c + 1) * 32, w);
          tmem_ld_wait();
          uint32_t pv[16], pw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pv[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            pw[i] = pack_bf16x2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
          }
          if (valid && v8ok) {
            st_global_v8(out + c * 4, pv);
            st_global_v8(out + c * 4 + 2, pv + 8);
            st_global_v8(out + c * 4 + 4, pw);
            st_global_v8(out + c * 4 + 6, pw + 8);
          } else if (valid) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              out[c * 4 + i] = make_uint4(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              out[c * 4 + 4 + i] =
                  make_uint4(pw[4 * i], pw[4 * i + 1], pw[4 * i + 2], pw[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_global();
      epi_sync();
      if (leader) {
        if (lead) mbar_arrive(&sm.tempty[acc]); else mbar_arrive_cluster(tempty_rank0[acc]);
        if (tk.own >= 0) {
          if (tk.kind == kPG1) {
            red_release_add_u32(g1cnt + tk.own, 1u);
          } else {
            const int last = min(tk.row0 + kTileM, rows_lim) - 1;
            for (int b = tk.row0 / d.tb; b <= last / d.tb; ++b)
              red_release_add_u32(flags + ((size_t)tk.o * d.NBM + b) * d.nt2 + tk.nt, 1u);
            red_release_add_u32(queue + 3, 1u);  // output tiles finished (the scale's gate)
            span_end(a.p.span, kSpanLastTile);
          }
        }
      }
    }
  }

  // Both CTAs meet here: the leader's MMAs have drained (they read both CTAs'
  // shared memory and write both CTAs' TMEM) and every copy has landed.
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, 2 * kPAccCols);
  }
  if (threadIdx.x == 0) span_end(a.p.span);
}

}  // namespace

cudaError_t preload_producer_pair() {
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, ffn_pair_kernel<false>)) != cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, ffn_pair_kernel<true>)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(ffn_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)PairCfg<false>::kSmem)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(ffn_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)PairCfg<true>::kSmem);
}

namespace {
template <bool FUSED>
int max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(PairCfg<FUSED>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<FUSED>::kSmem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ffn_pair_kernel<FUSED>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}
}  // namespace

int producer_pair_max_clusters(bool fused) {
  return fused ? max_clusters<true>() : max_clusters<false>();
}

cudaError_t launch_producer_pair(const ProducerArgs& a, int grid, bool fused, cudaStream_t s) {
  grid = grid < 2 ? 2 : grid & ~1;
  if (fused)
    ffn_pair_kernel<true><<<grid, PairCfg<true>::kThreads, PairCfg<true>::kSmem, s>>>(a);
  else
    ffn_pair_kernel<false><<<grid, PairCfg<false>::kThreads, PairCfg<false>::kSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

// Persistent grouped expert-FFN producer (sm_103a: TMA + tcgen05 + TMEM).
//
// TileMoE notes (zhongzhuzhou.org), section 5.1: one persistent kernel covers
// every local expert; each CTA takes tiles of the remote-first schedule in
// order and, in the epilogue of every finished output tile, makes the tile
// globally visible and then sets that tile's device-resident ready flag
// (section 2.3: the epilogue is the natural place for the signal).
//
// Here the FFN is SiLU-gated and all W logical ranks share one launch:
//   GEMM1 tile (128 rows x 128 hidden columns): gate and up accumulate side by
//     side in one 128x256 fp32 TMEM accumulator; the epilogue writes
//     h = bf16(SiLU(g) * u) and counts the tile for its 128-row block.
//   GEMM2 tile (128 rows x N2 output columns): Y = bf16(h Wd^T); the epilogue
//     adds one release increment to the ready flag of every row band it covers.
// Tasks come from one atomic ticket counter. Tickets decode to scheduling
// units of up to kTileGroup tiles: a unit's GEMM1 tasks are emitted `lag`
// units ahead of its GEMM2 tasks. GEMM1 tasks are hidden-column-major inside the
// unit, so consecutive tickets reuse one gate/up weight tile from L2; GEMM2 tasks
// are tile-major, so a tile's hidden activations are read once while the
// expert's W_down tiles stay in L2. A GEMM2 task waits
// (bounded) until its block's GEMM1 tiles are all counted; the waits only ever
// point at lower tickets, which are held by running CTAs, so the kernel cannot
// deadlock.
//
// Warp roles: warp 0 lane 0 fetches tickets and issues TMA loads into a
// kStages-deep shared-memory ring; warp 1 lane 0 issues tcgen05.mma into one of
// two TMEM accumulators; warps 2-5 drain the accumulator (tcgen05.ld), apply
// the epilogue, store bf16 rows and publish the signal. Every wait is bounded
// by timeout_ns; on expiry the CTA records MOE_DEV_TIMEOUT, stops taking work,
// drains its own copies and MMAs and frees its TMEM.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kABytes = kTileM * kBlockK * 2;  // 16 KB
constexpr int kBBytes = 256 * kBlockK * 2;     // 32 KB (GEMM1: gate 128 rows + up 128 rows)
constexpr int kUnitCache = 4096;               // scheduling units kept in shared memory
constexpr int kAccCols = 256;                  // TMEM columns per accumulator

enum TaskKind : int { kEnd = -1, kG1 = 0, kG2 = 1 };

struct Task {
  int kind;
  int m;     // global tile index
  int nt;    // tile along F (GEMM1) or D (GEMM2)
  int o;     // owner rank
  int row0;  // first X row of the tile in the owner's buffer
  int li;    // local expert index
  int pad0, pad1;
};

struct Smem {
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[2], tempty[2];
  uint64_t qfull[kTaskRing], qempty[kTaskRing];
  uint64_t drain;
  Task task[kTaskRing];
  Task etask;  // the epilogue's copy of its current task
  int eok;     // outcome of the epilogue leader's last wait
  uint32_t tmem_base;
  int abort;
  int nunits;
  int unit_begin[kUnitCache + 1];
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kStages * (kABytes + kBBytes) +
                              sizeof(Smem);

__device__ __forceinline__ int unit_at(const Smem& sm, const int32_t* gub, int u) {
  return u <= kUnitCache ? sm.unit_begin[u] : gub[u];
}

// Tasks before unit u: GEMM1 tasks of units < u, GEMM2 tasks of units < u - lag.
__device__ __forceinline__ long long tasks_before(const Smem& sm, const int32_t* gub, int u,
                                                  int NU, int lag, int nt1, int nt2) {
  const int u1 = min(u, NU);
  const int u2 = max(0, min(u - lag, NU));
  return (long long)nt1 * unit_at(sm, gub, u1) + (long long)nt2 * unit_at(sm, gub, u2);
}

__device__ Task decode_ticket(const Smem& sm, const ProducerArgs& a, long long ticket) {
  const Dims& d = a.p.d;
  const int32_t* gub = a.p.a[PA_UNIT_BEGIN];
  const int NU = sm.nunits;
  const int NM = unit_at(sm, gub, NU);
  Task tk{};
  tk.kind = kEnd;
  const long long total = (long long)NM * (d.nt1 + d.nt2);
  if (ticket >= total || NU == 0) return tk;
  int lo = 0, hi = NU + a.lag - 1;  // largest u with tasks_before(u) <= ticket
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tasks_before(sm, gub, mid, NU, a.lag, d.nt1, d.nt2) <= ticket) lo = mid; else hi = mid - 1;
  }
  const int u = lo;
  long long r = ticket - tasks_before(sm, gub, u, NU, a.lag, d.nt1, d.nt2);
  const int sz1 = u < NU ? unit_at(sm, gub, u + 1) - unit_at(sm, gub, u) : 0;
  if (r < (long long)d.nt1 * sz1) {
    tk.kind = kG1;
    tk.m = unit_at(sm, gub, u) + (int)(r % sz1);
    tk.nt = (int)(r / sz1);
  } else {
    r -= (long long)d.nt1 * sz1;
    const int u2 = u - a.lag;
    const int sz2 = unit_at(sm, gub, u2 + 1) - unit_at(sm, gub, u2);
    (void)sz2;
    tk.kind = kG2;
    tk.m = unit_at(sm, gub, u2) + (int)(r / d.nt2);  // tile-major: a tile's hidden rows
    tk.nt = (int)(r % d.nt2);                         // stay in L2 for its nt2 tasks
  }
  const int tr = a.p.a[PA_TILE_ROW][tk.m];
  tk.o = tr >> 24;
  tk.row0 = tr & 0xFFFFFF;
  tk.li = a.p.a[PA_TILE_EXPERT][tk.m] - tk.o * d.L;
  return tk;
}

__global__ void __launch_bounds__(kProducerThreads, 1)
    ffn_producer_kernel(const __grid_constant__ ProducerArgs a) {
  extern __shared__ uint8_t smem_raw[];
  allow_dependent_launch();  // a scale launched behind this kernel may start beside it
  const Dims d = a.p.d;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* stage_base = smem_raw + pad;
  uint8_t* a_tiles = stage_base;                              // kStages x 16 KB
  uint8_t* b_tiles = stage_base + (size_t)kStages * kABytes;  // kStages x 32 KB
  Smem& sm = *reinterpret_cast<Smem*>(stage_base + (size_t)kStages * (kABytes + kBBytes));

  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  uint32_t* queue = reinterpret_cast<uint32_t*>(a.p.a[PA_QUEUE]);
  uint32_t* g1cnt = reinterpret_cast<uint32_t*>(a.p.a[PA_G1CNT]);
  uint32_t* flags = reinterpret_cast<uint32_t*>(a.p.a[PA_FLAGS]);
  // Waits on other CTAs (a block's GEMM1 tiles) are bounded by timeout_ns. Waits
  // inside the CTA (TMA landing, MMAs completing, task hand-offs) depend only on
  // this CTA's own progress and on at most one cross-CTA wait, so they get
  // timeout_ns + 4 s: they expire only if something is broken.
  const long long timeout = a.p.timeout_ns;
  const long long itimeout = a.p.timeout_ns + 4000000000LL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tfull[i], 1);
      mbar_init(&sm.tempty[i], 1);
    }
    for (int i = 0; i < kTaskRing; ++i) {
      mbar_init(&sm.qfull[i], 1);
      mbar_init(&sm.qempty[i], 2);  // the MMA thread and the epilogue leader
    }
    mbar_init(&sm.drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sm.abort = 0;
    sm.nunits = a.p.a[PA_TOTALS][2];
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, 2 * kAccCols);
  __syncthreads();
  {
    const int NU = sm.nunits;
    const int32_t* gub = a.p.a[PA_UNIT_BEGIN];
    for (int u = threadIdx.x; u <= min(NU, kUnitCache); u += blockDim.x) sm.unit_begin[u] = gub[u];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;
  if (threadIdx.x == 0) span_begin(a.p.span);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    for (int r = 0; r < d.W; ++r) {
      tma_prefetch_desc(&a.tm_x[r]);
      tma_prefetch_desc(&a.tm_h[r]);
      tma_prefetch_desc(&a.tm_wg[r]);
      tma_prefetch_desc(&a.tm_wu[r]);
      tma_prefetch_desc(&a.tm_wd[r]);
    }
    uint32_t kit = 0;
    long long next = atomicAdd(queue, 1u);
    for (int it = 0;; ++it) {
      const int slot = it % kTaskRing;
      const uint32_t qph = (it / kTaskRing) & 1;
      Task tk = decode_ticket(sm, a, next);
      if (tk.kind != kEnd && ld_relaxed_u32(status) != 0) tk.kind = kEnd;
      if (tk.kind != kEnd) next = atomicAdd(queue, 1u);
      if (tk.kind == kG2) {
        // Wait for every GEMM1 tile of this 128-row block (bounded).
        const uint32_t* c = g1cnt + tk.m;
        if (ld_acquire_u32(c) < (uint32_t)d.nt1) {
          const unsigned long long t0 = globaltimer();
          while (ld_acquire_u32(c) < (uint32_t)d.nt1) {
            if (ld_relaxed_u32(status) != 0) {
              tk.kind = kEnd;
              break;
            }
            if ((long long)(globaltimer() - t0) > timeout) {
              report_error(status, MOE_DEV_TIMEOUT, 0x40000000u | (uint32_t)tk.m);
              tk.kind = kEnd;
              break;
            }
            __nanosleep(64);
          }
        }
        fence_proxy_async_global();
      }
      if (!mbar_wait_bounded(&sm.qempty[slot], qph ^ 1, &sm.abort, itimeout, status, 0x10000000u))
        break;
      sm.task[slot] = tk;
      mbar_arrive(&sm.qfull[slot]);
      if (tk.kind == kEnd) break;

      const bool g1 = tk.kind == kG1;
      const int nk = (g1 ? d.D : d.F) / kBlockK;
      const uint32_t bytes = kABytes + (g1 ? 2 * kN1 : d.N2) * kBlockK * 2;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++kit) {
        const int st = kit % kStages;
        const uint32_t ph = (kit / kStages) & 1;
        if (!mbar_wait_bounded(&sm.empty[st], ph ^ 1, &sm.abort, itimeout, status, 0x11000000u)) {
          ok = false;
          break;
        }
        uint8_t* As = a_tiles + (size_t)st * kABytes;
        uint8_t* Bs = b_tiles + (size_t)st * kBBytes;
        mbar_arrive_expect_tx(&sm.full[st], bytes);
        const int kx = kb * kBlockK;
        if (g1) {
          tma_load_2d(As, &a.tm_x[tk.o], &sm.full[st], kx, tk.row0);
          const int wrow = tk.li * d.F + tk.nt * kN1;
          tma_load_2d(Bs, &a.tm_wg[tk.o], &sm.full[st], kx, wrow);
          tma_load_2d(Bs + kN1 * kBlockK * 2, &a.tm_wu[tk.o], &sm.full[st], kx, wrow);
        } else {
          tma_load_2d(As, &a.tm_h[tk.o], &sm.full[st], kx, tk.row0);
          tma_load_2d(Bs, &a.tm_wd[tk.o], &sm.full[st], kx, tk.li * d.D + tk.nt * d.N2);
        }
      }
      if (!ok) break;
    }
    // Let every copy this CTA issued land before the CTA can exit.
    for (uint32_t i = kit > (uint32_t)kStages ? kit - kStages : 0; i < kit; ++i) {
      volatile int never = 0;
      mbar_wait_bounded(&sm.full[i % kStages], (i / kStages) & 1, &never, itimeout, status,
                        0x12000000u);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t kit = 0;
    for (int it = 0;; ++it) {
      const int slot = it % kTaskRing;
      if (!mbar_wait_bounded(&sm.qfull[slot], (it / kTaskRing) & 1, &sm.abort, itimeout, status,
                             0x20000000u))
        break;
      const Task tk = sm.task[slot];
      mbar_arrive(&sm.qempty[slot]);
      if (tk.kind == kEnd) break;
      const int acc = it & 1;
      if (!mbar_wait_bounded(&sm.tempty[acc], ((it >> 1) & 1) ^ 1, &sm.abort, itimeout, status,
                             0x21000000u))
        break;
      tc_fence_after();
      const bool g1 = tk.kind == kG1;
      const int nk = (g1 ? d.D : d.F) / kBlockK;
      const uint32_t idesc = idesc_bf16_f32(kTileM, g1 ? 2 * kN1 : d.N2);
      const uint32_t dt = tmem_base + (uint32_t)(acc * kAccCols);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++kit) {
        const int st = kit % kStages;
        if (!mbar_wait_bounded(&sm.full[st], (kit / kStages) & 1, &sm.abort, itimeout, status,
                               0x22000000u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(a_tiles + (size_t)st * kABytes);
        const uint32_t b0 = smem_u32(b_tiles + (size_t)st * kBBytes);
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k)
          tc_mma(dt, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                 (kb | k) != 0 ? 1u : 0u);
        tc_commit(&sm.empty[st]);
      }
      if (!ok) break;
      tc_commit(&sm.tfull[acc]);
    }
    // Every MMA this thread issued completes before TMEM can be released.
    tc_commit(&sm.drain);
    volatile int never = 0;
    mbar_wait_bounded(&sm.drain, 0, &never, itimeout, status, 0x23000000u);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // One leader thread performs every bounded wait and broadcasts the outcome
    // through shared memory, so the 128 threads always take the same path
    // through the named barrier.
    const bool leader = threadIdx.x == 64;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    for (int it = 0;; ++it) {
      const int slot = it % kTaskRing;
      if (leader) {
        const bool ok = mbar_wait_bounded(&sm.qfull[slot], (it / kTaskRing) & 1, &sm.abort,
                                          itimeout, status, 0x30000000u);
        if (ok) {
          sm.etask = sm.task[slot];
          mbar_arrive(&sm.qempty[slot]);
        }
        sm.eok = ok;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (!sm.eok) break;
      const Task tk = sm.etask;
      if (tk.kind == kEnd) break;
      const int e = tk.o * d.L + tk.li;
      const int rows_lim = a.p.a[PA_EXPERT_START][e] + a.p.a[PA_ROWS_ALLOC][e];
      const int acc = it & 1;
      if (leader)
        sm.eok = mbar_wait_bounded(&sm.tfull[acc], (it >> 1) & 1, &sm.abort, itimeout, status,
                                   0x31000000u);
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (!sm.eok) break;
      tc_fence_after();
      const int grow = tk.row0 + r;
      const bool valid = grow < rows_lim;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kAccCols);
      // Each thread writes its row's 64-byte runs as two 32-byte stores (whole L2 sectors):
      // row and column offsets are multiples of 64 bytes (D, F multiples of 128), so the
      // output's base alignment decides; an unaligned base keeps 16-byte stores.
      const bool v8ok = ((reinterpret_cast<uintptr_t>(tk.kind == kG1 ? (const void*)a.h[tk.o]
                                                                    : (const void*)a.y[tk.o])) &
                         31) == 0;
      if (tk.kind == kG1) {
        uint4* out = reinterpret_cast<uint4*>(a.h[tk.o] + (size_t)grow * d.F + tk.nt * kN1);
#pragma unroll 1
        for (int c = 0; c < kN1 / 32; ++c) {
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
#pragma unroll 1
        for (int c = 0; c < d.N2 / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
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
      }
      tc_fence_before();
      fence_proxy_async_global();
      // All 128 threads' stores and TMEM reads precede the leader's signals.
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (leader) {
        mbar_arrive(&sm.tempty[acc]);
        if (tk.kind == kG1) {
          red_release_add_u32(g1cnt + tk.m, 1u);
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

  // All roles meet here; then TMEM is released by the warp that allocated it.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem_base, 2 * kAccCols);
  }
  if (threadIdx.x == 0) span_end(a.p.span);
}

}  // namespace

cudaError_t preload_producer() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, ffn_producer_kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(ffn_producer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemBytes);
}

cudaError_t launch_producer(const ProducerArgs& a, int grid, cudaStream_t s) {
  ffn_producer_kernel<<<grid, kProducerThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

// Shared definitions of the sm_103a expert-combine library: problem dimensions,
// workspace layout, device-side PTX wrappers and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_tsg.h"

namespace moe {

// ---------------------------------------------------------------------------
// Tiling constants of the producer (persistent tcgen05 FFN kernel).
// ---------------------------------------------------------------------------
constexpr int kTileM = 128;      // rows per producer tile (one tcgen05.mma M)
constexpr int kBlockK = 64;      // K elements per pipeline stage (128 B of bf16: one swizzle row)
constexpr int kN1 = 128;         // GEMM1 hidden columns per tile (gate and up each)
constexpr int kStages = 4;       // shared-memory pipeline depth
constexpr int kTaskRing = 4;     // task descriptors in flight inside one CTA
constexpr int kTileGroup = 32;   // tiles per scheduling unit at most (weight reuse in L2)
constexpr int kProducerThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kConsumerThreads = 32;         // one warp: lane 0 drives the bulk copies
constexpr int kChunkBytes = 20 * 1024;       // consumer copy chunk (one shared-memory slot)
constexpr int kChunkSlots = 6;               // 120 KB (+ the tail): one consumer CTA per SM
constexpr int kLoadsInFlight = 4;            // consumer bulk loads outstanding at most
constexpr size_t kConsumerSmemTail = 12 * 1024;  // barriers, counters and records after the slots
constexpr size_t kConsumerSmem = (size_t)kChunkSlots * kChunkBytes + kConsumerSmemTail;
constexpr int kSegRec = 8;                   // ints per consumer segment record
constexpr int kMaxSegChunks = 256;           // copy chunks one segment may have
constexpr int kSpanRing = 1024;              // per-combine device-clock records kept while timing
// One record of the span ring: eight u64 device-clock stamps (ns) of one combine.
enum SpanWord {
  kSpanProdStart = 0,    // ~(first producer CTA start), folded in with atomicMax
  kSpanProdEnd = 1,      // last producer CTA end
  kSpanScaleStart = 2,   // ~(first CTA start) of the scale (moe_scale or moe_scale_gated)
  kSpanScaleEnd = 3,     // last CTA end of the scale
  kSpanLastTile = 4,     // the producer's last finished output tile (its ready-flag release)
  kSpanConsStart = 5,    // ~(first CTA start) of the consumer kernel (not the fused copy warp)
  kSpanConsEnd = 6,      // last CTA end of the consumer kernel
  kSpanCombineWords = 7, // words [0, 7) are zeroed by each combine
  kSpanGateStart = 7,    // ~(first CTA start) of the gate before this combine (zeroed by it)
  kSpanGateEnd = 8,      // last CTA end of that gate
  kSpanGatherStart = 9,  // ~(first CTA start) of the layout gather before this combine
  kSpanGatherEnd = 10,   // last CTA end of that gather (both zeroed by the plan build)
  kSpanWords = 12
};

// ---------------------------------------------------------------------------
// Dimensions derived from a configuration (host and device).
// ---------------------------------------------------------------------------
struct Dims {
  int W, L, E, k, T, D, F, tb, mgb;
  int TW;        // 32-bit words per (expert, rank) token bitmap
  int RM;        // worst-case rows of one owner's X
  int NBM;       // worst-case bands per owner (RM / tb)
  int NMM;       // worst-case producer tiles per owner
  int N2;        // GEMM2 output columns per tile (256 or 128)
  int nt1, nt2;  // tiles along F (GEMM1) and along D (GEMM2)
  int parts;     // producer tiles touching one band (tb/128, at least 1)
  int rpc;       // rows per consumer copy chunk
};

// Scheduling units of one rank and phase (remote or local tiles) at most. A unit
// starts only at the start of an expert's run of tiles (at most L runs per phase) or
// inside a run longer than kTileGroup (a new unit every kTileGroup tiles at most), so
// a phase of n <= NMM tiles has at most L + n / kTileGroup + 1 units.
__host__ __device__ inline int unit_cap(const Dims& d) { return d.L + d.NMM / kTileGroup + 1; }

// Fields of the plan workspace, in placement order. The public moe_field enum
// exposes a subset; the rest are internal.
enum PlanArray {
  PA_STATUS = 0, PA_TOTALS,
  // zeroed at the start of every combine (one memset):
  PA_QUEUE, PA_G1CNT, PA_FLAGS, PA_GROUP_DONE, PA_GROUP_SIG,
  // zeroed at the start of every plan build (and of every gate, whose routing tail
  // fills it):
  PA_BITMAP,
  // plain arrays:
  PA_WPRE, PA_CNT, PA_GROUP_START, PA_RECV_OFF,
  PA_EXPERT_START, PA_ROWS_ALLOC, PA_NB, PA_NRB,
  PA_RANK_ROWS, PA_RANK_NB, PA_RANK_NREMOTE, PA_RECV_ROWS, PA_RANK_NSEG,
  PA_BAND_EXPERT, PA_BAND_DST, PA_BAND_VALID, PA_BAND_DST_ROW, PA_BAND_TILE,
  PA_SCHED, PA_SEG_FIRST, PA_SEG_NB, PA_SEG_GIDX, PA_GROUP_NSEG,
  PA_RANK_TILES, PA_TILE_ROW, PA_TILE_EXPERT, PA_UNIT_BEGIN, PA_SEG_ORDER,
  PA_SEG_REC, PA_GROUP_NCHUNK,
  PA_XSRC, PA_SCALE_SRC,
  PA_PAIR, PA_PAIR_UNIT_BEGIN,
  PA_SPANS,  // [kSpanRing][kSpanWords] u64: device-clock records of each combine while timing
  PA_XPREV,  // [W][RM] what each X row held after the last gather: token, -1 zero, else unknown
  PA_CHUNK_T,  // [chunks] u64: device clock when each copy chunk had landed (timing on)
  PA_CHUNK_REC,  // [chunks] segment record (consumer order) of every copy chunk
  PA_UNIT_TMP,   // [2][W][2][unit_cap] plan-internal: each unit's first tile in its rank's
                 // phase, then its position in the global tile order
  PA_PAIR_RUN,   // [pairs] the pair's run of one expert in its unit: first pair's offset in
                 // the unit + 2^16 * the run's pairs
  PA_COUNT
};

struct PlanPtrs {
  int32_t* a[PA_COUNT];
  size_t count[PA_COUNT];
};

// Byte offsets of the per-rank workspace.
struct RankLayout {
  size_t x_off, h_off, y_off, bytes;
};

// Host helpers (api.cu).
int dims_from_cfg(const moe_cfg* cfg, Dims* d);
size_t plan_layout(const Dims& d, size_t* offsets, size_t* counts);  // returns total bytes
RankLayout rank_layout(const Dims& d);

// Kernel parameters that the host fills per call.
struct DevPlan {
  Dims d;
  int32_t* a[PA_COUNT];
  long long timeout_ns;
  // Timing on: this combine's record of the span ring (kSpanWords u64, zeroed by the
  // host) and the chunk landing stamps; both null otherwise.
  unsigned long long* span;
  unsigned long long* chunk_t;
};

// ---------------------------------------------------------------------------
// Launchers (defined next to their kernels).
// ---------------------------------------------------------------------------
// Loads every kernel's module and sets its shared-memory limit. With lazy module
// loading, the first launch of a kernel may wait for kernels already running; the
// producer's first launch would then wait for a consumer that spins on the
// producer's flags. Plan creation therefore loads all kernels up front.
cudaError_t preload_producer();
cudaError_t preload_consumer();
cudaError_t preload_plan();
cudaError_t preload_route_scale();
cudaError_t launch_route(const DevPlan& p, const float* logits, const int32_t* forced,
                         int32_t* ids, float* w, cudaStream_t s);
// marked: the token bitmaps are already in the plan (the gate's routing tail set
// them), so the bitmap kernel is skipped.
cudaError_t launch_plan(const DevPlan& p, const int32_t* ids, cudaStream_t s, bool marked = false);
cudaError_t launch_gather(const DevPlan& p, const __nv_bfloat16* const* x,
                          __nv_bfloat16* const* xbuf, int num_sms, cudaStream_t s);

// Gate: router GEMM (tcgen05) fused with softmax and top-k. E <= kGateMaxE.
constexpr int kGateMaxE = 256;
struct GateArgs {
  CUtensorMap tm_x[MOE_MAX_RANKS];  // rank s's tokens [T][D], boxes of 128 rows
  CUtensorMap tm_r;                 // router [E][D], boxes of npad rows
  const int32_t* forced;            // [W][T][k] or null
  int32_t* ids;                     // [W][T][k]
  float* w;                         // [W][T][k]
  float* logits;                    // [W][T][E] or null
  DevPlan p;
  int npad;    // MMA N: E rounded up to 32
  int splits;  // CTAs of one cluster sharing a token tile, each summing a K range
  int rows;    // tokens per tile: a multiple of 8, at most 128 (the x maps' box height)
};
cudaError_t preload_gate();
// Clusters of `splits` CTAs (1, 2, 4 or 8) resident at once on an idle GPU, for E
// experts (0: that split cannot be launched).
int gate_clusters(int E, int splits);
cudaError_t launch_gate(const GateArgs& a, cudaStream_t s);

// The gate for E <= 16 with the token rows streamed into registers (gate_rows.cu).
struct GateRowsArgs {
  const __nv_bfloat16* x[MOE_MAX_RANKS];  // rank s's tokens [T][D]
  const __nv_bfloat16* router;            // [E][D]
  const int32_t* forced;                  // [W][T][k] or null
  int32_t* ids;                           // [W][T][k]
  float* w;                               // [W][T][k]
  float* logits;                          // [W][T][E] or null
  DevPlan p;
  int rows;     // tokens per CTA, at most 128 (CTA j of rank s: tokens [j*rows, ...))
  int kslices;  // warps sharing a 16-token group, each a contiguous range of 64 columns
};
cudaError_t preload_gate_rows();
// Whether the kernel takes E experts of D columns (E <= 16, D a multiple of 64).
bool gate_rows_fits(int E, int D);
// Tokens per CTA and K slices for T tokens per rank on W ranks and num_sms SMs; with
// `beside`, CTAs small enough to share an SM with a running producer CTA.
void gate_rows_shape(int W, int T, int E, int D, int num_sms, bool beside, int* rows,
                     int* kslices);
cudaError_t launch_gate_rows(const GateRowsArgs& a, cudaStream_t s);

struct ProducerArgs {
  CUtensorMap tm_x[MOE_MAX_RANKS];
  CUtensorMap tm_h[MOE_MAX_RANKS];
  CUtensorMap tm_wg[MOE_MAX_RANKS];
  CUtensorMap tm_wu[MOE_MAX_RANKS];
  CUtensorMap tm_wd[MOE_MAX_RANKS];
  __nv_bfloat16* h[MOE_MAX_RANKS];
  __nv_bfloat16* y[MOE_MAX_RANKS];
  __nv_bfloat16* recv[MOE_MAX_RANKS];  // receive buffers (the fused pair producer copies into them)
  DevPlan p;
  int lag;  // scheduling units between a unit's GEMM1 tiles and its GEMM2 tiles
};
cudaError_t launch_producer(const ProducerArgs& a, int grid, cudaStream_t s);
// CTA-pair producer (clusters of two, tcgen05 cta_group::2); grid is rounded down
// to an even count. Its tm_wd maps use boxes of N2/2 rows.
cudaError_t preload_producer_pair();
// Clusters of two resident at once on an idle GPU (0: unknown).
int producer_pair_max_clusters(bool fused);
// fused: the variant whose every CTA also runs the combine copy in one warp.
cudaError_t launch_producer_pair(const ProducerArgs& a, int grid, bool fused, cudaStream_t s);

struct ConsumerArgs {
  const __nv_bfloat16* y[MOE_MAX_RANKS];
  __nv_bfloat16* recv[MOE_MAX_RANKS];
  DevPlan p;
};
cudaError_t launch_consumer(const ConsumerArgs& a, int grid, cudaStream_t s);

struct ScaleArgs {
  const __nv_bfloat16* recv[MOE_MAX_RANKS];
  const __nv_bfloat16* y[MOE_MAX_RANKS];
  __nv_bfloat16* out[MOE_MAX_RANKS];
  const float* w;
  DevPlan p;
};
cudaError_t launch_scale(const ScaleArgs& a, int num_sms, cudaStream_t s);
// The scale overlapped with the kernel before it on the stream (a programmatic
// dependent launch): its per-token waits on group signals and ready flags.
cudaError_t launch_scale_gated(const ScaleArgs& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A kernel's span (timing on): the first CTA's start (stored complemented, so that
// atomicMax keeps the earliest) and the last CTA's end, in the combine's span record.
__device__ __forceinline__ void span_begin(unsigned long long* span, int word = kSpanProdStart) {
  if (span != nullptr) atomicMax(span + word, ~globaltimer());
}
__device__ __forceinline__ void span_end(unsigned long long* span, int word = kSpanProdEnd) {
  if (span != nullptr) atomicMax(span + word, globaltimer());
}

// Lets the kernel launched after this one on the stream with programmatic stream
// serialization start once every CTA of this grid has executed it (or exited); that
// kernel synchronises with this one only through device-memory flags.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// First error wins; detail is written by the same winner.
__device__ __forceinline__ void report_error(uint32_t* status, uint32_t code, uint32_t detail) {
  if (atomicCAS(status, 0u, code) == 0u) {
    atomicExch(status + 1, detail);
  }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
// Orders this thread's generic-proxy global accesses with its async-proxy (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase (try_wait may suspend the thread for a while).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false (and records a timeout) when the deadline passes
// or when another role of the CTA has already given up (*abort set).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, long long timeout_ns,
                                                  uint32_t* status, uint32_t detail) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((long long)(globaltimer() - t0) > timeout_ns) {
      report_error(status, MOE_DEV_TIMEOUT, detail);
      *abort = 1;
      return false;
    }
  }
}

// --- TMA ------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Untiled bulk copies (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --- thread-block clusters ------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Every thread of every CTA of the cluster; orders shared-memory writes before the
// barrier with reads of any CTA after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// 16-byte load from the shared memory of a CTA of the cluster (cl_addr 16-byte aligned).
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t cl_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cl_addr)
               : "memory");
  return v;
}

// --- tcgen05 --------------------------------------------------------------
// Shared-memory matrix descriptor for a K-major operand stored by TMA with the
// 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, 16-byte units
  d |= (uint64_t)1 << 16;                    // leading-dimension offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride-dimension offset: 1024 B
  d |= (uint64_t)1 << 46;                    // descriptor version of tcgen05
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}
// Instruction descriptor: bf16 A and B, fp32 accumulator, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// One 32-byte store (a whole L2 sector); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i receives lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32,
// at most 1024). `scratch` holds 33 ints of shared memory. Returns the exclusive
// prefix; *total receives the block sum. Every thread must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) scratch[lane] = s;  // inclusive warp totals
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  const int base = wid > 0 ? scratch[wid - 1] : 0;
  const int tot = scratch[32];
  __syncthreads();
  *total = tot;
  return base + x - v;
}

#endif  // __CUDACC__

}  // namespace moe

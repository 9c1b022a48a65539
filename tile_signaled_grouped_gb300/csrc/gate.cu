// Gate: the router GEMM on the tensor cores, fused with the softmax and the top k.
//
// TileMoE notes (zhongzhuzhou.org), section 2.1 (a small gating network scores
// every token against the E experts) and 2.2 step 1 (every rank gates its own
// tokens). The router is one bias-free linear layer, logits = x W_r^T with W_r
// [E][D] held alike by every rank; then each token's softmax and top k exactly as
// the routing kernel takes them (route_topk.cuh). The logits never travel through
// HBM unless the caller asks for them.
//
// Work split. A token tile is 128 rows of one rank (the MMA's M); its scores are
// one tcgen05.mma accumulator of 128 x npad fp32 (npad = E rounded up to 32, at
// most 256 columns of TMEM). With few tiles (large E comes with few tokens per
// rank in the page's shapes) a cluster of `splits` CTAs shares a tile, each CTA
// summing one contiguous range of the K blocks into its own TMEM. Each CTA drains
// its partial to shared memory; after a cluster barrier CTA r owns rows
// [r*128/splits, (r+1)*128/splits) of the tile and adds the partials of all CTAs
// in CTA order (a fixed order: the result does not depend on timing) with 16-byte
// loads through distributed shared memory, all of them issued before the sums.
//
// Routing (route_topk.cuh). With E <= 32 each thread takes one token and holds its
// scores in registers (PER = E rounded up to 8, 16 or 32): no lane exchanges at
// all. Above, a warp takes one token, each lane holding PER = 2, 4 or 8 of its
// scores, and the maximum and the argmax of each of the k rounds are full-warp
// reductions. The 16 warps route 16 tokens at once (each a chain of dependent
// reductions, so more warps in flight hide more of their latency).
//
// Roles (512 threads): warp 0 lane 0 issues the TMA loads of x and W_r (stages of
// 64 K columns, 128-byte swizzle, as many as fit in 192 KB: 8 for E <= 64, 4 for
// E > 192); warp 1 lane 0 issues the MMAs; warps 8-15
// drain TMEM (lane quarter = warp & 3, alternate 32-column chunks per warp pair).
// All sixteen warps reduce and route.
//
// TMEM: the CTA allocates a power of two >= npad columns (at most 256). The stage
// buffers take more than half of an SM's shared memory, so one CTA runs per SM and
// an allocation never waits on another CTA.
// Every wait is on this CTA's own copies and MMAs, bounded by timeout_ns + 4 s.
#include "moe_common.cuh"
#include "route_topk.cuh"

namespace moe {
namespace {

constexpr int kGateThreads = 512;
constexpr int kGateDrainWarp0 = 8;  // warps 8-15: two per TMEM lane quarter
constexpr int kGateMaxStages = 8;
constexpr uint32_t kGateStageBudget = 192 * 1024;
constexpr uint32_t kGateABytes = (uint32_t)kTileM * kBlockK * 2;  // 16 KB of x per stage

__host__ __device__ constexpr uint32_t gate_stage_bytes(int npad) {
  return kGateABytes + (uint32_t)npad * kBlockK * 2;
}
// Floats per partial row: 16-byte aligned rows for the cluster loads.
__host__ __device__ constexpr uint32_t gate_part_stride(int npad) { return (uint32_t)npad + 4; }
// Pipeline depth: the stages that fit in the budget, at most 8.
__host__ __device__ constexpr int gate_stages(int npad) {
  return kGateStageBudget / gate_stage_bytes(npad) < (uint32_t)kGateMaxStages
             ? (int)(kGateStageBudget / gate_stage_bytes(npad))
             : kGateMaxStages;
}
__host__ __device__ constexpr size_t gate_smem_bytes(int npad) {
  return 1024 /*alignment slack*/ +
         ((size_t)gate_stages(npad) * gate_stage_bytes(npad) >
                  (size_t)kTileM * gate_part_stride(npad) * 4
              ? (size_t)gate_stages(npad) * gate_stage_bytes(npad)
              : (size_t)kTileM * gate_part_stride(npad) * 4);
}
__host__ __device__ constexpr uint32_t gate_tmem_cols(int npad) {
  return npad <= 32 ? 32u : npad <= 64 ? 64u : npad <= 128 ? 128u : 256u;
}
static_assert(gate_smem_bytes(kGateMaxE) <= 227 * 1024, "gate shared memory");
constexpr bool gate_one_cta_per_sm() {
  for (int n = 32; n <= kGateMaxE; n += 32)
    if (gate_stages(n) < 4 || gate_smem_bytes(n) <= 114 * 1024) return false;
  return true;
}
static_assert(gate_one_cta_per_sm(), "one CTA per SM, with at least four stages");

struct GSmem {
  alignas(8) uint64_t full[kGateMaxStages];
  alignas(8) uint64_t empty[kGateMaxStages];
  alignas(8) uint64_t done;
  uint32_t tmem;
  int abort;
};

template <int G, int PER>
__global__ void __launch_bounds__(kGateThreads, 1) gate_kernel(const __grid_constant__ GateArgs a) {
  extern __shared__ uint8_t gate_smem_raw[];
  __shared__ GSmem sm;
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(gate_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Dims d = a.p.d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.splits;
  const int npad = a.npad;
  const int crank = (int)(blockIdx.x % (unsigned)C);  // cluster dims (C, 1, 1)
  const int tile = (int)(blockIdx.x / (unsigned)C);
  const int rows = a.rows;  // tokens of this tile (the MMA computes 128 rows; the rest is void)
  const int tpr = (d.T + rows - 1) / rows;
  const int s = tile / tpr;
  const int t0 = (tile % tpr) * rows;
  const int nk = d.D / kBlockK;
  const int kb0 = crank * nk / C, kb1 = (crank + 1) * nk / C;
  const int nkl = kb1 - kb0;
  const uint32_t stage_bytes = gate_stage_bytes(npad);
  const uint32_t tx_bytes = (uint32_t)rows * kBlockK * 2 + (uint32_t)npad * kBlockK * 2;
  const int S = gate_stages(npad);
  const uint32_t ncols = gate_tmem_cols(npad);
  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  const long long itimeout = a.p.timeout_ns + 4000000000LL;

  // The TMA thread initialises the barriers and issues the first S stages' loads at
  // once (every stage starts free), before the CTA waits for its TMEM allocation.
  const int early = nkl < S ? nkl : S;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.done, 1);
    sm.abort = 0;
    span_begin(a.p.span, kSpanGateStart);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&a.tm_x[s]);
    tma_prefetch_desc(&a.tm_r);
    for (int i = 0; i < early; ++i) {
      uint8_t* As = base + (size_t)i * stage_bytes;
      mbar_arrive_expect_tx(&sm.full[i], tx_bytes);
      const int kx = (kb0 + i) * kBlockK;
      tma_load_2d(As, &a.tm_x[s], &sm.full[i], kx, t0);
      tma_load_2d(As + kGateABytes, &a.tm_r, &sm.full[i], kx, 0);
    }
  }
  if (warp == 1) tmem_alloc(&sm.tmem, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA
    int i = early;
    for (; i < nkl; ++i) {
      const int st = i % S;
      if (!mbar_wait_bounded(&sm.empty[st], ((i / S) & 1) ^ 1, &sm.abort, itimeout,
                             status, 0x50000000u))
        break;
      uint8_t* As = base + (size_t)st * stage_bytes;
      mbar_arrive_expect_tx(&sm.full[st], tx_bytes);
      const int kx = (kb0 + i) * kBlockK;
      tma_load_2d(As, &a.tm_x[s], &sm.full[st], kx, t0);
      tma_load_2d(As + kGateABytes, &a.tm_r, &sm.full[st], kx, 0);
    }
    // Every copy issued lands before the CTA moves on.
    for (int j = i > S ? i - S : 0; j < i; ++j) {
      volatile int never = 0;
      mbar_wait_bounded(&sm.full[j % S], (j / S) & 1, &never, itimeout,
                        status, 0x51000000u);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA
    const uint32_t idesc = idesc_bf16_f32(kTileM, npad);
    for (int i = 0; i < nkl; ++i) {
      const int st = i % S;
      if (!mbar_wait_bounded(&sm.full[st], (i / S) & 1, &sm.abort, itimeout, status,
                             0x52000000u))
        break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(base + (size_t)st * stage_bytes);
      const uint32_t b0 = a0 + kGateABytes;
#pragma unroll
      for (int k = 0; k < kBlockK / 16; ++k)
        tc_mma(tmem, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
               (i | k) != 0 ? 1u : 0u);
      tc_commit(&sm.empty[st]);
    }
    // Arrives when every MMA above has completed (at once if there was none).
    if (nkl > 0) tc_commit(&sm.done); else mbar_arrive(&sm.done);
  } else if (warp >= kGateDrainWarp0) {
    // ------------------------------------------------------------ TMEM drain
    // Row q*32 + lane of the accumulator into this CTA's partial rows. The
    // stage buffers are free once `done` has fired: every copy was consumed.
    volatile int never = 0;
    const bool ok = mbar_wait_bounded(&sm.done, 0, &never, itimeout, status, 0x53000000u);
    tc_fence_after();
    const int q = warp & 3;
    const int r = q * 32 + lane;
    float4* row = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) +
                                            (size_t)r * gate_part_stride(npad));
    for (int c = (warp - kGateDrainWarp0) >> 2; c < npad / 32; c += 2) {
      uint32_t v[32];
      if (nkl > 0 && ok) {
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        row[c * 8 + j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                     __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
    }
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync_all();  // every CTA's partial sums are in its shared memory
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, ncols);
  }

  const int R = rows / C;  // rows this CTA routes: [crank * R, crank * R + R)
  const uint32_t stride = gate_part_stride(npad);
  float* part = reinterpret_cast<float*>(base);
  if (C > 1) {
    // ---------------------------------------------------------- K-split sum
    // Element (r, 4 columns) of the owned rows: the C partials, CTA 0 first, summed
    // into this CTA's own copy of the row (only this CTA reads its owned rows).
    const int n4 = npad / 4;
    uint32_t pb[8];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) pb[cc] = cc < C ? map_shared(base, (uint32_t)cc) : 0u;
    for (int idx = threadIdx.x; idx < R * n4; idx += kGateThreads) {
      const int r = crank * R + idx / n4;
      const uint32_t off = 4u * ((uint32_t)r * stride + 4u * (uint32_t)(idx % n4));
      float4 p[8];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        if (cc < C) p[cc] = ld_cluster_v4(pb[cc] + off);
      float4 acc = p[0];
#pragma unroll
      for (int cc = 1; cc < 8; ++cc)
        if (cc < C) {
          acc.x += p[cc].x;
          acc.y += p[cc].y;
          acc.z += p[cc].z;
          acc.w += p[cc].w;
        }
      *reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(part) + off) = acc;
    }
    __syncwarp();
    cluster_sync_all();  // every pull is done: no CTA reads another's memory from here
  }

  // ------------------------------------------------------------ route
  {
    const int lig = G == 1 ? 0 : lane;
    const int first = G == 1 ? (int)threadIdx.x : warp;
    const int step = G == 1 ? kGateThreads : kGateThreads / 32;
    for (int rr = first; rr < R; rr += step) {
      const int r = crank * R + rr;
      const int t = t0 + r;
      if (t >= d.T) break;  // the same for the whole group
      const size_t tok = (size_t)s * d.T + t;
      const float* row = part + (size_t)r * stride;
      float v[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lig + G * i;
        v[i] = e < d.E ? row[e] : -INFINITY;
        if (e < d.E && a.logits != nullptr) a.logits[tok * d.E + e] = v[i];
      }
      const TokenMark mk{reinterpret_cast<uint32_t*>(a.p.a[PA_BITMAP]), (size_t)d.W * d.TW,
                         (size_t)s * d.TW + (t >> 5), 1u << (t & 31)};
      route_group<G, PER>(v, d.E, d.k, a.forced != nullptr ? a.forced + tok * d.k : nullptr,
                          a.ids + tok * d.k, a.w + tok * d.k, lig,
                          a.forced != nullptr ? nullptr : &mk);
      if (a.forced != nullptr) mark_token<G>(a.p, a.ids, a.forced, tok, s, t, lig, status);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) span_end(a.p.span, kSpanGateEnd);
}

template <int G, int PER>
cudaError_t launch_gate_gp(const GateArgs& a, int tiles, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * a.splits), 1, 1);
  cfg.blockDim = dim3(kGateThreads, 1, 1);
  cfg.dynamicSmemBytes = gate_smem_bytes(a.npad);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gate_kernel<G, PER>, a);
}

template <int G, int PER>
int clusters_gp(int npad, int splits) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits, 1, 1);
  cfg.blockDim = dim3(kGateThreads, 1, 1);
  cfg.dynamicSmemBytes = gate_smem_bytes(npad);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gate_kernel<G, PER>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  return n;
}

}  // namespace

// The instantiation for E experts: one thread per token up to 32 experts, a warp
// per token above. CALL(G, PER) is expanded with the kernel's template arguments.
#define MOE_GATE_DISPATCH(E, CALL)                 \
  ((E) <= 8     ? CALL(1, 8)                       \
   : (E) <= 16  ? CALL(1, 16)                      \
   : (E) <= 32  ? CALL(1, 32)                      \
   : (E) <= 64  ? CALL(32, 2)                      \
   : (E) <= 128 ? CALL(32, 4)                      \
                : CALL(32, 8))

cudaError_t preload_gate() {
  const int smem = (int)gate_smem_bytes(kGateMaxE);
#define MOE_GATE_SET(G, PER) \
  cudaFuncSetAttribute(gate_kernel<G, PER>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
  const cudaError_t e[6] = {MOE_GATE_SET(1, 8),  MOE_GATE_SET(1, 16), MOE_GATE_SET(1, 32),
                            MOE_GATE_SET(32, 2), MOE_GATE_SET(32, 4), MOE_GATE_SET(32, 8)};
#undef MOE_GATE_SET
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

int gate_clusters(int E, int splits) {
#define MOE_GATE_CLUSTERS(G, PER) clusters_gp<G, PER>((E + 31) / 32 * 32, splits)
  return MOE_GATE_DISPATCH(E, MOE_GATE_CLUSTERS);
#undef MOE_GATE_CLUSTERS
}

cudaError_t launch_gate(const GateArgs& a, cudaStream_t s) {
  const Dims& d = a.p.d;
  const int tiles = d.W * ((d.T + a.rows - 1) / a.rows);
#define MOE_GATE_LAUNCH(G, PER) launch_gate_gp<G, PER>(a, tiles, s)
  return MOE_GATE_DISPATCH(d.E, MOE_GATE_LAUNCH);
#undef MOE_GATE_LAUNCH
}

#undef MOE_GATE_DISPATCH

}  // namespace moe

// Gate routing and the gated weighted sum (scale).
//
// TileMoE notes (zhongzhuzhou.org), section 2.1 and 2.2 steps 1 and 5: the
// router forms a probability distribution over the E experts per token and
// keeps the top k; the owner rank combines the k expert outputs of a token
// with the gate weights.
#include <algorithm>

#include "moe_common.cuh"
#include "route_topk.cuh"

namespace moe {
namespace {

// One warp per token: its E logits (fp32) through route_group. Each lane holds PER
// logits (E <= 32 * PER); the launcher picks the smallest PER.
template <int PER>
__global__ void __launch_bounds__(256) route_kernel(DevPlan p, const float* __restrict__ logits,
                                                    const int32_t* __restrict__ forced,
                                                    int32_t* __restrict__ ids,
                                                    float* __restrict__ w) {
  const Dims d = p.d;
  const int lane = threadIdx.x & 31;
  const int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tok >= d.W * d.T) return;
  const float* lg = logits + (size_t)tok * d.E;
  float v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < d.E ? lg[e] : -INFINITY;
  }
  route_group<32, PER>(v, d.E, d.k, forced != nullptr ? forced + (size_t)tok * d.k : nullptr,
                       ids + (size_t)tok * d.k, w + (size_t)tok * d.k, lane);
}

// Scale: out_s[t] = sum_j w_j * row_j, fp32 in slot order, bf16 out, by whole warps:
// lane j < k holds slot j's source (scale map) and weight. A round covers 32 * CPL
// 16-byte chunks of the output row (CPL per lane) and walks the slots in groups of SG,
// loading a group's SG * CPL chunks per lane before accumulating, so every lane keeps
// eight independent 16-byte loads in flight: SG = 4, CPL = 2 for k >= 4; SG = 2,
// CPL = 4 for k < 4 (for k = 1 half of them; measured faster than SG = 1, CPL = 8, whose
// 95 registers leave two CTAs per SM). Each element's sum is its k products added in
// slot order (a group's unused slots add 0 * 0).
__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    acc[2 * q] = fmaf(w, f.x, acc[2 * q]);
    acc[2 * q + 1] = fmaf(w, f.y, acc[2 * q + 1]);
  }
}

// One round of token (s, t): chunks c0 + 32 i + lane, i < CPL. L2ONLY reads the rows
// from L2 (__ldcg) for rows that a kernel still running beside this one has written
// (the read-only and L1 paths are not kept coherent with such writes); otherwise
// through the read-only path.
template <int SG, int CPL, bool L2ONLY>
__device__ __forceinline__ void scale_round(const ScaleArgs& a, const Dims& d, int s, int t,
                                            int src_l, float w_l, int lane, int c0) {
  const int n16 = d.D / 8;
  float acc[CPL][8];
#pragma unroll
  for (int i = 0; i < CPL; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  for (int j0 = 0; j0 < d.k; j0 += SG) {
    uint4 v[SG][CPL];
    float wj[SG];
#pragma unroll
    for (int q = 0; q < SG; ++q) {
      const int j = j0 + q;
      const int sj = __shfl_sync(0xffffffffu, src_l, j & 31);
      wj[q] = __shfl_sync(0xffffffffu, w_l, j & 31);
      // Slots past k, and invalid routing slots (reported by the plan), add nothing.
      const bool live = j < d.k && sj != INT_MIN;
      if (!live) wj[q] = 0.f;
      const uint4* row = reinterpret_cast<const uint4*>(
          sj >= 0 ? a.recv[s] + (size_t)sj * d.D : a.y[s] + (size_t)(-sj - 1) * d.D);
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int c = c0 + 32 * i + lane;
        v[q][i] = !(live && c < n16) ? make_uint4(0, 0, 0, 0)
                  : L2ONLY           ? __ldcg(row + c)
                                     : __ldg(row + c);
      }
    }
#pragma unroll
    for (int q = 0; q < SG; ++q)
#pragma unroll
      for (int i = 0; i < CPL; ++i) fma_bf16x8(acc[i], wj[q], v[q][i]);
  }
  uint4* out = reinterpret_cast<uint4*>(a.out[s] + (size_t)t * d.D);
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = c0 + 32 * i + lane;
    if (c < n16)
      out[c] = make_uint4(pack_bf16x2(acc[i][0], acc[i][1]), pack_bf16x2(acc[i][2], acc[i][3]),
                          pack_bf16x2(acc[i][4], acc[i][5]), pack_bf16x2(acc[i][6], acc[i][7]));
  }
}

// After the combine. A task is one round of one token; warps take tasks token-major,
// so a long row spreads over several warps (a 14 KB row with k = 8 over 14), and
// every task's sources and weights are fetched while the previous task is summed.
template <int SG, int CPL>
__global__ void __launch_bounds__(256) scale_kernel(const __grid_constant__ ScaleArgs a) {
  const Dims d = a.p.d;
  const int lane = threadIdx.x & 31;
  const int n16 = d.D / 8;
  const int nblk = (n16 + 32 * CPL - 1) / (32 * CPL);
  const int ntask = d.W * d.T * nblk;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  int task = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (threadIdx.x == 0) span_begin(a.p.span, kSpanScaleStart);
  int src_n = INT_MIN;
  float w_n = 0.f;
  if (task < ntask && lane < d.k) {
    const int tok = task / nblk;
    src_n = __ldg(a.p.a[PA_SCALE_SRC] + (size_t)tok * d.k + lane);
    w_n = __ldg(a.w + (size_t)tok * d.k + lane);
  }
  for (; task < ntask; task += warps) {
    const int src_l = src_n;
    const float w_l = w_n;
    const int nxt = task + warps;
    if (nxt < ntask && lane < d.k) {
      const int tok = nxt / nblk;
      src_n = __ldg(a.p.a[PA_SCALE_SRC] + (size_t)tok * d.k + lane);
      w_n = __ldg(a.w + (size_t)tok * d.k + lane);
    }
    const int tok = task / nblk;
    scale_round<SG, CPL, false>(a, d, tok / d.T, tok % d.T, src_l, w_l, lane,
                                (task % nblk) * 32 * CPL);
  }
  if (a.p.span != nullptr) {  // the same for the whole grid
    __syncthreads();
    if (threadIdx.x == 0) span_end(a.p.span, kSpanScaleEnd);
  }
}

// The scale overlapped with the combine (TileMoE notes section 2.2 step 5; the
// Perseus summary, section 4.1, Algorithm 1: the receiver acts on the one signal of
// each (sender, destination) group). Launched right behind the producer (or the
// consumer) on its stream as a programmatic dependent launch, so its CTAs are placed
// only once every CTA of that kernel is resident, and run beside it. Two gates, each
// watched by one thread with 1 us sleeps between reads: first every (sender,
// destination) group that sends rows has signalled, which makes every receive row
// final; then every output tile of the producer has been counted, which makes every
// local row final. Past the first gate, one warp per CTA sums the tokens whose slots
// are all remote while the producer still works through the local tiles it schedules
// last: one warp, so that this traffic beside the producer stays small. Past the
// second gate every warp takes what is left of those tokens, then the rest. Warps
// claim scale_kernel's tasks eight at a time from two counters of the plan (zeroed by
// the combine), and sum them with the same rounds: the same bits.
constexpr int kScaleClaim = 8;
constexpr int kGatePollNs = 1000;  // sleep between two reads of a gate
constexpr int kScaleThreads = 256;

template <int SG, int CPL>
__global__ void __launch_bounds__(kScaleThreads) scale_gated_kernel(const __grid_constant__ ScaleArgs a) {
  const Dims d = a.p.d;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n16 = d.D / 8;
  const int nblk = (n16 + 32 * CPL - 1) / (32 * CPL);
  const int ntask = d.W * d.T * nblk;
  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  const uint32_t* gsig = reinterpret_cast<const uint32_t*>(a.p.a[PA_GROUP_SIG]);
  uint32_t* queue = reinterpret_cast<uint32_t*>(a.p.a[PA_QUEUE]);
  uint32_t* claim = queue + 1;  // [1], [2]: the token counters of the two passes
  const uint32_t* tiles_done = queue + 3;  // output tiles (tile, N-tile) the producer finished
  __shared__ int s_ok;
  if (threadIdx.x == 0) span_begin(a.p.span, kSpanScaleStart);

  // Bounded wait of one thread for a gate (0: group signals, 1: finished tiles); false
  // when the status word is set or the wait ran out (then the status says so).
  auto wait_gate = [&](int gate) -> bool {
    const unsigned long long t0 = globaltimer();
    const uint32_t need = (uint32_t)a.p.a[PA_TOTALS][0] * (uint32_t)d.nt2;
    int g = 0;
    while (true) {
      bool open;
      if (gate == 0) {
        while (g < d.W * d.W &&
               (__ldg(a.p.a[PA_GROUP_NCHUNK] + g) == 0 || ld_relaxed_u32(gsig + g) != 0u))
          ++g;
        open = g == d.W * d.W;
      } else {
        open = ld_relaxed_u32(tiles_done) >= need;
      }
      if (open) break;
      if (ld_relaxed_u32(status) != 0u) return false;
      if ((long long)(globaltimer() - t0) > a.p.timeout_ns) {
        report_error(status, MOE_DEV_TIMEOUT, 0x70000000u | (uint32_t)gate);
        return false;
      }
      __nanosleep(kGatePollNs);
    }
    fence_acq_rel_gpu();  // the reads that opened the gate become acquires
    return true;
  };
  // One warp takes tasks of a pass (one round of one token each, as in scale_kernel),
  // kScaleClaim at a time, skipping tasks whose token belongs to the other pass; the
  // next task's sources and weights are fetched while the current one is summed.
  auto run_pass = [&](int pass) {
    int task = 0, end = 0;
    int src_n = INT_MIN;
    float w_n = 0.f;
    auto fetch = [&](int tk) {
      if (lane < d.k) {
        const int tok = tk / nblk;
        src_n = __ldg(a.p.a[PA_SCALE_SRC] + (size_t)tok * d.k + lane);
        w_n = __ldg(a.w + (size_t)tok * d.k + lane);
      }
    };
    while (true) {
      if (task == end) {
        int base = 0;
        if (lane == 0) base = (int)atomicAdd(claim + pass, (uint32_t)kScaleClaim);
        base = __shfl_sync(0xffffffffu, base, 0);
        if (base >= ntask) break;
        task = base;
        end = min(base + kScaleClaim, ntask);
        fetch(task);
      }
      const int src = src_n;
      const float wt = w_n;
      const int tok = task / nblk, c0 = (task % nblk) * 32 * CPL;
      if (++task < end) fetch(task);
      const bool local = src < 0 && src != INT_MIN;
      if (__any_sync(0xffffffffu, local) != (pass == 1)) continue;
      scale_round<SG, CPL, true>(a, d, tok / d.T, tok % d.T, src, wt, lane, c0);
    }
  };

  bool ok;
  if (warp == 0) {
    // The early warp: both gates itself, the all-remote tokens in between.
    ok = __shfl_sync(0xffffffffu, lane == 0 ? (wait_gate(0) ? 1 : 0) : 0, 0) != 0;
    fence_acq_rel_gpu();
    if (ok) run_pass(0);
    if (ok) ok = __shfl_sync(0xffffffffu, lane == 0 ? (wait_gate(1) ? 1 : 0) : 0, 0) != 0;
    fence_acq_rel_gpu();
  } else {
    // The other warps: one thread waits for both gates, then a barrier of these warps.
    if (threadIdx.x == 32) s_ok = wait_gate(0) && wait_gate(1) ? 1 : 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kScaleThreads - 32) : "memory");
    ok = s_ok != 0;
    fence_acq_rel_gpu();
  }
  if (ok) {
    run_pass(0);  // what the early warps left of the all-remote tokens
    run_pass(1);
  }
  __syncthreads();
  if (threadIdx.x == 0) span_end(a.p.span, kSpanScaleEnd);
}

}  // namespace

namespace {
// Resident blocks per SM of each scale kernel variant (k >= 4, k < 4), set at preload.
int g_scale_blocks_per_sm[2] = {0, 0};

int scale_variant(int k) { return k >= 4 ? 0 : 1; }

template <int SG, int CPL>
cudaError_t preload_scale_variant(int v) {
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, scale_kernel<SG, CPL>)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, scale_gated_kernel<SG, CPL>)) != cudaSuccess) return e;
  int n = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scale_kernel<SG, CPL>, 256, 0)) !=
      cudaSuccess)
    return e;
  g_scale_blocks_per_sm[v] = n;
  return cudaSuccess;
}

// Blocks of a scale launch over `units` warp tasks: as many as fit on the GPU at once
// (every warp then walks several tasks), fewer when there is less work.
int scale_blocks(int v, long long units, int num_sms) {
  const int per_sm = g_scale_blocks_per_sm[v] > 0 ? g_scale_blocks_per_sm[v] : 2;
  return (int)std::max(1LL, std::min((units + 7) / 8, (long long)num_sms * per_sm));
}

template <int SG, int CPL>
cudaError_t launch_scale_variant(const ScaleArgs& a, int num_sms, cudaStream_t s) {
  const int n16 = a.p.d.D / 8;
  const long long tasks = (long long)a.p.d.W * a.p.d.T * ((n16 + 32 * CPL - 1) / (32 * CPL));
  scale_kernel<SG, CPL><<<scale_blocks(scale_variant(a.p.d.k), tasks, num_sms), 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <int SG, int CPL>
cudaError_t launch_scale_gated_variant(const ScaleArgs& a, int num_sms, cudaStream_t s) {
  // As many CTAs as the plain scale; those that do not fit beside the running kernel
  // start as its CTAs leave. Programmatic stream serialization: the launch may begin
  // once every CTA of the previous kernel on the stream has allowed it.
  cudaLaunchConfig_t cfg = {};
  const int n16 = a.p.d.D / 8;
  const long long tasks = (long long)a.p.d.W * a.p.d.T * ((n16 + 32 * CPL - 1) / (32 * CPL));
  cfg.gridDim = dim3((unsigned)scale_blocks(scale_variant(a.p.d.k), tasks, num_sms));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, scale_gated_kernel<SG, CPL>, a);
}
}  // namespace

template <int PER>
cudaError_t launch_route_per(const DevPlan& p, const float* logits, const int32_t* forced,
                             int32_t* ids, float* w, cudaStream_t s) {
  const int ntok = p.d.W * p.d.T;
  route_kernel<PER><<<(ntok * 32 + 255) / 256, 256, 0, s>>>(p, logits, forced, ids, w);
  return cudaGetLastError();
}

cudaError_t preload_route_scale() {
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, route_kernel<1>)) != cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, route_kernel<2>)) != cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, route_kernel<4>)) != cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, route_kernel<8>)) != cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, route_kernel<16>)) != cudaSuccess ||
      (e = cudaFuncGetAttributes(&fa, route_kernel<32>)) != cudaSuccess)
    return e;
  if ((e = preload_scale_variant<4, 2>(0)) != cudaSuccess) return e;
  if ((e = preload_scale_variant<2, 4>(1)) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_route(const DevPlan& p, const float* logits, const int32_t* forced,
                         int32_t* ids, float* w, cudaStream_t s) {
  const int E = p.d.E;  // at most 1024 (checked when the plan is created)
  if (E <= 32) return launch_route_per<1>(p, logits, forced, ids, w, s);
  if (E <= 64) return launch_route_per<2>(p, logits, forced, ids, w, s);
  if (E <= 128) return launch_route_per<4>(p, logits, forced, ids, w, s);
  if (E <= 256) return launch_route_per<8>(p, logits, forced, ids, w, s);
  if (E <= 512) return launch_route_per<16>(p, logits, forced, ids, w, s);
  return launch_route_per<32>(p, logits, forced, ids, w, s);
}

cudaError_t launch_scale(const ScaleArgs& a, int num_sms, cudaStream_t s) {
  switch (scale_variant(a.p.d.k)) {
    case 0: return launch_scale_variant<4, 2>(a, num_sms, s);
    default: return launch_scale_variant<2, 4>(a, num_sms, s);
  }
}

cudaError_t launch_scale_gated(const ScaleArgs& a, int num_sms, cudaStream_t s) {
  switch (scale_variant(a.p.d.k)) {
    case 0: return launch_scale_gated_variant<4, 2>(a, num_sms, s);
    default: return launch_scale_gated_variant<2, 4>(a, num_sms, s);
  }
}

}  // namespace moe

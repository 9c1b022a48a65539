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

// One warp per token (s, t): out_s[t] = sum_j w_j * row_j, fp32 in slot order.
// Lane j < k holds slot j's source (scale map) and weight; the next token's are
// fetched while the current token is summed. Each lane covers two 16-byte chunks
// of the row per pass and gathers up to four slots' chunks into registers before
// accumulating, so a lane keeps up to eight independent 16-byte loads in flight.
// Slot order of the fp32 sum is kept (j ascending).
constexpr int kScaleGroup = 4;

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    acc[2 * q] = fmaf(w, f.x, acc[2 * q]);
    acc[2 * q + 1] = fmaf(w, f.y, acc[2 * q + 1]);
  }
}

__global__ void __launch_bounds__(256) scale_kernel(const __grid_constant__ ScaleArgs a) {
  const Dims d = a.p.d;
  const int lane = threadIdx.x & 31;
  const int n16 = d.D / 8;
  const int ntok = d.W * d.T;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int src_n = INT_MIN;
  float w_n = 0.f;
  if (tok < ntok && lane < d.k) {
    src_n = __ldg(a.p.a[PA_SCALE_SRC] + (size_t)tok * d.k + lane);
    w_n = __ldg(a.w + (size_t)tok * d.k + lane);
  }
  for (; tok < ntok; tok += warps) {
    const int src_l = src_n;
    const float w_l = w_n;
    const int nxt = tok + warps;
    if (nxt < ntok && lane < d.k) {
      src_n = __ldg(a.p.a[PA_SCALE_SRC] + (size_t)nxt * d.k + lane);
      w_n = __ldg(a.w + (size_t)nxt * d.k + lane);
    }
    const int s = tok / d.T, t = tok % d.T;
    uint4* out = reinterpret_cast<uint4*>(a.out[s] + (size_t)t * d.D);
    for (int c0 = 0; c0 < n16; c0 += 64) {
      const int ca = c0 + lane, cb = c0 + 32 + lane;
      float acc0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float acc1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j0 = 0; j0 < d.k; j0 += kScaleGroup) {
        uint4 va[kScaleGroup], vb[kScaleGroup];
        float wj[kScaleGroup];
#pragma unroll
        for (int q = 0; q < kScaleGroup; ++q) {
          const int j = j0 + q;
          const int sj = __shfl_sync(0xffffffffu, src_l, j & 31);
          wj[q] = __shfl_sync(0xffffffffu, w_l, j & 31);
          // Slots past k, and invalid routing slots (reported by the plan), add nothing.
          const bool live = j < d.k && sj != INT_MIN;
          if (!live) wj[q] = 0.f;
          const uint4* row = reinterpret_cast<const uint4*>(
              sj >= 0 ? a.recv[s] + (size_t)sj * d.D : a.y[s] + (size_t)(-sj - 1) * d.D);
          va[q] = live && ca < n16 ? __ldg(row + ca) : make_uint4(0, 0, 0, 0);
          vb[q] = live && cb < n16 ? __ldg(row + cb) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < kScaleGroup; ++q) {
          fma_bf16x8(acc0, wj[q], va[q]);
          fma_bf16x8(acc1, wj[q], vb[q]);
        }
      }
      if (ca < n16)
        out[ca] = make_uint4(pack_bf16x2(acc0[0], acc0[1]), pack_bf16x2(acc0[2], acc0[3]),
                             pack_bf16x2(acc0[4], acc0[5]), pack_bf16x2(acc0[6], acc0[7]));
      if (cb < n16)
        out[cb] = make_uint4(pack_bf16x2(acc1[0], acc1[1]), pack_bf16x2(acc1[2], acc1[3]),
                             pack_bf16x2(acc1[4], acc1[5]), pack_bf16x2(acc1[6], acc1[7]));
    }
  }
}

// scale_kernel's sum of one token (s, t), for rows that a kernel still running
// beside this one has written: the same operations in the same order (so the same
// bits), but the rows are read from L2 (__ldcg), since the read-only and L1 paths
// are not kept coherent with such writes. Lane j < k holds slot j's source and
// weight.
__device__ __forceinline__ void scale_token_l2(const ScaleArgs& a, int s, int t, int src_l,
                                               float w_l, int lane) {
  const Dims d = a.p.d;
  const int n16 = d.D / 8;
  uint4* out = reinterpret_cast<uint4*>(a.out[s] + (size_t)t * d.D);
  for (int c0 = 0; c0 < n16; c0 += 64) {
    const int ca = c0 + lane, cb = c0 + 32 + lane;
    float acc0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float acc1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < d.k; j0 += kScaleGroup) {
      uint4 va[kScaleGroup], vb[kScaleGroup];
      float wj[kScaleGroup];
#pragma unroll
      for (int q = 0; q < kScaleGroup; ++q) {
        const int j = j0 + q;
        const int sj = __shfl_sync(0xffffffffu, src_l, j & 31);
        wj[q] = __shfl_sync(0xffffffffu, w_l, j & 31);
        // Slots past k, and invalid routing slots (reported by the plan), add nothing.
        const bool live = j < d.k && sj != INT_MIN;
        if (!live) wj[q] = 0.f;
        const uint4* row = reinterpret_cast<const uint4*>(
            sj >= 0 ? a.recv[s] + (size_t)sj * d.D : a.y[s] + (size_t)(-sj - 1) * d.D);
        va[q] = live && ca < n16 ? __ldcg(row + ca) : make_uint4(0, 0, 0, 0);
        vb[q] = live && cb < n16 ? __ldcg(row + cb) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kScaleGroup; ++q) {
        fma_bf16x8(acc0, wj[q], va[q]);
        fma_bf16x8(acc1, wj[q], vb[q]);
      }
    }
    if (ca < n16)
      out[ca] = make_uint4(pack_bf16x2(acc0[0], acc0[1]), pack_bf16x2(acc0[2], acc0[3]),
                           pack_bf16x2(acc0[4], acc0[5]), pack_bf16x2(acc0[6], acc0[7]));
    if (cb < n16)
      out[cb] = make_uint4(pack_bf16x2(acc1[0], acc1[1]), pack_bf16x2(acc1[2], acc1[3]),
                           pack_bf16x2(acc1[4], acc1[5]), pack_bf16x2(acc1[6], acc1[7]));
  }
}

// The scale overlapped with the combine (TileMoE notes section 2.2 step 5; the
// Perseus summary, section 4.1, Algorithm 1: the receiver acts on the one signal of
// each (sender, destination) group). Launched right behind the producer (or the
// consumer) on its stream as a programmatic dependent launch, so its CTAs are placed
// only once every CTA of that kernel is resident, and run beside it. A token's sum
// starts once its rows are final: for each remote slot the signal of its (sender,
// destination) group, for each local slot the ready flags of the owner's band that
// holds the row. Warps claim tokens 32 at a time from two counters of the plan
// (zeroed by the combine): first the tokens whose slots are all remote (their groups
// signal as the remote tiles finish, while the producer works through the local
// ones), then the rest. The arithmetic is scale_kernel's: the same bits.
constexpr int kScaleClaim = 32;

__global__ void __launch_bounds__(256, 4) scale_gated_kernel(const __grid_constant__ ScaleArgs a) {
  const Dims d = a.p.d;
  const int lane = threadIdx.x & 31;
  const int ntok = d.W * d.T;
  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  const uint32_t* flags = reinterpret_cast<const uint32_t*>(a.p.a[PA_FLAGS]);
  const uint32_t* gsig = reinterpret_cast<const uint32_t*>(a.p.a[PA_GROUP_SIG]);
  uint32_t* claim = reinterpret_cast<uint32_t*>(a.p.a[PA_QUEUE]) + 1;  // [1], [2]: the passes
  // First receive row of each sender at each destination: receive rows are ordered by
  // sender rank, and a sender's first expert starts its range.
  __shared__ int s_start[MOE_MAX_RANKS][MOE_MAX_RANKS];  // [destination][sender]
  for (int i = threadIdx.x; i < d.W * d.W; i += blockDim.x) {
    const int s = i / d.W, o = i % d.W;
    s_start[s][o] = o == s ? INT_MAX : __ldg(a.p.a[PA_RECV_OFF] + (size_t)o * d.L * d.W + s);
  }
  if (threadIdx.x == 0) span_begin(a.p.span, kSpanScaleStart);
  __syncthreads();

  unsigned long long seen = 0;  // groups (sender * W + destination) seen signalled, warp-uniform
  bool ok = true;
  for (int pass = 0; pass < 2 && ok; ++pass) {
    while (ok) {
      int base = 0;
      if (lane == 0) base = (int)atomicAdd(claim + pass, (uint32_t)kScaleClaim);
      base = __shfl_sync(0xffffffffu, base, 0);
      if (base >= ntok) break;
      for (int tok = base; tok < min(base + kScaleClaim, ntok) && ok; ++tok) {
        int src = INT_MIN;
        float wt = 0.f;
        if (lane < d.k) {
          src = __ldg(a.p.a[PA_SCALE_SRC] + (size_t)tok * d.k + lane);
          wt = __ldg(a.w + (size_t)tok * d.k + lane);
        }
        const bool local = src < 0 && src != INT_MIN;
        if (__any_sync(0xffffffffu, local) != (pass == 1)) continue;
        const int s = tok / d.T;
        int g = -1;
        if (src >= 0) {  // the sender: the last rank whose first receive row is <= src
          int o = 0;
          for (int q = 0; q < d.W; ++q)
            if (s_start[s][q] <= src) o = q;
          g = o * d.W + s;
        }
        const uint32_t* f = local ? flags + ((size_t)s * d.NBM + (-src - 1) / d.tb) * d.nt2 : nullptr;
        // Bounded wait until every slot's rows are final (relaxed reads, then one
        // acquire fence per lane before the row loads).
        const unsigned long long t0 = globaltimer();
        while (true) {
          bool ready = true;
          if (g >= 0 && !((seen >> g) & 1ull)) ready = ld_relaxed_u32(gsig + g) != 0u;
          if (f != nullptr)
            for (int i = 0; i < d.nt2; ++i) ready &= ld_relaxed_u32(f + i) >= (uint32_t)d.parts;
          if (__all_sync(0xffffffffu, ready)) break;
          bool stop = false;
          if (lane == 0)
            stop = ld_relaxed_u32(status) != 0u ||
                   ((long long)(globaltimer() - t0) > a.p.timeout_ns &&
                    (report_error(status, MOE_DEV_TIMEOUT, 0x70000000u | (uint32_t)tok), true));
          if (__shfl_sync(0xffffffffu, stop ? 1 : 0, 0)) {
            ok = false;
            break;
          }
          __nanosleep(256);
        }
        if (!ok) break;
        fence_acq_rel_gpu();
        __syncwarp();
        const unsigned long long mine = g >= 0 ? 1ull << g : 0ull;
        seen |= (unsigned long long)__reduce_or_sync(0xffffffffu, (uint32_t)mine) |
                ((unsigned long long)__reduce_or_sync(0xffffffffu, (uint32_t)(mine >> 32)) << 32);
        scale_token_l2(a, s, tok % d.T, src, wt, lane);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) span_end(a.p.span, kSpanScaleEnd);
}

}  // namespace

namespace {
int g_scale_blocks_per_sm = 0;  // resident scale blocks per SM (set at preload)
}

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
  if ((e = cudaFuncGetAttributes(&fa, scale_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, scale_gated_kernel)) != cudaSuccess) return e;
  int n = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, scale_kernel, 256, 0)) != cudaSuccess)
    return e;
  g_scale_blocks_per_sm = n;
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
  // Eight warps per block, one token per warp at a time; as many blocks as fit on
  // the GPU at once, so every warp walks several tokens (and prefetches the next).
  const int tokens = a.p.d.W * a.p.d.T;
  const int per_sm = g_scale_blocks_per_sm > 0 ? g_scale_blocks_per_sm : 4;
  const int blocks = std::min((tokens + 7) / 8, num_sms * per_sm);
  scale_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_scale_gated(const ScaleArgs& a, int num_sms, cudaStream_t s) {
  // As many CTAs as the plain scale; those that do not fit beside the running kernel
  // start as its CTAs leave. Programmatic stream serialization: the launch may begin
  // once every CTA of the previous kernel on the stream has allowed it.
  const int tokens = a.p.d.W * a.p.d.T;
  const int per_sm = g_scale_blocks_per_sm > 0 ? g_scale_blocks_per_sm : 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(1, std::min((tokens + 7) / 8, num_sms * per_sm)));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, scale_gated_kernel, a);
}

}  // namespace moe

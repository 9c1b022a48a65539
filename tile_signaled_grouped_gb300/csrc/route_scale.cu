// Gate routing and the gated weighted sum (scale).
//
// TileMoE notes (zhongzhuzhou.org), section 2.1 and 2.2 steps 1 and 5: the
// router forms a probability distribution over the E experts per token and
// keeps the top k; the owner rank combines the k expert outputs of a token
// with the gate weights.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kMaxPerLane = 32;  // E <= 1024

// One warp per token: softmax over E logits (fp32), then k rounds of a warp
// argmax on (logit descending, expert id ascending). Comparing logits decides
// the same order as comparing probabilities, without rounding ties.
__global__ void route_kernel(DevPlan p, const float* __restrict__ logits,
                             const int32_t* __restrict__ forced, int32_t* __restrict__ ids,
                             float* __restrict__ w) {
  const Dims d = p.d;
  const int lane = threadIdx.x & 31;
  const int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tok >= d.W * d.T) return;
  const float* lg = logits + (size_t)tok * d.E;
  float v[kMaxPerLane];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < d.E ? lg[e] : -INFINITY;
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i)
    if (lane + 32 * i < d.E) sum += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.0f / sum;

  if (forced != nullptr) {
    for (int j = lane; j < d.k; j += 32) {
      const int e = forced[(size_t)tok * d.k + j];
      ids[(size_t)tok * d.k + j] = e;
      w[(size_t)tok * d.k + j] = (e >= 0 && e < d.E) ? expf(lg[e] - mx) * inv : 0.f;
    }
    return;
  }
  uint32_t taken = 0;  // bit i: this lane's candidate i already chosen
  for (int j = 0; j < d.k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX, bi = -1;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < d.E && !(taken >> i & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (bi >= 0 && lane + 32 * bi == be) taken |= 1u << bi;
    if (lane == 0) {
      ids[(size_t)tok * d.k + j] = be;
      w[(size_t)tok * d.k + j] = expf(bv - mx) * inv;
    }
  }
}

// One thread per 16-byte chunk (8 columns) of the outputs of kScaleTok tokens
// that are total/kScaleTok apart: out_s[t][c] = sum_j w_j * row_j[c], fp32 in slot
// order. Each token's row addresses depend on its scale-map entry, so a thread
// keeps the chains of its tokens independent and all their loads in flight.
constexpr int kScaleTok = 2;

__global__ void scale_kernel(const __grid_constant__ ScaleArgs a) {
  const Dims d = a.p.d;
  const int n16 = d.D / 8;
  const int total = d.W * d.T * n16;  // < 2^31 (checked when the plan is created)
  const int span = (total + kScaleTok - 1) / kScaleTok;
  const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
  if (i0 >= span) return;
  float acc[kScaleTok][8];
  int tok[kScaleTok], c[kScaleTok];
  bool live[kScaleTok];
#pragma unroll
  for (int u = 0; u < kScaleTok; ++u) {
    const int i = i0 + u * span;
    live[u] = i < total;
    tok[u] = live[u] ? i / n16 : 0;
    c[u] = live[u] ? i - tok[u] * n16 : 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
  }
  for (int j = 0; j < d.k; ++j) {
    int sj[kScaleTok];
    float wj[kScaleTok];
#pragma unroll
    for (int u = 0; u < kScaleTok; ++u) {
      sj[u] = live[u] ? a.p.a[PA_SCALE_SRC][(size_t)tok[u] * d.k + j] : INT_MIN;
      wj[u] = live[u] ? a.w[(size_t)tok[u] * d.k + j] : 0.f;
    }
    uint4 v[kScaleTok];
#pragma unroll
    for (int u = 0; u < kScaleTok; ++u) {
      v[u] = make_uint4(0, 0, 0, 0);
      if (sj[u] == INT_MIN) continue;  // invalid routing slot (reported by the plan)
      const int s = tok[u] / d.T;
      const __nv_bfloat16* row = sj[u] >= 0 ? a.recv[s] + (size_t)sj[u] * d.D
                                            : a.y[s] + (size_t)(-sj[u] - 1) * d.D;
      v[u] = __ldg(reinterpret_cast<const uint4*>(row) + c[u]);
    }
#pragma unroll
    for (int u = 0; u < kScaleTok; ++u) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        acc[u][2 * q] = fmaf(wj[u], f.x, acc[u][2 * q]);
        acc[u][2 * q + 1] = fmaf(wj[u], f.y, acc[u][2 * q + 1]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kScaleTok; ++u) {
    if (!live[u]) continue;
    const int s = tok[u] / d.T, t = tok[u] % d.T;
    reinterpret_cast<uint4*>(a.out[s] + (size_t)t * d.D)[c[u]] =
        make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                   pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7]));
  }
}

}  // namespace

cudaError_t preload_route_scale() {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, route_kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncGetAttributes(&fa, scale_kernel);
}

cudaError_t launch_route(const DevPlan& p, const float* logits, const int32_t* forced,
                         int32_t* ids, float* w, cudaStream_t s) {
  const int ntok = p.d.W * p.d.T;
  route_kernel<<<(ntok * 32 + 255) / 256, 256, 0, s>>>(p, logits, forced, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_scale(const ScaleArgs& a, int num_sms, cudaStream_t s) {
  (void)num_sms;
  const long long total = (long long)a.p.d.W * a.p.d.T * (a.p.d.D / 8);
  const long long span = (total + kScaleTok - 1) / kScaleTok;
  scale_kernel<<<(unsigned)((span + 255) / 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

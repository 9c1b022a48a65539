// Gate for few experts (E <= 16): the token rows streamed from HBM straight into
// registers, the router contraction on mma.sync, the softmax and the top k in the
// same launch.
//
// TileMoE notes (zhongzhuzhou.org), section 2.1 (a small gating network scores every
// token against the E experts) and 2.2 step 1 (every rank gates its own tokens): the
// router is one bias-free linear layer, logits = x W_r^T with W_r [E][D], then each
// token's softmax and top k exactly as the routing kernel takes them (route_topk.cuh).
//
// Why a second gate kernel. With E <= 16 the contraction is 8 or 16 columns wide: 2E
// FLOPs per 2 bytes of x, far below the ridge of any tensor path, so the launch is a
// one-shot read of x and its speed is how fast every SM gets its share of x in flight.
// The tcgen05 gate (gate.cu) stages x in shared memory through 2-D TMA boxes of
// 128-byte row pieces and waits a stage's refill round trip per 64 columns; plain
// 16-byte loads from every thread of a 1024-thread CTA ramp up faster and keep more
// bytes in flight, and they are the MMA's operands as loaded, with no staging.
//
// The contraction. A warp owns a group of 16 tokens of its CTA and a contiguous range
// of 64-column steps (the K slice). In step kb, lane (g = lane / 4, q = lane % 4)
// loads 32 bytes of each of tokens g and g + 8, columns [64 kb + 16 q, 64 kb + 16 q +
// 16): two 16-byte loads per row, the A operands of the step's four m16n8k16 MMAs.
// MMA m takes columns 16 q + 4 m + {0, 1} as its k = 2q, 2q + 1 and 16 q + 4 m +
// {2, 3} as its k = 2q + 8, 2q + 9; together the four MMAs cover each of the 64
// columns once. A sum over k does not depend on which k a column is given, so the
// router operand (B) takes the same assignment, and its fragment is the same 32
// bytes of router row 8 nt + g that lane loads: router rows are loaded like token
// rows, through L1 (the CTA's warps of one K slice share them), while x bypasses L1.
// Both are loaded one step ahead of the MMAs. E <= 8 is one n-tile of 8 experts
// (NT = 1), E <= 16 two; experts past E have zero operands and are never routed to.
//
// Sums. Each warp's accumulator is a 16 x 8NT fp32 partial of its K slice (the MMA's C
// fragment), written to shared memory; after the CTA barrier each token's scores are
// its group's partials added in slice order (a fixed order: the same bits on every
// call). An octet of lanes routes a token (route_lanes<8, NT>: butterflies instead of
// one thread's long dependent chain) and sets the plan's token bitmap bits from the ids it
// holds; prescribed ids go through a thread per token and the plan build's checks.
//
// Grid. CTA j of rank s takes tokens [j rows, (j + 1) rows) of that rank; a CTA has
// ceil(rows / 16) groups x kslices warps. gate_rows_shape picks small CTAs (32 tokens
// and 8 warps, or 16 and 4 with two n-tiles) that fit beside a producer CTA and, with
// enough tokens, fill an idle GPU as well; with few tokens, CTAs of up to 128 tokens
// and 32 warps (16 with two n-tiles) that spread them over one wave of SMs. The kernel
// has no wait but its two CTA barriers.
#include "moe_common.cuh"
#include "route_topk.cuh"

namespace moe {
namespace {

constexpr int kRowsMaxTokens = 128;
constexpr int kRowsSmemLimit = 48 * 1024;

__host__ __device__ constexpr int rows_nt(int E) { return E <= 8 ? 1 : 2; }
// Warps per CTA at most: 32 with one n-tile (64 registers a thread), 16 with two
// (their router operands double the registers the pipeline holds).
__host__ __device__ constexpr int rows_max_warps(int nt) { return nt == 1 ? 32 : 16; }
// Shared memory: one 16 x (8 NT + 4) fp32 partial block per warp (rows padded to 16
// bytes so that the routing threads' row loads do not collide in banks).
__host__ __device__ constexpr size_t rows_smem_bytes(int nt, int warps) {
  return (size_t)warps * 16 * (8 * nt + 4) * 4;
}
static_assert(rows_smem_bytes(1, rows_max_warps(1)) <= kRowsSmemLimit &&
                  rows_smem_bytes(2, rows_max_warps(2)) <= kRowsSmemLimit,
              "partials fit the default shared memory");

__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x is read once: no L1 allocation, so the router's lines stay in L1 for the warps of
// the SM that share them.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int NT>
__global__ void __launch_bounds__(rows_max_warps(NT) * 32, 1)
    gate_rows_kernel(const __grid_constant__ GateRowsArgs a) {
  extern __shared__ __align__(16) uint8_t rows_smem[];
  constexpr int EP = 8 * NT;
  constexpr int PS = EP + 4;  // floats per partial row
  const Dims d = a.p.d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int KS = a.kslices;
  const int cpr = (d.T + a.rows - 1) / a.rows;  // CTAs per rank
  const int s = (int)blockIdx.x / cpr;
  const int t0 = ((int)blockIdx.x % cpr) * a.rows;
  const int nrows = min(a.rows, d.T - t0);  // this CTA's tokens (>= 1)
  const int gi = warp / KS, ks = warp % KS;
  const int nk = d.D / 64;
  const int k0 = ks * nk / KS, k1 = (ks + 1) * nk / KS;
  float* part = reinterpret_cast<float*>(rows_smem);
  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  if (threadIdx.x == 0) span_begin(a.p.span, kSpanGateStart);

  // A operands: this thread's two token rows of the group (rows past the CTA's tokens
  // load zeros). B operands: router row 8 nt + g (zero past E), the same columns.
  const int ra = gi * 16 + g, rb = ra + 8;
  const bool va = ra < nrows, vb = rb < nrows;
  // Row g + 8 is D 16-byte words after row g (and is loaded only where row g is).
  const uint4* xa =
      reinterpret_cast<const uint4*>(a.x[s] + (size_t)(t0 + (va ? ra : 0)) * d.D) + 2 * q;
  bool vr[NT];
  const uint4* wr[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    vr[nt] = 8 * nt + g < d.E;
    wr[nt] = reinterpret_cast<const uint4*>(a.router + (size_t)(vr[nt] ? 8 * nt + g : 0) * d.D) +
             2 * q;
  }
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  // Step kb: columns [64 kb + 16 q, 64 kb + 16 q + 16) of both rows and of the router
  // rows, 16 bytes per load.
  auto load = [&](int kb, uint4(&v)[4], uint4(&b)[NT][2]) {
    v[0] = va ? ld_stream_v4(xa + kb * 8) : z;
    v[1] = va ? ld_stream_v4(xa + kb * 8 + 1) : z;
    v[2] = vb ? ld_stream_v4(xa + d.D + kb * 8) : z;
    v[3] = vb ? ld_stream_v4(xa + d.D + kb * 8 + 1) : z;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      b[nt][0] = vr[nt] ? __ldg(wr[nt] + kb * 8) : z;
      b[nt][1] = vr[nt] ? __ldg(wr[nt] + kb * 8 + 1) : z;
    }
  };

  float c[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 4; ++j) c[nt][j] = 0.f;
  uint4 cur[4], nxt[4], bc[NT][2], bn[NT][2];
  if (k0 < k1) load(k0, cur, bc);
  for (int kb = k0; kb < k1; ++kb) {
    if (kb + 1 < k1) load(kb + 1, nxt, bn);
#pragma unroll
    for (int m = 0; m < 4; ++m) {  // MMA m: 16-byte piece h = m / 2, words wi and wi + 1
      const int h = m >> 1, wi = 2 * (m & 1);
      const uint32_t a0 = word_of(cur[h], wi), a1 = word_of(cur[2 + h], wi);
      const uint32_t a2 = word_of(cur[h], wi + 1), a3 = word_of(cur[2 + h], wi + 1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_16816_bf16(c[nt], a0, a1, a2, a3, word_of(bc[nt][h], wi), word_of(bc[nt][h], wi + 1));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bc[nt][0] = bn[nt][0];
      bc[nt][1] = bn[nt][1];
    }
  }

  // This warp's partial: C fragment rows g and g + 8, columns 8 nt + 2q, 2q + 1.
  {
    float* pa = part + ((size_t)warp * 16 + g) * PS;
    float* pb = pa + 8 * PS;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      *reinterpret_cast<float2*>(pa + 8 * nt + 2 * q) = make_float2(c[nt][0], c[nt][1]);
      *reinterpret_cast<float2*>(pb + 8 * nt + 2 * q) = make_float2(c[nt][2], c[nt][3]);
    }
  }
  __syncthreads();

  // Each token's scores: its group's K-slice partials in slice order.
  auto score = [&](int r, int e) {
    const float* src = part + ((size_t)(r >> 4) * KS * 16 + (r & 15)) * PS + e;
    float v = 0.f;
    for (int k2 = 0; k2 < KS; ++k2) v += src[(size_t)k2 * 16 * PS];
    return v;
  };
  if (a.forced == nullptr) {
    // The gate's own top k: an octet of lanes per token (route_lanes), lane li holding
    // experts li and li + 8.
    constexpr int PER = NT;
    const int li = lane & 7;
    const int nwarps = (int)(blockDim.x >> 5);
    for (int r0 = warp * 4; r0 < nrows; r0 += nwarps * 4) {  // uniform across the warp
      const int r = r0 + (lane >> 3);
      const bool active = r < nrows;
      const int t = t0 + (active ? r : 0);
      const size_t tok = (size_t)s * d.T + t;
      float v[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = li + 8 * i;
        v[i] = active ? score(r, e) : 0.f;
        if (e < d.E) {
          if (active && a.logits != nullptr) a.logits[tok * d.E + e] = v[i];
        } else {
          v[i] = -INFINITY;
        }
      }
      const TokenMark mk{reinterpret_cast<uint32_t*>(a.p.a[PA_BITMAP]), (size_t)d.W * d.TW,
                         (size_t)s * d.TW + (t >> 5), 1u << (t & 31)};
      route_lanes<8, PER>(v, d.k, a.ids + tok * d.k, a.w + tok * d.k, li, active, &mk);
    }
  } else {
    // Prescribed ids: a thread per token, the ids checked and marked (mark_token).
    for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
      float v[EP];
#pragma unroll
      for (int e = 0; e < EP; ++e) v[e] = e < d.E ? score(r, e) : -INFINITY;
      const int t = t0 + r;
      const size_t tok = (size_t)s * d.T + t;
      if (a.logits != nullptr) {
#pragma unroll
        for (int e = 0; e < EP; ++e)
          if (e < d.E) a.logits[tok * d.E + e] = v[e];
      }
      route_group<1, EP>(v, d.E, d.k, a.forced + tok * d.k, a.ids + tok * d.k,
                         a.w + tok * d.k, 0);
      mark_token<1>(a.p, a.ids, a.forced, tok, s, t, 0, status);
    }
  }

  __syncthreads();
  if (threadIdx.x == 0) span_end(a.p.span, kSpanGateEnd);
}

template <int NT>
cudaError_t launch_rows_nt(const GateRowsArgs& a, cudaStream_t s) {
  const Dims& d = a.p.d;
  const int warps = (a.rows + 15) / 16 * a.kslices;
  if (warps > rows_max_warps(NT)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(d.W * ((d.T + a.rows - 1) / a.rows)), 1, 1);
  cfg.blockDim = dim3((unsigned)(warps * 32), 1, 1);
  cfg.dynamicSmemBytes = rows_smem_bytes(NT, warps);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, gate_rows_kernel<NT>, a);
}

}  // namespace

cudaError_t preload_gate_rows() { return cudaSuccess; }

bool gate_rows_fits(int E, int D) { return E >= 1 && E <= 16 && D % 64 == 0; }

void gate_rows_shape(int W, int T, int E, int D, int num_sms, bool beside, int* rows,
                     int* kslices) {
  // Small CTAs: a pair-producer CTA leaves about 25 K registers and 11 KB of shared
  // memory of its SM, room for 8 warps of 64 registers (one n-tile) or 4 of 104 (two)
  // with 6 KB of partials: two 16-token groups (one with two n-tiles) of up to 4 K
  // slices. On an idle GPU up to four of them share an SM, which keeps more loads in
  // flight than one wave-filling CTA and evens out the SMs' ends, so they are also the
  // automatic choice whenever there are enough of them to fill every SM once.
  const int small_ks = std::max(1, std::min(4, D / 64));
  const int small_groups = std::max(1, (rows_nt(E) == 1 ? 8 : 4) / small_ks);
  const int small_rows = std::min(T, 16 * small_groups);
  if (beside || (long long)W * ((T + small_rows - 1) / small_rows) >= num_sms) {
    *rows = small_rows;
    *kslices = small_ks;
    return;
  }
  // Otherwise as many tokens per CTA as make the W ranks' CTAs one wave (at most 128),
  // then as many K slices per 16-token group as the CTA's warps allow (at least one
  // step each).
  const int per_rank = std::max(1, num_sms / std::max(1, W));
  const int r = std::min(kRowsMaxTokens, std::max(1, (T + per_rank - 1) / per_rank));
  const int groups = (r + 15) / 16;
  *rows = r;
  *kslices = std::max(1, std::min(rows_max_warps(rows_nt(E)) / groups, D / 64));
}

cudaError_t launch_gate_rows(const GateRowsArgs& a, cudaStream_t s) {
  if (a.rows < 1 || a.rows > kRowsMaxTokens || a.kslices < 1 || !gate_rows_fits(a.p.d.E, a.p.d.D))
    return cudaErrorInvalidValue;
  return a.p.d.E <= 8 ? launch_rows_nt<1>(a, s) : launch_rows_nt<2>(a, s);
}

}  // namespace moe

// Combine consumer: polls the producer's per-tile ready flags and copies every
// finished segment's valid rows into its destination rank's receive buffer.
//
// TileMoE notes (zhongzhuzhou.org), section 5.2: the transfer unit is a row
// band (tb_M rows x the full output width: one owner, contiguous), merged into
// segments; section 5.3: a persistent consumer on its own SMs, coordinated with
// the producer only through device memory; section 4.5: destination, offset and
// valid-row count come from the precomputed combine plan (padding is never sent).
// Perseus summary (papercache.org), section 4.1, Algorithm 1: data moves without
// signals, then ONE fence per destination group precedes that group's signal.
//
// Here a group is (sender rank o, destination rank s). Its segments are split
// into `parts_per_group` parts (segment index modulo parts); a part is owned by
// one CTA, which copies the part's segments in the producer's tile order, then
// issues a single release (bar.sync + fence + atomic) for the whole part. The
// CTA that completes a group's last part stores the group signal. With one part
// per group this is exactly one fence per destination group.
#include "moe_common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(kConsumerThreads, 1)
    consumer_kernel(const __grid_constant__ ConsumerArgs a) {
  const Dims d = a.p.d;
  uint32_t* status = reinterpret_cast<uint32_t*>(a.p.a[PA_STATUS]);
  const uint32_t* flags = reinterpret_cast<const uint32_t*>(a.p.a[PA_FLAGS]);
  uint32_t* group_done = reinterpret_cast<uint32_t*>(a.p.a[PA_GROUP_DONE]);
  uint32_t* group_sig = reinterpret_cast<uint32_t*>(a.p.a[PA_GROUP_SIG]);
  const int32_t* order = a.p.a[PA_SEG_ORDER];
  const int R = a.parts_per_group;
  const int nseg = a.p.a[PA_TOTALS][1];
  const int tid = threadIdx.x, lane = tid & 31;
  __shared__ int s_go;

  for (int idx = 0; idx < nseg; ++idx) {
    const int code = order[idx];
    const int o = code / d.NBM, j = code % d.NBM;
    const size_t rb = (size_t)o * d.NBM;
    const int gidx = a.p.a[PA_SEG_GIDX][rb + j];
    const int first = a.p.a[PA_SEG_FIRST][rb + j];
    const int nbands = a.p.a[PA_SEG_NB][rb + j];
    const int b0 = a.p.a[PA_SCHED][rb + first];
    const int dst = a.p.a[PA_BAND_DST][rb + b0];
    const int g = o * d.W + dst;
    const int part = g * R + gidx % R;
    if (part % (int)gridDim.x != (int)blockIdx.x) continue;

    // Wait (bounded) until every tile of every band of the segment is flagged.
    if (tid < 32) {
      bool ok = true;
      const unsigned long long t0 = globaltimer();
      for (int b = b0; b < b0 + nbands && ok; ++b) {
        const uint32_t* f = flags + (rb + b) * d.nt2;
        for (int c = lane; c < d.nt2 && ok; c += 32) {
          while (ld_acquire_u32(f + c) < (uint32_t)d.parts) {
            if (ld_relaxed_u32(status) != 0) {
              ok = false;
              break;
            }
            if ((long long)(globaltimer() - t0) > a.p.timeout_ns) {
              report_error(status, MOE_DEV_TIMEOUT, 0x50000000u | (uint32_t)(rb + b));
              ok = false;
              break;
            }
            __nanosleep(32);
          }
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (lane == 0) s_go = ok;
    }
    __syncthreads();
    if (!s_go) return;  // an error is recorded; nothing waits on this CTA

    // Valid rows of the segment are contiguous: only a group's last band is partial.
    const int vrows = (nbands - 1) * d.tb + a.p.a[PA_BAND_VALID][rb + b0 + nbands - 1];
    const int drow = a.p.a[PA_BAND_DST_ROW][rb + b0];
    const uint4* src = reinterpret_cast<const uint4*>(a.y[o] + (size_t)b0 * d.tb * d.D);
    uint4* out = reinterpret_cast<uint4*>(a.recv[dst] + (size_t)drow * d.D);
    const long long n16 = (long long)vrows * d.D / 8;
    long long i = tid;
    for (; i + 3LL * kConsumerThreads < n16; i += 4LL * kConsumerThreads) {
      const uint4 v0 = __ldcg(src + i);
      const uint4 v1 = __ldcg(src + i + kConsumerThreads);
      const uint4 v2 = __ldcg(src + i + 2 * kConsumerThreads);
      const uint4 v3 = __ldcg(src + i + 3 * kConsumerThreads);
      __stcg(out + i, v0);
      __stcg(out + i + kConsumerThreads, v1);
      __stcg(out + i + 2 * kConsumerThreads, v2);
      __stcg(out + i + 3 * kConsumerThreads, v3);
    }
    for (; i < n16; i += kConsumerThreads) __stcg(out + i, __ldcg(src + i));

    // Last segment of this part: one release for the part, and the group signal
    // from whoever completes the group.
    const int gn = a.p.a[PA_GROUP_NSEG][o * d.W + dst];
    if (gidx + R >= gn) {
      __syncthreads();
      if (tid == 0) {
        fence_acq_rel_gpu();
        const uint32_t done = atomicAdd(group_done + g, 1u) + 1u;
        if (done == (uint32_t)min(R, gn)) {
          fence_acq_rel_gpu();
          st_release_u32(group_sig + g, 1u);
        }
      }
    }
    __syncthreads();  // s_go is rewritten by the next segment
  }
}

}  // namespace

cudaError_t launch_consumer(const ConsumerArgs& a, int grid, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(consumer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kConsumerSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // The dynamic shared memory is reserved, not used: it keeps a consumer CTA from
  // sharing an SM with a producer CTA, so the two kernels run on disjoint SMs.
  consumer_kernel<<<grid, kConsumerThreads, kConsumerSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

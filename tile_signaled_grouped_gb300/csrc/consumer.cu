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
// GB300 form (the body is combine_copy.cuh, shared with the copy warp of the fused
// pair producer): each segment is cut into chunks of rpc rows (up to 20 KB); the
// chunks of all segments, in the producer's tile order, are dealt round-robin to
// the consumer CTAs, so every CTA follows production and the last segment is
// copied by all of them. A CTA is one warp: in rounds of 32 of its chunks, each lane
// reads one chunk's segment record (through the plan's chunk-to-record map) and
// polls its flags, and lane 0 moves the chunks with TMA bulk copies through a
// six-slot shared-memory ring (global -> shared completes on an mbarrier,
// shared -> global as a bulk group). A group is (sender o, destination s). At
// each wait for the producer, and at its end, a CTA waits for its stores, issues
// one fence, and adds to each group's chunk count the chunks of it stored since
// the last release (one release increment per group, the groups spread over the
// lanes); the increment that completes a group stores the group signal.
#include "combine_copy.cuh"

namespace moe {
namespace {

using ConsumerSmem = CopySmem<kChunkSlots>;
static_assert(sizeof(ConsumerSmem) <= kConsumerSmemTail, "consumer shared memory layout");

__global__ void __launch_bounds__(kConsumerThreads, 1)
    consumer_kernel(const __grid_constant__ ConsumerArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  allow_dependent_launch();  // a scale launched behind this kernel may start beside it
  ConsumerSmem& sm =
      *reinterpret_cast<ConsumerSmem*>(smem_raw + (size_t)kChunkSlots * kChunkBytes);
  if (threadIdx.x == 0) span_begin(a.p.span, kSpanConsStart);
  combine_copy<kChunkSlots, kLoadsInFlight>(a.p, a.y, a.recv, smem_raw, sm, blockIdx.x,
                                            gridDim.x);
  __syncwarp();
  if (threadIdx.x == 0) span_end(a.p.span, kSpanConsEnd);
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
  // 132 KB of shared memory per CTA also keeps a consumer CTA from sharing an SM
  // with a producer CTA or another consumer CTA: the kernels run on disjoint SMs.
  consumer_kernel<<<grid, kConsumerThreads, kConsumerSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

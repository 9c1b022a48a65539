// Plan build for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc: a serving loop that reserved all of its
// device memory up front and forbids allocation afterwards, or a runtime whose
// allocator belongs to someone else (an inference server handing out fixed
// arenas). moe_plan_build needs a caller-provided workspace that holds both the
// plan and the plan kernels' internal scratch (token bitmaps, popcount prefixes,
// tile ordering, segment indices). This variant runs the same plan kernels, but
// keeps that internal scratch in a file-scope device array of fixed size; the
// caller passes only the routing ids (input) and a buffer for the plan arrays
// (output), and every array that moe_expert_combine and moe_scale read lands in
// that buffer.
#include <atomic>
#include <cstring>

#include "moe_common.cuh"

using namespace moe;

namespace {

// Scratch shared by every call on a device; held by each GPU that loads the
// library until the process exits. 1 MiB covers every workload shape of the
// tests (the largest, a 256-expert layer, needs about 200 KB).
constexpr size_t kScratchBytes = 1u << 20;
static __device__ __align__(256) uint8_t g_plan_scratch[kScratchBytes];

// Plan-workspace arrays that only the plan kernels themselves read. They live in
// the static scratch; every other array (among them everything the producer, the
// consumer and the scale read: tile list, scheduling units, CTA pairs, segment
// records, chunk counts per group, scale map) is written to the caller's output
// buffer at its moe_plan_build offset.
constexpr int kInternal[] = {PA_BITMAP,    PA_WPRE,     PA_NB,         PA_RANK_NB,
                             PA_BAND_TILE, PA_SEG_GIDX, PA_GROUP_NSEG, PA_RANK_TILES,
                             PA_UNIT_TMP};

constexpr int kMaxDevices = 64;
// Device address of g_plan_scratch per device ordinal, looked up by the first
// call made with that device current. In host code the array's name is only a
// host-side stand-in, so kernels must receive this address instead. Atomic, so
// host threads that make their first calls at the same time do not race on it
// (each stores the same address).
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

extern "C" int moe_plan_build_noalloc(const moe_cfg* cfg, const int32_t* topk_ids, void* plan_out,
                                      size_t plan_out_bytes, moe_stream_t stream) {
  Dims d;
  const int rc = dims_from_cfg(cfg, &d);
  if (rc != MOE_OK) return rc;
  if (topk_ids == nullptr || (reinterpret_cast<uintptr_t>(topk_ids) & 15) != 0 ||
      plan_out == nullptr || (reinterpret_cast<uintptr_t>(plan_out) & 255) != 0)
    return MOE_ERR_ARG;
  size_t off[PA_COUNT], cnt[PA_COUNT];
  if (plan_out_bytes < plan_layout(d, off, cnt)) return MOE_ERR_WORKSPACE;

  // Place the internal arrays in the static scratch; refuse shapes that exceed it.
  size_t pos = 0, soff[PA_COUNT] = {};
  for (int a : kInternal) {
    soff[a] = pos;
    pos += align256(cnt[a] * 4);
  }
  if (pos > kScratchBytes) return MOE_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* addr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr == nullptr) {
    if (cudaGetSymbolAddress(&addr, g_plan_scratch) != cudaSuccess || addr == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev].store(addr, std::memory_order_release);
  }
  uint8_t* scratch = static_cast<uint8_t*>(addr);
  uint8_t* out = static_cast<uint8_t*>(plan_out);

  DevPlan dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.d = d;
  for (int i = 0; i < PA_COUNT; ++i) dp.a[i] = reinterpret_cast<int32_t*>(out + off[i]);
  for (int a : kInternal) dp.a[a] = reinterpret_cast<int32_t*>(scratch + soff[a]);
  dp.timeout_ns = cfg->timeout_ns > 0 ? cfg->timeout_ns : 2000000000LL;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // A launch error is read back with cudaGetLastError after the launches; take any
  // error left pending by earlier, unrelated calls first, so it is not reported as
  // this call's.
  (void)cudaGetLastError();
  // The scratch keeps the previous call's contents: the token bitmaps must start at
  // zero (every other internal array is fully rewritten by the plan kernels).
  if (cudaMemsetAsync(dp.a[PA_BITMAP], 0, cnt[PA_BITMAP] * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_plan(dp, topk_ids, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

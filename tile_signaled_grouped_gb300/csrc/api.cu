// Host side of the C ABI: configuration checks, workspace carving, tensor maps
// and the stream choreography of the overlapped producer and consumer.
#include <cudaTypedefs.h>

#include <algorithm>
#include <vector>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <new>

#include "moe_common.cuh"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

enum TimingSlot { kTRoute = 0, kTPlan, kTProducer, kTConsumer, kTScale, kTGather, kTSlots };
constexpr int kTRing = 64;  // event pairs kept per timing slot

}  // namespace

struct moe_plan {
  moe_cfg cfg;
  Dims d;
  uint8_t* plan_ws;
  uint8_t* rank_ws[MOE_MAX_RANKS];
  size_t offsets[PA_COUNT];
  size_t counts[PA_COUNT];
  RankLayout rl;
  int num_sms;
  int pair_clusters;        // CTA pairs of the pair producer resident at once (0: unknown)
  int pair_clusters_fused;  // the same for its fused variant
  int gate_npad;            // gate MMA N (E rounded up to 32), 0 when E > kGateMaxE
  int gate_clusters[4];     // gate clusters resident at once for splits 1, 2, 4, 8
  PFN_cuTensorMapEncodeTiled_v12000 encode;
  cudaEvent_t ev_ready, ev_join;
  cudaEvent_t ev_t0[kTSlots][kTRing], ev_t1[kTSlots][kTRing];
  int nrec[kTSlots];  // measurements recorded since timing was enabled
  int nspan;          // combines whose device-clock records were kept since timing was enabled
  int last_span;      // ring record of the last combine (-1: none)
  bool xprev_ready;   // PA_XPREV holds the rows' contents (set by the first plan build)
  bool timing;        // CUDA events around each kernel
  bool spans;         // device-clock records (span ring, chunk landing stamps)
  bool gated_armed;   // a combine was enqueued since the last moe_scale_gated
  cudaStream_t combine_stream;  // the producer stream of the last combine
  bool gate_marked;   // the last routing call was moe_gate: its token bitmaps are in the plan
  const int32_t* gate_ids;  // the ids that moe_gate wrote
};

namespace moe {

int dims_from_cfg(const moe_cfg* c, Dims* d) {
  if (c == nullptr || d == nullptr) return MOE_ERR_ARG;
  if (c->W < 1 || c->W > MOE_MAX_RANKS || c->L < 1 || c->L > 256) return MOE_ERR_ARG;
  const long long E = (long long)c->W * c->L;
  if (E > 1024 || c->topk < 1 || c->topk > std::min<long long>(E, 32)) return MOE_ERR_ARG;
  if (c->T < 1 || c->T > (1 << 20)) return MOE_ERR_ARG;
  if (c->d_model < 128 || c->d_model % 128 || c->d_ff < 128 || c->d_ff % 128) return MOE_ERR_ARG;
  // A token row must fit one copy chunk (the combine copy moves whole rows through
  // kChunkBytes shared-memory slots): d_model <= 10240.
  if ((long long)c->d_model * 2 > kChunkBytes || c->d_ff > 65536) return MOE_ERR_UNSUPPORTED;
  if (c->tb_M != 64 && c->tb_M != 128 && c->tb_M != 256) return MOE_ERR_ARG;
  if (c->producer_pairs != 0 && c->producer_pairs != 1) return MOE_ERR_ARG;
  if (c->mgb < 1 || c->consumer_ctas < -1) return MOE_ERR_ARG;
  if (c->consumer_ctas == MOE_CONSUMER_FUSED && c->producer_pairs != 1) return MOE_ERR_ARG;
  Dims x{};
  x.W = c->W;
  x.L = c->L;
  x.E = (int)E;
  x.k = c->topk;
  x.T = c->T;
  x.D = c->d_model;
  x.F = c->d_ff;
  x.tb = c->tb_M;
  x.mgb = c->mgb;
  x.TW = (c->T + 31) / 32;
  // Worst case rows of one owner: every token reaching min(k, L) of its experts,
  // plus at most tb-1 zero rows per (expert, source rank) group.
  const long long rm = (long long)c->W * c->T * std::min(c->topk, c->L) +
                       (long long)c->L * c->W * (c->tb_M - 1);
  const long long RM = (rm + c->tb_M - 1) / c->tb_M * c->tb_M;
  if (RM >= (1LL << 24)) return MOE_ERR_UNSUPPORTED;
  if ((long long)c->W * c->T * (c->d_model / 8) >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  x.RM = (int)RM;
  x.NBM = x.RM / x.tb;
  x.parts = x.tb >= kTileM ? x.tb / kTileM : 1;
  x.NMM = x.NBM * x.parts;
  x.N2 = x.D % 256 == 0 ? 256 : 128;
  x.nt1 = x.F / kN1;
  x.nt2 = x.D / x.N2;
  x.rpc = std::max(1, kChunkBytes / (x.D * 2));
  // A segment spans at most mgb bands of tb rows; it must split into at most
  // kMaxSegChunks copy chunks.
  if (((long long)c->mgb * c->tb_M + x.rpc - 1) / x.rpc > kMaxSegChunks) return MOE_ERR_UNSUPPORTED;
  *d = x;
  return MOE_OK;
}

size_t plan_layout(const Dims& d, size_t* off, size_t* cnt) {
  size_t n[PA_COUNT] = {};
  const size_t W = d.W, E = d.E, NBM = d.NBM, NMM = d.NMM;
  n[PA_STATUS] = 4;
  n[PA_TOTALS] = 8;
  n[PA_QUEUE] = 4;
  n[PA_G1CNT] = W * NMM;
  n[PA_FLAGS] = W * NBM * d.nt2;
  n[PA_GROUP_DONE] = W * W;
  n[PA_GROUP_SIG] = W * W;
  n[PA_BITMAP] = E * W * d.TW;
  n[PA_WPRE] = E * W * d.TW;
  n[PA_CNT] = n[PA_GROUP_START] = n[PA_RECV_OFF] = E * W;
  n[PA_EXPERT_START] = n[PA_ROWS_ALLOC] = n[PA_NB] = n[PA_NRB] = E;
  n[PA_RANK_ROWS] = n[PA_RANK_NB] = n[PA_RANK_NREMOTE] = n[PA_RECV_ROWS] = n[PA_RANK_NSEG] = W;
  n[PA_BAND_EXPERT] = n[PA_BAND_DST] = n[PA_BAND_VALID] = n[PA_BAND_DST_ROW] = W * NBM;
  n[PA_BAND_TILE] = W * NBM;
  n[PA_SCHED] = n[PA_SEG_FIRST] = n[PA_SEG_NB] = n[PA_SEG_GIDX] = W * NBM;
  n[PA_GROUP_NSEG] = W * W;
  n[PA_RANK_TILES] = 2 * W * NMM;
  n[PA_TILE_ROW] = n[PA_TILE_EXPERT] = W * NMM;
  n[PA_UNIT_BEGIN] = 2 * W * (size_t)unit_cap(d) + 1;
  n[PA_SEG_ORDER] = W * NBM;
  n[PA_SEG_REC] = W * NBM * kSegRec;
  n[PA_GROUP_NCHUNK] = W * W;
  n[PA_XSRC] = W * (size_t)d.RM;
  n[PA_SCALE_SRC] = W * (size_t)d.T * d.k;
  n[PA_PAIR] = 4 * W * NMM;
  n[PA_PAIR_UNIT_BEGIN] = n[PA_UNIT_BEGIN];
  n[PA_SPANS] = 2 * kSpanWords * kSpanRing;
  n[PA_XPREV] = W * (size_t)d.RM;
  // Copy chunks of one combine: at most one partial chunk per segment beyond the
  // remote rows (at most W * T * topk) cut into chunks of rpc rows.
  n[PA_CHUNK_REC] = W * (size_t)d.T * d.k / d.rpc + W * NBM + 1;
  n[PA_CHUNK_T] = 2 * n[PA_CHUNK_REC];
  n[PA_UNIT_TMP] = 4 * W * (size_t)unit_cap(d);
  n[PA_PAIR_RUN] = W * NMM;
  size_t pos = 0;
  for (int i = 0; i < PA_COUNT; ++i) {
    if (off) off[i] = pos;
    if (cnt) cnt[i] = n[i];
    // The per-combine zeroed arrays are packed back to back (one memset); every
    // array after them starts on a kAlign boundary again.
    const bool packed = i >= PA_QUEUE && i < PA_GROUP_SIG;
    pos = packed ? pos + n[i] * 4 : align_up(pos + n[i] * 4, kAlign);
  }
  return align_up(pos, kAlign);
}

RankLayout rank_layout(const Dims& d) {
  RankLayout r{};
  const size_t xb = align_up((size_t)d.RM * d.D * 2, 1024);
  const size_t hb = align_up((size_t)d.RM * d.F * 2, 1024);
  r.x_off = 0;
  r.h_off = xb;
  r.y_off = xb + hb;
  r.bytes = xb + hb + xb;
  return r;
}

}  // namespace moe

namespace {

#define CUDA_TRY(x)                      \
  do {                                   \
    if ((x) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

DevPlan dev_plan(const moe_plan* p) {
  DevPlan dp{};
  dp.d = p->d;
  for (int i = 0; i < PA_COUNT; ++i)
    dp.a[i] = reinterpret_cast<int32_t*>(p->plan_ws + p->offsets[i]);
  dp.timeout_ns = p->cfg.timeout_ns > 0 ? p->cfg.timeout_ns : 2000000000LL;
  dp.span = nullptr;
  dp.chunk_t = nullptr;
  return dp;
}

unsigned long long* span_record(const moe_plan* p, int slot) {
  return reinterpret_cast<unsigned long long*>(p->plan_ws + p->offsets[PA_SPANS]) +
         (size_t)kSpanWords * (slot % kSpanRing);
}

// Host copy of the whole ring of device-clock records (kSpanRing x kSpanWords words).
cudaError_t copy_span_ring(const moe_plan* p, std::vector<unsigned long long>& ring) {
  try {
    ring.assign((size_t)kSpanWords * kSpanRing, 0ull);
  } catch (...) {  // no exception leaves the C ABI
    return cudaErrorMemoryAllocation;
  }
  return cudaMemcpy(ring.data(), p->plan_ws + p->offsets[PA_SPANS],
                    ring.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
}

struct LaunchShape {
  int producer, consumer;
};

// Grids of the producer and the consumer. Overlapped: the consumer's CTAs and the
// producer's share the SMs (one CTA of either per SM). The pair producer's grid
// also stops at the clusters that fit at once: the others would only start once
// the rest had finished.
LaunchShape launch_shape(const moe_plan* p, bool serial) {
  LaunchShape ls{};
  const bool fused = p->cfg.consumer_ctas == MOE_CONSUMER_FUSED;
  ls.consumer = serial ? p->num_sms : fused ? 0 : p->cfg.consumer_ctas;
  ls.producer = serial || fused ? p->num_sms : p->num_sms - p->cfg.consumer_ctas;
  if (p->cfg.producer_pairs) {
    const int clusters = fused ? p->pair_clusters_fused : p->pair_clusters;
    if (clusters > 0) ls.producer = std::min(ls.producer, 2 * clusters);
    ls.producer = std::max(2, ls.producer & ~1);
  }
  return ls;
}

bool aligned16(const void* ptr) { return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }
// An optional pointer: null, or 16-byte aligned.
bool null_or_aligned16(const void* ptr) { return ptr == nullptr || aligned16(ptr); }

void tstart(moe_plan* p, int slot, cudaStream_t s) {
  if (p->timing) cudaEventRecord(p->ev_t0[slot][p->nrec[slot] % kTRing], s);
}
void tstop(moe_plan* p, int slot, cudaStream_t s) {
  if (p->timing) {
    cudaEventRecord(p->ev_t1[slot][p->nrec[slot] % kTRing], s);
    p->nrec[slot]++;
  }
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix, box = box_rows x 64
// columns (128 B, the swizzle span), 128-byte swizzle, zero fill out of bounds.
bool make_map(const moe_plan* p, CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
              uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBlockK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = p->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int moe_workspace_size(const moe_cfg* cfg, size_t* plan_bytes, size_t* rank_bytes, int* recv_rows) {
  Dims d;
  const int rc = dims_from_cfg(cfg, &d);
  if (rc != MOE_OK) return rc;
  if (plan_bytes) *plan_bytes = plan_layout(d, nullptr, nullptr);
  if (rank_bytes) *rank_bytes = rank_layout(d).bytes;
  if (recv_rows) *recv_rows = d.T * d.k;
  return MOE_OK;
}

int moe_field(const moe_cfg* cfg, int field, size_t* byte_offset, size_t* count) {
  Dims d;
  const int rc = dims_from_cfg(cfg, &d);
  if (rc != MOE_OK) return rc;
  if (field >= MOE_RANK_X && field <= MOE_RANK_Y) {
    const RankLayout r = rank_layout(d);
    const size_t offs[3] = {r.x_off, r.h_off, r.y_off};
    const size_t cols[3] = {(size_t)d.D, (size_t)d.F, (size_t)d.D};
    if (byte_offset) *byte_offset = offs[field - MOE_RANK_X];
    if (count) *count = (size_t)d.RM * cols[field - MOE_RANK_X];
    return MOE_OK;
  }
  static const int map[MOE_PLAN_NFIELDS] = {
      PA_CNT,          PA_GROUP_START, PA_RECV_OFF,   PA_EXPERT_START, PA_ROWS_ALLOC,
      PA_NRB,          PA_RANK_ROWS,   PA_RANK_NREMOTE, PA_RECV_ROWS,  PA_RANK_NSEG,
      PA_BAND_EXPERT,  PA_BAND_DST,    PA_BAND_VALID, PA_BAND_DST_ROW, PA_SCHED,
      PA_SEG_FIRST,    PA_SEG_NB,      PA_XSRC,       PA_SCALE_SRC,    PA_TOTALS,
      PA_TILE_ROW,     PA_TILE_EXPERT, PA_SEG_ORDER,  PA_STATUS,       PA_FLAGS,
      PA_GROUP_SIG,    PA_PAIR};
  if (field < 0 || field >= MOE_PLAN_NFIELDS) return MOE_ERR_ARG;
  size_t off[PA_COUNT], cnt[PA_COUNT];
  plan_layout(d, off, cnt);
  if (byte_offset) *byte_offset = off[map[field]];
  if (count) *count = cnt[map[field]];
  return MOE_OK;
}

int moe_plan_create(const moe_cfg* cfg, void* plan_ws, size_t plan_ws_bytes, void* const* rank_ws,
                    size_t rank_ws_bytes, moe_plan** out) {
  if (out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  Dims d;
  int rc = dims_from_cfg(cfg, &d);
  if (rc != MOE_OK) return rc;
  if (!aligned16(plan_ws) || rank_ws == nullptr) return MOE_ERR_ARG;
  for (int r = 0; r < d.W; ++r)
    if (!aligned16(rank_ws[r]) || (reinterpret_cast<uintptr_t>(rank_ws[r]) & 1023)) return MOE_ERR_ARG;
  size_t off[PA_COUNT], cnt[PA_COUNT];
  const size_t need = plan_layout(d, off, cnt);
  const RankLayout rl = rank_layout(d);
  if (plan_ws_bytes < need || rank_ws_bytes < rl.bytes) return MOE_ERR_WORKSPACE;

  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;

  if (preload_producer() != cudaSuccess || preload_producer_pair() != cudaSuccess ||
      preload_consumer() != cudaSuccess ||
      preload_plan() != cudaSuccess || preload_route_scale() != cudaSuccess ||
      preload_gate() != cudaSuccess || preload_gate_rows() != cudaSuccess)
    return MOE_ERR_CUDA;

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      fn == nullptr || q != cudaDriverEntryPointSuccess)
    return MOE_ERR_CUDA;

  moe_plan* p = new (std::nothrow) moe_plan();
  if (p == nullptr) return MOE_ERR_ARG;
  p->cfg = *cfg;
  p->d = d;
  p->last_span = -1;
  p->plan_ws = static_cast<uint8_t*>(plan_ws);
  for (int r = 0; r < d.W; ++r) p->rank_ws[r] = static_cast<uint8_t*>(rank_ws[r]);
  std::memcpy(p->offsets, off, sizeof(off));
  std::memcpy(p->counts, cnt, sizeof(cnt));
  p->rl = rl;
  p->num_sms = prop.multiProcessorCount;
  p->pair_clusters = producer_pair_max_clusters(false);
  p->pair_clusters_fused = producer_pair_max_clusters(true);
  p->gate_npad = d.E <= kGateMaxE ? (d.E + 31) / 32 * 32 : 0;
  for (int i = 0; i < 4; ++i)
    p->gate_clusters[i] = p->gate_npad > 0 ? gate_clusters(d.E, 1 << i) : 0;
  p->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  bool ok = cudaEventCreateWithFlags(&p->ev_ready, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < kTSlots && ok; ++i)
    for (int j = 0; j < kTRing && ok; ++j)
      ok = cudaEventCreate(&p->ev_t0[i][j]) == cudaSuccess &&
           cudaEventCreate(&p->ev_t1[i][j]) == cudaSuccess;
  if (!ok) {
    moe_plan_destroy(p);
    return MOE_ERR_CUDA;
  }
  if (p->cfg.consumer_ctas >= p->num_sms) p->cfg.consumer_ctas = p->num_sms / 2;
  *out = p;
  return MOE_OK;
}

void moe_plan_destroy(moe_plan* p) {
  if (p == nullptr) return;
  if (p->ev_ready) cudaEventDestroy(p->ev_ready);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  for (int i = 0; i < kTSlots; ++i)
    for (int j = 0; j < kTRing; ++j) {
      if (p->ev_t0[i][j]) cudaEventDestroy(p->ev_t0[i][j]);
      if (p->ev_t1[i][j]) cudaEventDestroy(p->ev_t1[i][j]);
    }
  delete p;
}

int moe_route(moe_plan* p, const float* logits, const int32_t* forced, int32_t* ids, float* w,
              moe_stream_t stream) {
  if (p == nullptr || !aligned16(logits) || !null_or_aligned16(forced) || !aligned16(ids) ||
      !aligned16(w))
    return MOE_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const DevPlan dp = dev_plan(p);
  tstart(p, kTRoute, s);
  CUDA_TRY(launch_route(dp, logits, forced, ids, w, s));
  tstop(p, kTRoute, s);
  p->gate_marked = false;
  return MOE_OK;
}

int moe_gate(moe_plan* p, const void* const* x, const void* w_router, const int32_t* forced,
             int32_t* ids, float* w, float* logits, int splits, moe_stream_t stream) {
  if (p == nullptr || x == nullptr || !aligned16(w_router) || !null_or_aligned16(forced) ||
      !aligned16(ids) || !aligned16(w) || !null_or_aligned16(logits))
    return MOE_ERR_ARG;
  if (splits != MOE_GATE_BESIDE && splits != 0 && splits != 1 && splits != 2 && splits != 4 &&
      splits != 8)
    return MOE_ERR_ARG;
  const Dims& d = p->d;
  for (int r = 0; r < d.W; ++r)
    if (!aligned16(x[r])) return MOE_ERR_ARG;
  // MOE_GATE_BESIDE with E <= 16: the rows kernel in CTAs that fit beside a producer
  // CTA; with larger E the tcgen05 kernel as with splits == 0 (its CTAs cannot).
  const bool beside = splits == MOE_GATE_BESIDE;
  if (beside) splits = 0;
  const int lg = splits == 8 ? 3 : splits == 4 ? 2 : splits == 2 ? 1 : 0;
  if (p->gate_npad == 0 || (splits != 0 && p->gate_clusters[lg] == 0)) return MOE_ERR_UNSUPPORTED;
  // splits == 0 with E <= 16: the kernel that streams the token rows into registers;
  // otherwise the tcgen05 kernel.
  const bool rows_kernel = splits == 0 && gate_rows_fits(d.E, d.D);
  GateArgs ga{};
  GateRowsArgs ra{};
  if (rows_kernel) {
    for (int r = 0; r < d.W; ++r) ra.x[r] = static_cast<const __nv_bfloat16*>(x[r]);
    ra.router = static_cast<const __nv_bfloat16*>(w_router);
    ra.forced = forced;
    ra.ids = ids;
    ra.w = w;
    ra.logits = logits;
    ra.p = dev_plan(p);
    gate_rows_shape(d.W, d.T, d.E, d.D, p->num_sms, beside, &ra.rows, &ra.kslices);
  } else {
    ga.npad = p->gate_npad;
    ga.forced = forced;
    ga.ids = ids;
    ga.w = w;
    ga.logits = logits;
    ga.p = dev_plan(p);
    if (splits == 0) {
      // The largest split whose clusters all run at once (one wave: a second wave
      // costs a whole tile's time) and that leaves every CTA at least four K blocks.
      const int tiles = d.W * ((d.T + kTileM - 1) / kTileM);
      const int nk = d.D / kBlockK;
      splits = 1;
      for (int i = 1; i < 4; ++i)
        if (tiles <= p->gate_clusters[i] && nk >= (4 << i)) splits = 1 << i;
    }
    ga.splits = splits;
    // Tokens per tile: as few (a multiple of 8, at most 128) as fill one wave of
    // clusters, so that every SM streams its share of the token rows.
    {
      const int lgs = splits == 8 ? 3 : splits == 4 ? 2 : splits == 2 ? 1 : 0;
      const int per_rank = std::max(1, p->gate_clusters[lgs] / d.W);
      const int want = (d.T + per_rank - 1) / per_rank;
      ga.rows = std::min(kTileM, std::max(8, (want + 7) / 8 * 8));
    }
    for (int r = 0; r < d.W; ++r)
      if (!make_map(p, &ga.tm_x[r], x[r], d.T, d.D, (uint32_t)ga.rows)) return MOE_ERR_ARG;
    if (!make_map(p, &ga.tm_r, w_router, d.E, d.D, (uint32_t)ga.npad)) return MOE_ERR_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The routing tail sets the plan's token bitmaps: they start at zero.
  CUDA_TRY(cudaMemsetAsync(p->plan_ws + p->offsets[PA_BITMAP], 0, p->counts[PA_BITMAP] * 4, s));
  if (p->spans) {
    unsigned long long* span = span_record(p, p->nspan);
    ga.p.span = span;
    ra.p.span = span;
    CUDA_TRY(cudaMemsetAsync(span + kSpanGateStart, 0, 2 * sizeof(unsigned long long), s));
  }
  tstart(p, kTRoute, s);
  CUDA_TRY(rows_kernel ? launch_gate_rows(ra, s) : launch_gate(ga, s));
  tstop(p, kTRoute, s);
  p->gate_marked = true;
  p->gate_ids = ids;
  return MOE_OK;
}

int moe_plan_build(moe_plan* p, const int32_t* ids, const void* const* x, moe_stream_t stream) {
  if (p == nullptr || x == nullptr) return MOE_ERR_ARG;
  // ids == NULL: the routing of the last moe_gate, whose token bitmaps are already
  // in the plan.
  const bool marked = ids == nullptr;
  if (marked) {
    if (!p->gate_marked) return MOE_ERR_ARG;
    ids = p->gate_ids;
  }
  if (!aligned16(ids)) return MOE_ERR_ARG;
  for (int r = 0; r < p->d.W; ++r)
    if (!aligned16(x[r])) return MOE_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const DevPlan dp = dev_plan(p);
  tstart(p, kTPlan, s);
  if (!marked)
    CUDA_TRY(cudaMemsetAsync(p->plan_ws + p->offsets[PA_BITMAP], 0, p->counts[PA_BITMAP] * 4, s));
  CUDA_TRY(launch_plan(dp, ids, s, marked));
  p->gate_marked = false;
  const __nv_bfloat16* xs[MOE_MAX_RANKS] = {};
  __nv_bfloat16* xb[MOE_MAX_RANKS] = {};
  for (int r = 0; r < p->d.W; ++r) {
    xs[r] = static_cast<const __nv_bfloat16*>(x[r]);
    xb[r] = reinterpret_cast<__nv_bfloat16*>(p->rank_ws[r] + p->rl.x_off);
  }
  if (!p->xprev_ready) {  // first build: every X row's content is unknown (0xFEFEFEFE)
    CUDA_TRY(cudaMemsetAsync(p->plan_ws + p->offsets[PA_XPREV], 0xFE, p->counts[PA_XPREV] * 4, s));
    p->xprev_ready = true;
  }
  DevPlan gp = dp;
  if (p->spans) {  // the gather's span goes to the record of the combine that follows
    gp.span = span_record(p, p->nspan);
    CUDA_TRY(cudaMemsetAsync(gp.span + kSpanGatherStart, 0, 2 * sizeof(unsigned long long), s));
  }
  tstart(p, kTGather, s);
  CUDA_TRY(launch_gather(gp, xs, xb, p->num_sms, s));
  tstop(p, kTGather, s);
  tstop(p, kTPlan, s);
  return MOE_OK;
}

int moe_expert_combine(moe_plan* p, const void* const* w_gate, const void* const* w_up,
                       const void* const* w_down, void* const* recv, moe_stream_t producer,
                       moe_stream_t consumer) {
  if (p == nullptr || w_gate == nullptr || w_up == nullptr || w_down == nullptr || recv == nullptr)
    return MOE_ERR_ARG;
  const Dims& d = p->d;
  for (int r = 0; r < d.W; ++r)
    if (!aligned16(w_gate[r]) || !aligned16(w_up[r]) || !aligned16(w_down[r]) || !aligned16(recv[r]))
      return MOE_ERR_ARG;
  cudaStream_t sp = reinterpret_cast<cudaStream_t>(producer);
  cudaStream_t sc = reinterpret_cast<cudaStream_t>(consumer);
  const bool fused = p->cfg.consumer_ctas == MOE_CONSUMER_FUSED;
  const bool serial = !fused && (p->cfg.consumer_ctas == 0 || sp == sc);
  const bool pairs = p->cfg.producer_pairs != 0;
  const LaunchShape ls = launch_shape(p, serial);
  const int cgrid = ls.consumer, pgrid = ls.producer;

  ProducerArgs pa;
  std::memset(&pa, 0, sizeof(pa));
  pa.p = dev_plan(p);
  if (p->spans) {  // the kernels fold their device-clock stamps into a zeroed ring record
    pa.p.span = span_record(p, p->nspan);
    pa.p.chunk_t = reinterpret_cast<unsigned long long*>(p->plan_ws + p->offsets[PA_CHUNK_T]);
    CUDA_TRY(cudaMemsetAsync(pa.p.span, 0, kSpanCombineWords * sizeof(unsigned long long), sp));
    p->last_span = p->nspan % kSpanRing;
    p->nspan++;
  }
  for (int r = 0; r < d.W; ++r) {
    uint8_t* ws = p->rank_ws[r];
    const void* X = ws + p->rl.x_off;
    __nv_bfloat16* H = reinterpret_cast<__nv_bfloat16*>(ws + p->rl.h_off);
    __nv_bfloat16* Y = reinterpret_cast<__nv_bfloat16*>(ws + p->rl.y_off);
    if (!make_map(p, &pa.tm_x[r], X, d.RM, d.D, kTileM) ||
        !make_map(p, &pa.tm_h[r], H, d.RM, d.F, kTileM) ||
        !make_map(p, &pa.tm_wg[r], w_gate[r], (uint64_t)d.L * d.F, d.D, kN1) ||
        !make_map(p, &pa.tm_wu[r], w_up[r], (uint64_t)d.L * d.F, d.D, kN1) ||
        !make_map(p, &pa.tm_wd[r], w_down[r], (uint64_t)d.L * d.D, d.F, pairs ? d.N2 / 2 : d.N2))
      return MOE_ERR_ARG;
    pa.h[r] = H;
    pa.y[r] = Y;
    pa.recv[r] = static_cast<__nv_bfloat16*>(recv[r]);
  }
  // GEMM2 tasks of a unit start `lag` units after its GEMM1 tasks: about two
  // tasks per CTA (or CTA pair) in flight separate them. A pair unit holds about
  // half as many tasks as a tile unit.
  const int workers = pairs ? pgrid / 2 : pgrid;
  const int per_unit = (pairs ? kTileGroup / 2 : kTileGroup) * (d.nt1 + d.nt2);
  pa.lag = (2 * workers + per_unit - 1) / per_unit + 1;

  ConsumerArgs ca;
  std::memset(&ca, 0, sizeof(ca));
  ca.p = pa.p;
  for (int r = 0; r < d.W; ++r) {
    ca.y[r] = pa.y[r];
    ca.recv[r] = static_cast<__nv_bfloat16*>(recv[r]);
  }

  // Ready flags, GEMM1 counters, the ticket counters (the producer's and the overlapped
  // scale's) and the group signals start at 0.
  const size_t z0 = p->offsets[PA_QUEUE];
  const size_t z1 = p->offsets[PA_GROUP_SIG] + p->counts[PA_GROUP_SIG] * 4;
  CUDA_TRY(cudaMemsetAsync(p->plan_ws + z0, 0, z1 - z0, sp));
  p->gated_armed = true;
  p->combine_stream = sp;
  if (fused) {
    tstart(p, kTProducer, sp);
    CUDA_TRY(launch_producer_pair(pa, pgrid, true, sp));
    tstop(p, kTProducer, sp);
  } else if (serial) {
    tstart(p, kTProducer, sp);
    CUDA_TRY(pairs ? launch_producer_pair(pa, pgrid, false, sp) : launch_producer(pa, pgrid, sp));
    tstop(p, kTProducer, sp);
    tstart(p, kTConsumer, sp);
    CUDA_TRY(launch_consumer(ca, cgrid, sp));
    tstop(p, kTConsumer, sp);
  } else {
    CUDA_TRY(cudaEventRecord(p->ev_ready, sp));
    CUDA_TRY(cudaStreamWaitEvent(sc, p->ev_ready, 0));
    tstart(p, kTConsumer, sc);
    CUDA_TRY(launch_consumer(ca, cgrid, sc));
    tstop(p, kTConsumer, sc);
    CUDA_TRY(cudaEventRecord(p->ev_join, sc));
    tstart(p, kTProducer, sp);
    CUDA_TRY(pairs ? launch_producer_pair(pa, pgrid, false, sp) : launch_producer(pa, pgrid, sp));
    tstop(p, kTProducer, sp);
    CUDA_TRY(cudaStreamWaitEvent(sp, p->ev_join, 0));
  }
  return MOE_OK;
}

int moe_scale(moe_plan* p, const float* topk_w, const void* const* recv, void* const* out,
              moe_stream_t stream) {
  if (p == nullptr || !aligned16(topk_w) || recv == nullptr || out == nullptr) return MOE_ERR_ARG;
  const Dims& d = p->d;
  ScaleArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p = dev_plan(p);
  // Its span goes to the record of the last combine (whose words it zeroed).
  if (p->spans && p->last_span >= 0) a.p.span = span_record(p, p->last_span);
  a.w = topk_w;
  for (int r = 0; r < d.W; ++r) {
    if (!aligned16(recv[r]) || !aligned16(out[r])) return MOE_ERR_ARG;
    a.recv[r] = static_cast<const __nv_bfloat16*>(recv[r]);
    a.y[r] = reinterpret_cast<const __nv_bfloat16*>(p->rank_ws[r] + p->rl.y_off);
    a.out[r] = static_cast<__nv_bfloat16*>(out[r]);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  tstart(p, kTScale, s);
  CUDA_TRY(launch_scale(a, p->num_sms, s));
  tstop(p, kTScale, s);
  return MOE_OK;
}

int moe_scale_gated(moe_plan* p, const float* topk_w, const void* const* recv, void* const* out,
                    moe_stream_t stream) {
  // Only the combine's producer stream orders the kernel after the zeroing of the
  // flags, signals and counters it waits on.
  if (p == nullptr || !aligned16(topk_w) || recv == nullptr || out == nullptr || !p->gated_armed ||
      reinterpret_cast<cudaStream_t>(stream) != p->combine_stream)
    return MOE_ERR_ARG;
  const Dims& d = p->d;
  ScaleArgs a;
  std::memset(&a, 0, sizeof(a));
  a.p = dev_plan(p);
  a.w = topk_w;
  for (int r = 0; r < d.W; ++r) {
    if (!aligned16(recv[r]) || !aligned16(out[r])) return MOE_ERR_ARG;
    a.recv[r] = static_cast<const __nv_bfloat16*>(recv[r]);
    a.y[r] = reinterpret_cast<const __nv_bfloat16*>(p->rank_ws[r] + p->rl.y_off);
    a.out[r] = static_cast<__nv_bfloat16*>(out[r]);
  }
  if (p->spans && p->last_span >= 0) a.p.span = span_record(p, p->last_span);
  // No CUDA events around this launch: an event between the previous kernel and this
  // one would keep the launch from starting beside it.
  CUDA_TRY(launch_scale_gated(a, p->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  p->gated_armed = false;
  return MOE_OK;
}

int moe_producer_spans(moe_plan* p, unsigned long long* start_ns, unsigned long long* end_ns,
                       int max_records, int* count) {
  if (p == nullptr || start_ns == nullptr || end_ns == nullptr || count == nullptr ||
      max_records < 0 || !p->spans)
    return MOE_ERR_ARG;
  CUDA_TRY(cudaDeviceSynchronize());
  std::vector<unsigned long long> ring;
  CUDA_TRY(copy_span_ring(p, ring));
  const int m = std::min(std::min(p->nspan, kSpanRing), max_records);
  for (int i = 0; i < m; ++i) {  // oldest first
    const unsigned long long* r =
        ring.data() + (size_t)kSpanWords * ((p->nspan - m + i) % kSpanRing);
    start_ns[i] = ~r[kSpanProdStart];
    end_ns[i] = r[kSpanProdEnd];
  }
  *count = m;
  return MOE_OK;
}

int moe_combine_overlap(moe_plan* p, double* landed_frac, double* tail_us, double* copy_bytes) {
  if (p == nullptr || !p->spans || p->last_span < 0) return MOE_ERR_ARG;
  CUDA_TRY(cudaDeviceSynchronize());
  unsigned long long rec[kSpanWords];
  CUDA_TRY(cudaMemcpy(rec, span_record(p, p->last_span), sizeof(rec), cudaMemcpyDeviceToHost));
  int32_t tot[8];
  CUDA_TRY(cudaMemcpy(tot, p->plan_ws + p->offsets[PA_TOTALS], sizeof(tot), cudaMemcpyDeviceToHost));
  const int nseg = tot[1], nch = tot[4];
  double total = 0.0, before = 0.0;
  long long tail = LLONG_MIN;
  if (nseg > 0 && nch > 0) {
    int32_t* recs = new (std::nothrow) int32_t[(size_t)nseg * kSegRec];
    unsigned long long* st = new (std::nothrow) unsigned long long[nch];
    if (recs == nullptr || st == nullptr) {  // host memory for the copies of the records
      delete[] recs;
      delete[] st;
      return MOE_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaMemcpy(recs, p->plan_ws + p->offsets[PA_SEG_REC],
                               (size_t)nseg * kSegRec * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
      e = cudaMemcpy(st, p->plan_ws + p->offsets[PA_CHUNK_T], (size_t)nch * 8,
                     cudaMemcpyDeviceToHost);
    const unsigned long long last_tile = rec[kSpanLastTile];
    for (int i = 0; e == cudaSuccess && i < nseg; ++i) {
      const int32_t* r = recs + (size_t)i * kSegRec;
      for (int k = 0; k < r[7]; ++k) {
        const int rows = std::min(p->d.rpc, r[4] - k * p->d.rpc);
        const double bytes = (double)rows * p->d.D * 2.0;
        const unsigned long long t = st[r[6] + k];
        total += bytes;
        if (t <= last_tile) before += bytes;
        tail = std::max(tail, (long long)(t - last_tile));
      }
    }
    delete[] recs;
    delete[] st;
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (landed_frac) *landed_frac = total > 0.0 ? before / total : 1.0;
  if (tail_us) *tail_us = tail == LLONG_MIN ? 0.0 : (double)tail * 1e-3;
  if (copy_bytes) *copy_bytes = total;
  return MOE_OK;
}

int moe_set_schedule(moe_plan* p, int consumer_ctas, int mgb) {
  if (p == nullptr) return MOE_ERR_ARG;
  moe_cfg c = p->cfg;
  c.consumer_ctas = consumer_ctas;
  c.mgb = mgb;
  Dims d;
  const int rc = dims_from_cfg(&c, &d);
  if (rc != MOE_OK) return rc;
  if (c.consumer_ctas >= p->num_sms) c.consumer_ctas = p->num_sms / 2;
  p->cfg = c;
  p->d = d;
  return MOE_OK;
}

int moe_launch_info(moe_plan* p, int* producer_ctas, int* consumer_ctas, int* num_sms,
                    int* pair_clusters) {
  if (p == nullptr) return MOE_ERR_ARG;
  const LaunchShape ls = launch_shape(p, false);
  if (producer_ctas) *producer_ctas = ls.producer;
  if (consumer_ctas) *consumer_ctas = ls.consumer;
  if (num_sms) *num_sms = p->num_sms;
  if (pair_clusters) *pair_clusters = p->pair_clusters;
  return MOE_OK;
}

int moe_status(moe_plan* p, moe_stream_t stream, int* code, int* detail) {
  if (p == nullptr) return MOE_ERR_ARG;
  CUDA_TRY(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  uint32_t st[2] = {0, 0};
  CUDA_TRY(cudaMemcpy(st, p->plan_ws + p->offsets[PA_STATUS], sizeof(st), cudaMemcpyDeviceToHost));
  if (code) *code = (int)st[0];
  if (detail) *detail = (int)st[1];
  return MOE_OK;
}

int moe_status_clear(moe_plan* p, moe_stream_t stream) {
  if (p == nullptr) return MOE_ERR_ARG;
  CUDA_TRY(cudaMemsetAsync(p->plan_ws + p->offsets[PA_STATUS], 0, 16,
                           reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_set_timing(moe_plan* p, int enable) {
  if (p == nullptr || enable < 0 || enable > 2) return MOE_ERR_ARG;
  if (enable != 0) {  // start from a clean span ring (instrumentation: synchronises the device)
    CUDA_TRY(cudaDeviceSynchronize());
    CUDA_TRY(cudaMemset(p->plan_ws + p->offsets[PA_SPANS], 0, p->counts[PA_SPANS] * 4));
    CUDA_TRY(cudaDeviceSynchronize());
  }
  p->timing = enable == 1;
  p->spans = enable != 0;
  for (int i = 0; i < kTSlots; ++i) p->nrec[i] = 0;
  p->nspan = 0;
  p->last_span = -1;
  return MOE_OK;
}

int moe_timings(moe_plan* p, float* ms, int n) {
  if (p == nullptr || ms == nullptr) return MOE_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    ms[i] = -1.f;
    if (i >= kTSlots || p->nrec[i] == 0) continue;
    const int m = std::min(p->nrec[i], kTRing);
    double sum = 0.0;
    for (int j = 0; j < m; ++j) {
      const int q = (p->nrec[i] - 1 - j) % kTRing;
      CUDA_TRY(cudaEventSynchronize(p->ev_t1[i][q]));
      float v = 0.f;
      CUDA_TRY(cudaEventElapsedTime(&v, p->ev_t0[i][q], p->ev_t1[i][q]));
      sum += v;
    }
    ms[i] = (float)(sum / m);
  }
  // Device-clock records: [6] the producer's span, [7] the scale's span (moe_scale or
  // moe_scale_gated), [8] the part of that span before the producer's end (means over
  // the records).
  for (int i = kTSlots; i < n && i < kTSlots + 4; ++i) ms[i] = -1.f;
  const int m = std::min(p->nspan, kSpanRing);
  if (n > kTSlots && m > 0) {
    CUDA_TRY(cudaDeviceSynchronize());
    std::vector<unsigned long long> ring;
    CUDA_TRY(copy_span_ring(p, ring));
    double prod = 0.0, scale = 0.0, beside = 0.0;
    int nscale = 0;
    for (int j = 0; j < m; ++j) {
      const unsigned long long* r =
          ring.data() + (size_t)kSpanWords * ((p->nspan - 1 - j) % kSpanRing);
      const unsigned long long p0 = ~r[kSpanProdStart], p1 = r[kSpanProdEnd];
      prod += (double)(p1 - p0) * 1e-6;
      if (r[kSpanScaleStart] != 0) {
        const unsigned long long s0 = ~r[kSpanScaleStart], s1 = r[kSpanScaleEnd];
        scale += (double)(s1 - s0) * 1e-6;
        beside += s0 < p1 ? (double)(std::min(s1, p1) - s0) * 1e-6 : 0.0;
        ++nscale;
      }
    }
    ms[kTSlots] = (float)(prod / m);
    if (nscale > 0 && n > kTSlots + 1) ms[kTSlots + 1] = (float)(scale / nscale);
    if (nscale > 0 && n > kTSlots + 2) ms[kTSlots + 2] = (float)(beside / nscale);
  }
  // [9] the gate's span, [10] the consumer kernel's, [11] the layout gather's (first CTA
  // start to last CTA end), each over the records that hold one. The gate and the
  // gather write the record of the combine that follows them.
  for (int i = kTSlots + 3; i < n && i < kTSlots + 6; ++i) ms[i] = -1.f;
  if (n > kTSlots + 3 && p->spans) {
    const int mg = std::min(p->nspan + 1, kSpanRing);
    CUDA_TRY(cudaDeviceSynchronize());
    std::vector<unsigned long long> ring;
    CUDA_TRY(copy_span_ring(p, ring));
    const int w0[3] = {kSpanGateStart, kSpanConsStart, kSpanGatherStart};
    const int w1[3] = {kSpanGateEnd, kSpanConsEnd, kSpanGatherEnd};
    for (int k = 0; k < 3 && kTSlots + 3 + k < n; ++k) {
      double sum = 0.0;
      int cnt = 0;
      for (int j = 0; j < mg; ++j) {
        const unsigned long long* r =
            ring.data() + (size_t)kSpanWords * ((p->nspan - j) % kSpanRing);
        if (r[w1[k]] != 0 && r[w0[k]] != 0) {
          sum += (double)(r[w1[k]] - ~r[w0[k]]) * 1e-6;
          ++cnt;
        }
      }
      if (cnt > 0) ms[kTSlots + 3 + k] = (float)(sum / cnt);
    }
  }
  return MOE_OK;
}

}  // extern "C"

/*
 * moe_tsg.h - C ABI of the tile-signalled grouped MoE expert-combine path (sm_103a).
 *
 * The path follows the TileMoE notes (zhongzhuzhou.org, "Fine-grained
 * Computation-Communication Overlap via Tile-level Signaling and Scheduling
 * for Mixture-of-Experts"):
 *   routing (section 2.2 step 1) -> expert problem construction and combine
 *   plan (section 4.2 row layout, 4.4 remote-first schedule / Algorithm 1,
 *   4.5 combine plan) -> overlapped execution: a persistent grouped expert-FFN
 *   producer that sets one ready flag per finished output tile, and a consumer
 *   on a disjoint set of SMs that polls the flags and copies finished segments
 *   (section 5.1-5.3) -> gated weighted sum (scale, section 2.2 step 5).
 * The consumer signals each (sender, destination) group once, after one
 * fence, as in the decoupled signalling of the Perseus summary
 * (papercache.org, section 4.1, Algorithm 1).
 *
 * Everything runs on ONE GPU. The W expert-parallel ranks of the pages are
 * logical: each has its own device allocations (token input, weights,
 * rank workspace, receive buffer, output), and the combine all-to-all is a
 * device-memory copy between those allocations.
 *
 * Conventions
 *  - All pointers are device pointers unless stated. The caller owns all
 *    memory; the library never allocates device memory and owns no stream.
 *  - Tensors are dense, row-major, bf16 unless stated; every tensor's base
 *    pointer (bf16, int32 and fp32 alike) must be 16-byte aligned, or the call
 *    returns MOE_ERR_ARG. d_model and d_ff must be multiples of 128.
 *  - Return value 0 (MOE_OK) or a negative MOE_ERR_* for errors detected on
 *    the host before anything is enqueued. Errors detected on the device
 *    (bad routing ids, a device wait that ran out of time) are sticky in the
 *    plan workspace and are read with moe_status().
 *  - Every call is asynchronous on the given stream(s) except moe_status(),
 *    moe_timings() and the pure-host queries.
 */
#ifndef MOE_TSG_H
#define MOE_TSG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

/* Largest number of logical ranks one plan can hold. */
#define MOE_MAX_RANKS 8

/* moe_cfg.consumer_ctas value: the combine copy runs inside the pair producer. */
#define MOE_CONSUMER_FUSED (-1)

/* moe_gate splits value: for E <= 16, CTAs small enough to share an SM with a running
 * producer CTA (a gate that runs beside the previous batch's combine). */
#define MOE_GATE_BESIDE (-1)

enum moe_error {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,         /* invalid configuration or argument */
  MOE_ERR_WORKSPACE = -2,   /* a workspace is smaller than moe_workspace_size() */
  MOE_ERR_CUDA = -3,        /* a CUDA runtime call failed (no device, launch error) */
  MOE_ERR_UNSUPPORTED = -4, /* the device is not sm_103 / the shape is outside the kernels' limits */
  /* Device-side codes, reported through moe_status(). */
  MOE_DEV_ROUTING = 1,      /* an expert id is out of range or repeated within a token */
  MOE_DEV_TIMEOUT = 2       /* a device-side wait exceeded cfg.timeout_ns */
};

/* Configuration of one MoE layer split over W logical ranks.
 * Expert e is owned by rank e / L (local index e % L), the placement of
 * Figure 2b of the TileMoE notes. */
typedef struct moe_cfg {
  int W;             /* logical expert-parallel ranks, 1..MOE_MAX_RANKS */
  int L;             /* experts per rank (E = W*L, 1..1024) */
  int topk;          /* experts per token, 1..min(E, 32) */
  int T;             /* tokens per rank, >= 1 */
  int d_model;       /* D, multiple of 128, at most 10240 (a token row fits one 20 KB
                        copy chunk; larger gives MOE_ERR_UNSUPPORTED) */
  int d_ff;          /* F, expert hidden size, multiple of 128 */
  int tb_M;          /* row-band height of the layout: 64, 128 or 256 */
  int mgb;           /* row bands merged into one middle segment (section 5.2), >= 1 */
  int consumer_ctas; /* consumer CTAs running beside the producer (cCTA of section 5.3).
                        0 = serial: the producer uses every SM, then the consumer runs
                        on every SM after it, on the producer stream.
                        MOE_CONSUMER_FUSED (-1, with producer_pairs = 1): no consumer
                        kernel; one warp of every producer CTA polls the flags and
                        copies, on every SM. */
  long long timeout_ns; /* bound on every device-side wait; <= 0 selects 2 s */
  int producer_pairs; /* 0: one producer CTA per 128-row tile (tcgen05.mma, M = 128).
                         1: CTA pairs (clusters of two): each task covers two 128-row
                         tiles of one expert, rows estart + 256 i and estart + 256 i + 128
                         of its block, with one tcgen05.mma of M = 256 (cta_group::2);
                         each CTA loads its own rows and half of the weight rows. */
} moe_cfg;

/* Opaque host-side handle; holds the configuration, the carved workspace
 * pointers and a few CUDA events. Created by moe_plan_create(). */
typedef struct moe_plan moe_plan;

/* Sizes of the caller-provided memory for cfg (pure host arithmetic).
 *  plan_bytes:  one device allocation shared by all ranks (plan arrays, flags).
 *  rank_bytes:  one device allocation per rank (its expert input X, hidden
 *               activations and expert outputs Y, sized for the worst case).
 *  recv_rows:   rows of the receive buffer every rank needs ([recv_rows, D] bf16);
 *               the worst case T*topk.
 * Any output pointer may be NULL. */
int moe_workspace_size(const moe_cfg *cfg, size_t *plan_bytes, size_t *rank_bytes,
                       int *recv_rows);

/* Bind a configuration to its workspaces. plan_ws: plan_bytes; rank_ws: W pointers,
 * each rank_bytes. Queries the current device; fails with MOE_ERR_UNSUPPORTED
 * on anything other than compute capability 10.3. *out must be released with
 * moe_plan_destroy(). Host memory only; enqueues nothing. */
int moe_plan_create(const moe_cfg *cfg, void *plan_ws, size_t plan_ws_bytes,
                    void *const *rank_ws, size_t rank_ws_bytes, moe_plan **out);
void moe_plan_destroy(moe_plan *plan);

/* Routing (TileMoE notes section 2.1 and 2.2 step 1): for every token, softmax over
 * the E gate logits, then the topk experts with the largest logits in descending
 * order (equal logits: the lower expert id first). The weights are the softmax
 * probabilities at the chosen ids, not renormalised.
 *  logits:     [W][T][E] fp32.
 *  forced_ids: NULL, or [W][T][topk] int32 prescribed routing; then ids = forced_ids
 *              and the weights are the probabilities at those ids.
 *  topk_ids:   out [W][T][topk] int32.   topk_w: out [W][T][topk] fp32. */
int moe_route(moe_plan *plan, const float *logits, const int32_t *forced_ids,
              int32_t *topk_ids, float *topk_w, moe_stream_t stream);

/* Gate from the token rows (TileMoE notes section 2.1: a small gating network;
 * 2.2 step 1: every rank gates its own tokens), in one kernel: the router's
 * scores logits[s][t][e] = sum_c x_s[t][c] * w_router[e][c] (bf16 operands, fp32
 * sums on the tensor cores), then the routing of moe_route on those scores.
 *  x:          W pointers, rank s's tokens [T][D] bf16, 16-byte aligned.
 *  w_router:   [E][D] bf16 (nn.Linear layout), one copy shared by every rank,
 *              16-byte aligned.
 *  forced_ids, topk_ids, topk_w: as moe_route.
 *  logits:     NULL, or out [W][T][E] fp32: the scores the routing used.
 *  splits:     0 picks the kernel: for E <= 16 one that streams the token rows
 *              from HBM into registers and takes the scores with mma.sync (the
 *              contraction is 8 or 16 columns wide and the launch a one-shot read
 *              of x), in CTAs of 32 tokens and 8 warps (16 tokens and 4 warps with
 *              9-16 experts) when there are enough of them to fill every SM, else in
 *              larger CTAs that spread the tokens over one wave; above, the tcgen05
 *              kernel with the K split it picks. 1, 2, 4 or 8 force the tcgen05
 *              kernel with that split (that many CTAs of one cluster share a
 *              128-token tile, each summing a range of D).
 *              MOE_GATE_BESIDE: for E <= 16 always the small CTAs, which fit in what a
 *              pair-producer CTA leaves of its SM, so the gate of the next batch runs
 *              beside a running combine instead of waiting for its SMs; above, as 0.
 * Both kernels add each score's partial sums in a fixed order, so a given choice
 * gives the same bits on every call; the two kernels' scores differ by rounding
 * only. A tcgen05 tile holds as many tokens (a multiple of 8, at most 128) as fill
 * one wave of CTAs.
 * The routing tail also sets the plan's token bitmaps (prescribed ids out of range
 * or repeated set MOE_DEV_ROUTING), for a following moe_plan_build(plan, NULL, ...).
 * E <= 256; larger E, or a split the GPU cannot hold, gives MOE_ERR_UNSUPPORTED.
 * The caller owns every buffer. Timed in slot [0] of moe_timings, its device-clock
 * span in slot [9]. */
int moe_gate(moe_plan *plan, const void *const *x, const void *w_router,
             const int32_t *forced_ids, int32_t *topk_ids, float *topk_w, float *logits,
             int splits, moe_stream_t stream);

/* Expert problem construction and combine plan (TileMoE notes section 4.2, 4.4
 * Algorithm 1, 4.5, 5.2) for all ranks, then the layout gather that fills each
 * owner's expert input X with its tokens' rows (zero rows for padding).
 *  topk_ids: [W][T][topk] int32, ids distinct within a token; or NULL: the routing of
 *            the last moe_gate on this plan (no moe_route or moe_plan_build since),
 *            whose routing tail already set the plan's token bitmaps, so the bitmap
 *            kernel is skipped; MOE_ERR_ARG if there is none.
 *  x:        W pointers, rank s's tokens [T][D] bf16.
 * Ids out of range or repeated set MOE_DEV_ROUTING; the offending assignments are
 * skipped. No device-to-host transfer: every size is read on the device. */
int moe_plan_build(moe_plan *plan, const int32_t *topk_ids, const void *const *x,
                   moe_stream_t stream);

/* Overlapped expert FFN and combine (TileMoE notes section 5.1-5.3).
 * The producer walks the remote-first schedule: per 128-row tile of X,
 * h = SiLU(X Wg^T) * (X Wu^T) (bf16), then Y = h Wd^T (bf16), fp32 accumulation,
 * and after each finished Y tile it sets that tile's ready flag. The consumer
 * (consumer_ctas CTAs on a high-priority stream, or after the producer in serial
 * mode) polls the flags and copies each finished segment's valid rows into the
 * destination rank's receive buffer at the planned offset. Padding rows are never
 * copied. Local rows stay in the owner's Y.
 *  w_gate, w_up: W pointers, [L][F][D] bf16.  w_down: W pointers, [L][D][F] bf16.
 *  recv:         W pointers, [recv_rows][D] bf16 (moe_workspace_size).
 *  producer, consumer: streams; the consumer stream should have higher priority.
 *  When consumer_ctas == 0 or both streams are equal, the call runs serially on
 *  `producer`. On return, work enqueued later on `producer` is ordered after both
 *  kernels. */
int moe_expert_combine(moe_plan *plan, const void *const *w_gate, const void *const *w_up,
                       const void *const *w_down, void *const *recv,
                       moe_stream_t producer, moe_stream_t consumer);

/* Scale (TileMoE notes section 2.2 step 5): out_s[t] = sum_j w[s][t][j] * y_j, where
 * y_j is token (s,t)'s output of its j-th expert, read from rank s's receive buffer
 * (remote expert) or rank s's own Y (local expert). fp32 accumulation in slot order,
 * bf16 result.
 *  topk_w: [W][T][topk] fp32.  recv: W pointers as given to moe_expert_combine.
 *  out:    W pointers, [T][D] bf16. */
int moe_scale(moe_plan *plan, const float *topk_w, const void *const *recv, void *const *out,
              moe_stream_t stream);

/* Scale overlapped with the combine (TileMoE notes section 2.2 step 5; the Perseus
 * summary, section 4.1, Algorithm 1: the receiver acts on the one signal of each
 * (sender, destination) group). Same arguments and the same results, bit for bit,
 * as moe_scale, for the routing of the last moe_expert_combine. Enqueue it on that
 * call's producer stream right after it: the kernel is launched with programmatic
 * stream serialization, so it starts once every CTA of the kernel before it on the
 * stream (the producer; the consumer in the serial schedule) is running, and works
 * beside it. A token's sum waits on the device until its rows are final: the signal
 * of each remote slot's (sender, destination) group and the ready flags of each
 * local slot's row band; tokens whose slots are all remote go first. Any other work
 * between the combine and this call on the stream (an event, a wait) makes it start
 * after the combine instead, with the same results. Waits are bounded by timeout_ns
 * (MOE_DEV_TIMEOUT); a status already set makes the kernel return. One call per
 * moe_expert_combine, on its producer stream (MOE_ERR_ARG otherwise). No CUDA events are recorded around it
 * (they would keep it from overlapping); with moe_set_timing(plan, 2) the device clock
 * records its span (moe_timings slots 7 and 8). */
int moe_scale_gated(moe_plan *plan, const float *topk_w, const void *const *recv,
                    void *const *out, moe_stream_t stream);

/* Overlap of the combine copy with the expert FFN in the last moe_expert_combine made
 * while device-clock records were on (moe_set_timing 1 or 2), the quantity of the TileMoE
 * notes' section 7.3 (overlap ratio of the second all-to-all): *landed_frac is the share
 * of the combine's bytes whose copies had landed when the producer finished its last
 * output tile, *tail_us how long after that tile the last copy landed (negative if
 * before), *copy_bytes the bytes copied. Synchronises the device. MOE_ERR_ARG if no
 * such combine was recorded; MOE_ERR_UNSUPPORTED if host memory for copies of the
 * segment records and stamps cannot be had. Any output pointer may be NULL. */
int moe_combine_overlap(moe_plan *plan, double *landed_frac, double *tail_us,
                        double *copy_bytes);

/* The device-clock intervals of the producer launches recorded while device-clock
 * records were on (moe_set_timing 1 or 2), oldest first: start_ns[i], end_ns[i] are
 * the i-th launch's first CTA start and last CTA end on the GPU's global timer
 * (nanoseconds; comparable across the plans of one device, so a caller running
 * several plans in turn can take the union of their launches). At most max_records of
 * the last 1024 launches; *count receives how many were written. Synchronises the
 * device. MOE_ERR_ARG without records. */
int moe_producer_spans(moe_plan *plan, unsigned long long *start_ns, unsigned long long *end_ns,
                       int max_records, int *count);

/* Plan build that allocates nothing, for callers that cannot call cudaMalloc (for
 * example a serving loop that reserved all of its device memory up front, or a
 * runtime whose device memory comes from an allocator it does not own). The pages
 * have no counterpart. It runs moe_plan_build's plan kernels on the same routing
 * and writes the same plan, but not the layout gather (X is not filled).
 *  topk_ids: [W][T][topk] int32 (input).
 *  plan_out: caller buffer of at least the plan_bytes of moe_workspace_size(),
 *            256-byte aligned; the plan arrays are written where moe_plan_build
 *            writes them in a plan workspace (moe_field() reports the public ones).
 *            Bad routing ids set the MOE_PLAN_STATUS word inside plan_out, which
 *            this call never clears. A plan handle created on plan_out
 *            (moe_plan_create) can then run moe_expert_combine and moe_scale on it,
 *            given rank workspaces whose X a moe_plan_build of the same routing
 *            filled. The regions of the plan kernels' internal arrays (token
 *            bitmaps, word prefixes, per-band and per-tile orderings, segment
 *            indices) are left untouched in plan_out, as is the per-combine region.
 * Those internal arrays live in a fixed 1 MiB array inside the library, which every
 * GPU that loads the library holds until the process exits; shapes whose internal
 * arrays exceed it return MOE_ERR_UNSUPPORTED. No cudaMalloc, cudaFree or
 * allocating library call is made. The first call on each device looks up that
 * array's device address (cudaGetSymbolAddress, with the device current) and may
 * load the library's kernels: make it before any stream capture. Every call shares
 * the one array, so calls that overlap on the GPU (other streams, other threads)
 * race; serialise them. Host threads may make calls at the same time. */
int moe_plan_build_noalloc(const moe_cfg *cfg, const int32_t *topk_ids, void *plan_out,
                           size_t plan_out_bytes, moe_stream_t stream);

/* Changes the schedule of an existing plan: the consumer partition (consumer_ctas of
 * moe_cfg; 0 = serial) and the segment merge width (mgb of moe_cfg, section 5.2). Host
 * only; a new mgb takes effect at the next moe_plan_build, a new consumer_ctas at the
 * next moe_expert_combine. Same limits as in moe_cfg: MOE_ERR_ARG for values out of
 * range, MOE_ERR_UNSUPPORTED if a segment of mgb bands would exceed the copy-chunk limit.
 * The workspaces are unchanged (their sizes do not depend on either value). */
int moe_set_schedule(moe_plan *plan, int consumer_ctas, int mgb);

/* How moe_expert_combine splits the GPU for this plan (pure host query; the
 * occupancy is read once by moe_plan_create).
 *  producer_ctas:   CTAs of one producer launch in the overlapped schedule (even
 *                   with producer_pairs: clusters of two that fit on the GPU at once).
 *  consumer_ctas:   CTAs of one consumer launch in the overlapped schedule.
 *  num_sms:         SMs of the device.
 *  pair_clusters:   clusters of two CTAs of the pair producer that fit on an idle
 *                   GPU at once (0 if the runtime could not tell).
 * Any output pointer may be NULL. */
int moe_launch_info(moe_plan *plan, int *producer_ctas, int *consumer_ctas, int *num_sms,
                    int *pair_clusters);

/* Synchronises `stream` and reads the device status word: *code is 0 or a
 * MOE_DEV_* value, *detail the first failing item (token, band or tile index).
 * The status stays set until moe_status_clear(). */
int moe_status(moe_plan *plan, moe_stream_t stream, int *code, int *detail);
int moe_status_clear(moe_plan *plan, moe_stream_t stream);

/* Named arrays of the plan workspace and the rank workspaces, for inspection:
 * byte offset of the array inside its workspace and its element count. Elements
 * are int32 except MOE_RANK_X/H/Y (bf16). Pure host arithmetic. */
enum moe_field {
  MOE_PLAN_CNT = 0,          /* [E][W] rows of expert e from rank s */
  MOE_PLAN_GROUP_START,      /* [E][W] first row of group (e, s) in expert e's block */
  MOE_PLAN_RECV_OFF,         /* [E][W] first receive row of (e, s) at rank s, -1 if local */
  MOE_PLAN_EXPERT_START,     /* [E]    first row of expert e's block in its owner's X */
  MOE_PLAN_ROWS_ALLOC,       /* [E]    rows of expert e's block (multiple of tb_M) */
  MOE_PLAN_NRB,              /* [E]    remote row bands of expert e */
  MOE_PLAN_RANK_ROWS,        /* [W]    rows of each owner's X */
  MOE_PLAN_RANK_NREMOTE,     /* [W]    remote prefix length of each owner's schedule */
  MOE_PLAN_RECV_ROWS,        /* [W]    rows received by each rank */
  MOE_PLAN_RANK_NSEG,        /* [W]    segments of each owner */
  MOE_PLAN_BAND_EXPERT,      /* [W][NBmax] per rank-local band: expert */
  MOE_PLAN_BAND_DST,         /* [W][NBmax] destination rank */
  MOE_PLAN_BAND_VALID,       /* [W][NBmax] valid (non-padding) rows */
  MOE_PLAN_BAND_DST_ROW,     /* [W][NBmax] first receive row at the destination, -1 if local */
  MOE_PLAN_SCHEDULE,         /* [W][NBmax] S: rank-local band ids in schedule order */
  MOE_PLAN_SEG_FIRST,        /* [W][NBmax] first schedule index of each segment */
  MOE_PLAN_SEG_NBANDS,       /* [W][NBmax] bands of each segment */
  MOE_PLAN_XSRC,             /* [W][RowsMax] per X row: source token s*T+t, or -1 */
  MOE_PLAN_SCALE_SRC,        /* [W][T][topk] >= 0: receive row; < 0: row -v-1 of own Y */
  MOE_PLAN_TOTALS,           /* [8] 0: tiles, 1: segments, 2: tile units, 3: bands,
                                4: consumer copy chunks, 5: producer CTA pairs */
  MOE_PLAN_TILE_ROW,         /* [tiles] per 128-row producer tile: rank*2^24 + first X row */
  MOE_PLAN_TILE_EXPERT,      /* [tiles] expert of each producer tile */
  MOE_PLAN_SEG_ORDER,        /* [segments] consumer order: rank*NBmax + segment */
  MOE_PLAN_STATUS,           /* [4] device status word */
  MOE_PLAN_FLAGS,            /* [W][NBmax][D/tile_N] ready flags of the last combine */
  MOE_PLAN_GROUP_SIG,        /* [W][W] group signals (sender, destination) of the last combine */
  MOE_PLAN_PAIR,             /* [pairs][4] producer CTA pairs in pair order: the earlier tile of
                                the tile order, its partner or -1, the earlier tile's
                                rank*2^24 + first X row, and its local expert + 2^16 if the
                                partner's rows lie 128 above */
  MOE_PLAN_NFIELDS,
  MOE_RANK_X = 100,          /* [RowsMax][D] bf16 expert input */
  MOE_RANK_H,                /* [RowsMax][F] bf16 hidden activation */
  MOE_RANK_Y                 /* [RowsMax][D] bf16 expert output */
};
int moe_field(const moe_cfg *cfg, int field, size_t *byte_offset, size_t *count);

/* Device time in ms of the kernels the calls enqueue, measured with CUDA events
 * recorded on the stream each kernel ran on: the mean over the calls made since
 * timing was last enabled (the most recent 64 of them). Synchronises on those
 * events. Order: [0] route (moe_route or moe_gate), [1] plan (all plan kernels and the gather),
 * [2] producer, [3] consumer, [4] scale, [5] gather only. Then, from the device clock,
 * means over the last 1024 combines: [6] the producer's execution span (its first CTA's
 * start to its last CTA's end; unlike [2] it excludes time spent queued behind other
 * kernels, for example those of another batch in flight, and the launch latency CUDA
 * events include), [7] the span of the scale (moe_scale or moe_scale_gated) after the
 * combine, [8] the part of [7] before the producer's end, [9] the span of moe_gate,
 * [10] the span of the consumer kernel (not the fused copy warp), [11] the span of the
 * layout gather of moe_plan_build. A slot with no measurement is -1. Instrumentation only: moe_set_timing(plan, 1) records the events
 * and the device-clock records, 2 only the device-clock records (no CUDA event enters
 * the streams, so kernels keep overlapping as without timing), 0 nothing; enabling
 * resets the counts. */
int moe_set_timing(moe_plan *plan, int enable);
int moe_timings(moe_plan *plan, float *ms, int n);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TSG_H */

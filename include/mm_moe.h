/*
 * mm_moe.h — C ABI of the GB300 (sm_103a) MoE-layer forward.
 *
 * One call computes the forward of one MoE layer on one GPU, with every expert
 * local (the MegaMoE data path of llm-infra-atlas "07 · MegaMoE", §1–§9,
 * without its cross-GPU dispatch and scatter):
 *   a1 dispatch    routing histogram, per-expert segment offsets, and a slot
 *                  for every (token, k) pair, ascending token order inside an
 *                  expert ("07 · MegaMoE" §4 and §7; nxmr.cn walkthrough §二.2.4);
 *   a2 gather      activation rows and their scales copied into the pool;
 *   a3 L1 GEMM     gate|up = x_hat · W1_hat^T per expert, block-scaled;
 *   a4 L1 epilogue a = silu(gate) · up · topk_w, requantised to e4m3
 *                  ("07 · MegaMoE" §8; MEGAMOE_SM90_DESIGN.md §10.1);
 *   a5 L2 GEMM     y = a_hat · W2_hat^T per expert;
 *   a6 L2 epilogue y written as fp32 partials [K][T][H];
 *   a7 combine     out[t] = bf16(sum over k = 0..K-1 of the partials), fixed order
 *                  (MEGAMOE_SM90_DESIGN.md §11.2).
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers to row-major, contiguous memory,
 *     owned by the caller.  The library allocates no device memory and keeps no
 *     state beyond a per-device cache of properties and kernel attributes.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: a return of MM_MOE_OK means the work was
 *     enqueued.  Errors found on the device (wait timeouts, bad routing) are
 *     reported by mm_moe_sync_status().
 *   - Inputs are read-only.  `out` is fully overwritten.
 *
 * Numeric formats ("variant"):
 *   MM_MOE_VARIANT_MX  e4m3 activations x e2m1 weights, one UE8M0 scale byte
 *                      (value 2^(b-127)) per 32 contiguous elements along the
 *                      contraction dimension; tcgen05 kind::mxf8f6f4.
 *   MM_MOE_VARIANT_F8  e4m3 activations with one fp32 scale per 1x128, e4m3
 *                      weights with one fp32 scale per 128x128 block; the
 *                      intermediate is requantised per 128 (or per 64, see
 *                      f8_act_gran) with a raw fp32 scale amax/448 (DeepGEMM
 *                      PR #440, "Why the order and not the pool size");
 *                      tcgen05 kind::f8f6f4.
 *
 * Layouts (T tokens, H hidden, I intermediate, E experts, K top-k):
 *   x        u8  [T, H]          e4m3 codes
 *   x_sf     MX: u8 [T, H/32]    F8: f32 [T, H/128]
 *   topk_idx i32 [T, K]          expert of slot k; -1 masks the slot; values < -1
 *                                or >= E are treated as masked and flagged
 *                                (MM_MOE_ERR_BAD_ROUTING from mm_moe_sync_status)
 *   topk_w   f32 [T, K]          router weight of slot k
 *   w1       MX: u8 [E, 2I, H/2] (two e2m1 per byte, low nibble = even column)
 *            F8: u8 [E, 2I, H]; rows [0, I) are the gate projection, [I, 2I) up
 *   w2       MX: u8 [E, H, I/2]  F8: u8 [E, H, I]
 *   w1_sf/w2_sf (canonical, input of mm_moe_prepare_weights only)
 *            MX: u8 [E, 2I, H/32] and u8 [E, H, I/32]
 *            F8: f32 [E, 2I/128, H/128] and f32 [E, H/128, I/128]
 *   w1_sfp/w2_sfp  the scales in the layout the kernels read, written by
 *            mm_moe_prepare_weights (sizes from mm_moe_weight_sf_size)
 *   out      bf16 [T, H]
 * Shape limits: H % 128 == 0, I % 128 == 0, 1 <= K <= 16, K <= E <= 1024,
 * T >= 0 (T = 0 computes nothing and only clears the workspace's status word).  w1/w2 must be 32-byte aligned, x/workspace
 * 256-byte aligned.
 */
#ifndef MM_MOE_H_
#define MM_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MM_MOE_OK 0
#define MM_MOE_ERR_INVALID_ARG 1          /* null pointer, bad shape, misalignment */
#define MM_MOE_ERR_UNSUPPORTED 2          /* not an sm_103a/sm_100-family device, or option not built */
#define MM_MOE_ERR_CUDA 3                 /* a CUDA runtime/driver call failed */
#define MM_MOE_ERR_TIMEOUT 4              /* a device wait passed its deadline (sync_status only) */
#define MM_MOE_ERR_BAD_ROUTING 5          /* topk_idx held values >= E or < -1 (sync_status only) */
#define MM_MOE_ERR_WORKSPACE_TOO_SMALL 6

#define MM_MOE_VARIANT_MX 0
#define MM_MOE_VARIANT_F8 1

typedef struct mm_moe_options {
  int variant;                  /* MM_MOE_VARIANT_MX (default) or MM_MOE_VARIANT_F8 */
  int fused;                    /* 1 (default): one persistent kernel runs gather, L1 and L2 as one
                                   lag-ordered task stream (MX format; the F8 variant and the L1
                                   debug dump always use separate launches); 0: separate gather /
                                   L1 / L2 launches.  Both give bit-identical results. */
  int lag_units;                /* fused stream: how many experts the L2 tiles trail the L1 tiles
                                   (0..E, larger values act as E); -1 = auto (E: every L1 tile
                                   before any L2 tile, the fastest order measured on one GPU) */
  int retain_intermediate;      /* keep the whole requantised intermediate readable after the call
                                   (mm_moe_read_intermediate) */
  unsigned wait_timeout_ms;     /* deadline of every device-side wait; 0 = default (2000 ms) */
  int num_sms;                  /* persistent grid size; 0 = all SMs */
  int debug_flags;              /* bit 0: the L1 epilogue also writes its raw fp32 gate|up accumulators
                                   to the DEBUG workspace region ([P, 2I], pool-row order) and the
                                   call stops after L1; bit 1: the GEMM kernels record per-CTA
                                   wait/busy times of their roles into the PROF workspace region;
                                   bit 2: in the fused stream every L2 tile waits for one more L1
                                   completion than will ever arrive, and in the FP8 L1 GEMM the
                                   last stage of each CTA's last task is never loaded, so the call
                                   ends with MM_MOE_ERR_TIMEOUT after wait_timeout_ms (tests the
                                   device-side timeout path); bit 4: FP8 requant divides for every
                                   code (the fast path is bit-equal; for tests); 0 for normal use */
  int cta_pairs;                /* reserved: 0 (default) or 1; any other value makes mm_moe_forward
                                   return MM_MOE_ERR_UNSUPPORTED */
  int partials_bf16;            /* 0 (default): the L2 epilogue writes fp32 partials [K, T, H] and the
                                   combine sums them in fixed k order; 1: the partials are cast to
                                   bf16 (round to nearest even) first, halving their traffic (the
                                   L2 BF16 epilogue + combine of the pages' SM90 design) */
  float activation_clamp;       /* > 0: gate and up are each clamped to [-c, c] before the SwiGLU (the
                                   pages' optional activation clamp); <= 0 (default): no clamp */
  int precise_swiglu;           /* 0 (default): silu(g) = g * rcp.approx(1 + __expf(-g)), the pages'
                                   fast-math SwiGLU; 1: g / (1 + expf(-g)) with the IEEE division */
  int x_bf16;                   /* 0 (default): x holds e4m3 codes and x_sf their scales; 1: x is bf16
                                   [T, H] (row-major, 16-byte aligned), x_sf is ignored (may be NULL),
                                   and the gather quantises each row on its way into the pool with
                                   the variant's rule (MX: UE8M0 per 32, 448 * 2^e >= amax; F8: fp32
                                   max(amax, 1e-10) / 448 per 128).  Non-finite inputs give
                                   unspecified codes. */
  int early_combine;            /* fused stream (MX): 1 = once a CTA has no GEMM work left, its epilogue
                                   warps combine every token whose experts have finished L2 (the pages'
                                   early combine) and no combine kernel runs; 0 (default) = a combine
                                   kernel after the GEMM, which measures as fast or faster on one
                                   GB300.  Bit-identical either way. */
  int swap_ab;                  /* MX variant: which operand is the tensor-core MMA's M side.  0 (default):
                                   the tokens, in pool blocks of 128 (every MMA computes 128 token rows
                                   x 256 weight rows); 1: the weights (128 rows per MMA) with each pool
                                   block's tokens as N, rounded up to 16, so a block's MMA work follows
                                   its token count and an expert whose tokens fit one block streams
                                   its weights once (the pages' swap-AB form); 2: the same on 2-CTA
                                   clusters, 256 weight rows per MMA (tcgen05 cta_group::2, half of
                                   them and half of the block's tokens in each CTA of the pair).
                                   Results agree with the oracle either way; the forms sum the same
                                   products in a different tensor-core order, so their bits may
                                   differ. */
  int block_m;                  /* tokens per pool block: 0 (default) = the form's own choice (128 for
                                   swap_ab 0; for swap_ab 1, 160 when the expected tokens per expert
                                   T*K/E exceed 64, else 80); otherwise 128 (swap_ab 0) or 80 / 160
                                   (swap_ab 1 or 2), anything else MM_MOE_ERR_UNSUPPORTED */
  int f8_act_gran;              /* F8 variant: width of the intermediate's fp32 scale blocks along I (the
                                   pages' l2_act_sf_gran_k).  0 (default) or 128: per 128; 64: per 64,
                                   and the L2 GEMM dequantises each 64-wide half of a 128-K step with
                                   its own scale; -1: the pages' shape rule (128 when H % 512 == 0 and
                                   2*I % 512 == 0, else 64).  Any other value: MM_MOE_ERR_INVALID_ARG.
                                   The MX variant ignores it (its intermediate scales are UE8M0 per 32). */
  int shared_experts;           /* S >= 0 shared experts (default 0): experts E .. E+S-1 of w1 / w2 and
                                   their scales, which every token uses with weight 1 after its K
                                   routed slots; their outputs join the fixed-order top-k sum as slots
                                   K .. K+S-1.  w1, w2 and their scale arrays then hold E + S experts
                                   (mm_moe_weight_sf_size / mm_moe_prepare_weights take E + S), topk_idx
                                   still names routed experts only (ids >= E are out of range), and
                                   K + S <= 16, E + S <= 1024.  The shared experts' tiles run in the same
                                   launches as the routed ones. */
  int ring_blocks;              /* the intermediate as a wrapping ring of R pool blocks (DeepGEMM PR #440
                                   "Ring sizing, recycling, and why that granularity"): 0 (default) =
                                   the whole pool, one slot per block; R > 0 = R slots of 128 rows, block
                                   b using slot b % R, for the MX fused stream with swap_ab = 0 only
                                   (otherwise MM_MOE_ERR_UNSUPPORTED, as with retain_intermediate or
                                   debug_flags bit 0).  R >= ceil(T / 128) is required (else
                                   MM_MOE_ERR_INVALID_ARG).  A block's L1 tiles wait until every L2 tile
                                   of the block R slots back has read it.  The kernel shortens lag_units,
                                   for this launch, to the largest lag at which every lag + 1 consecutive
                                   experts own at most R / 2 blocks (0 if one expert owns more), so each
                                   of those waits points at tiles earlier in the stream and half the
                                   ring is slack; results are bit-identical to R = 0.  Routing
                                   that gives one expert more than R blocks (a token naming an expert
                                   twice) ends with MM_MOE_ERR_BAD_ROUTING, site 114, and no output. */
  void* trace_buf;              /* optional per-task trace (device memory, 16-byte aligned, zeroed by the
                                   caller; NULL = off, the default).  The token-M MX kernel (swap_ab = 0)
                                   then runs its timing instantiation (its timing branches cost the MMA
                                   issue loop some cycles; the trace itself is not timed) and writes one
                                   64-byte record per task it runs: uint32 cta, task (its index within
                                   the CTA), type (1 = L1, 2 = L2), expert, tile, pool block, valid rows,
                                   launch mode (3 = fused stream, 1 / 2 = the L1 / L2 launch of the
                                   two-launch path), then uint64 globaltimer nanoseconds: t_issue (the
                                   MMA warp issued the task's first k-block), t_mma_done (the epilogue
                                   saw the accumulator complete), t_epi_done (the first epilogue warp
                                   finished the task's output), and one reserved word.  Layout:
                                   [launch][CTA][cap] records with cap = trace_bytes / (64 * grid *
                                   launches), grid = the persistent grid (num_sms or the SM count),
                                   launches = 1 for the fused stream, 2 for two launches; tasks past
                                   cap are not recorded, and unwritten records keep type 0.  A buffer
                                   smaller than one record per CTA and launch: MM_MOE_ERR_INVALID_ARG;
                                   with the F8 variant or swap_ab > 0: MM_MOE_ERR_UNSUPPORTED (the
                                   pages' instrumented event traces; off the default path). */
  size_t trace_bytes;
  void* timing_events;          /* optional array of MM_MOE_NUM_TIMING_EVENTS cudaEvent_t (created by the
                                   caller) that mm_moe_forward records on `stream` at the start, between
                                   its kernels and at the end: [0] start, [1] dispatch done, [2] gather
                                   done, [3] L1 done, [4] L2 done, [5] combine done; NULL = none, and a
                                   NULL entry is skipped.  The GEMM of the fused stream and the combine
                                   are launched programmatically (they start their setup while the
                                   kernel before them finishes) unless an event is recorded between
                                   them and that kernel ([1]/[2], resp. [3]/[4]). */
} mm_moe_options;

#define MM_MOE_NUM_TIMING_EVENTS 6

/* Fill `opt` with the defaults. */
void mm_moe_default_options(mm_moe_options* opt);

/* Bytes of workspace mm_moe_forward needs for this shape (opt may be NULL = defaults). */
int mm_moe_workspace_size(const mm_moe_options* opt, int T, int H, int I, int E, int K, size_t* bytes);

/* Bytes of the prepared scale buffers w1_sfp / w2_sfp. */
int mm_moe_weight_sf_size(const mm_moe_options* opt, int H, int I, int E, size_t* w1_sfp_bytes,
                          size_t* w2_sfp_bytes);

/* One-time relayout of the weight scales into the layout the GEMM kernels
 * stream (MX: 512-byte blocks, one per 128 weight rows x 128 K, in the
 * tensor-memory scale-factor order; the L1 blocks pair 64 gate rows with the
 * matching 64 up rows).  The codes w1/w2 are used as given.
 * (llm-infra-atlas "07 · MegaMoE" §11: the weights are transformed once before use.) */
int mm_moe_prepare_weights(const mm_moe_options* opt, const void* w1_sf, const void* w2_sf, int H, int I,
                           int E, void* w1_sfp, void* w2_sfp, void* stream);

/* The forward (steps a1–a7 above).  `workspace` must hold mm_moe_workspace_size()
 * bytes; its contents need no initialisation and are overwritten. */
int mm_moe_forward(const void* x, const void* x_sf, const int32_t* topk_idx, const float* topk_w,
                   const void* w1, const void* w1_sfp, const void* w2, const void* w2_sfp, void* out, int T,
                   int H, int I, int E, int K, void* workspace, size_t workspace_bytes,
                   const mm_moe_options* opt, void* stream);

/* Step a1 alone, into caller buffers: cnt[E], blk_off[E+1] (in blocks of
 * block_m rows), slot[T*K] (pool row or -1), src[src_capacity] (t*K+k or -1 for
 * padding rows; rows past blk_off[E]*block_m are left untouched).  block_m must
 * be a multiple of 16 in [16, 256]; src_capacity >= T*K + min(T*K, E)*(block_m-1).
 * `scratch` (device, 4-byte aligned, at least 4*E bytes; mm_moe_dispatch_scratch_size
 * gives the size that lets the work spread over all SMs) receives per-CTA
 * expert counts; fewer bytes only means fewer CTAs.  `status` is a device
 * int[4], zeroed by the caller, that receives MM_MOE_ERR_BAD_ROUTING when
 * topk_idx holds values >= E or < -1. */
int mm_moe_dispatch_scratch_size(int T, int K, int E, size_t* bytes);
int mm_moe_dispatch(const int32_t* topk_idx, int T, int K, int E, int block_m, int32_t* cnt,
                    int32_t* blk_off, int32_t* slot, int32_t* src, int64_t src_capacity, void* scratch,
                    size_t scratch_bytes, int32_t* status, void* stream);

/* mm_moe_dispatch for callers that cannot allocate device memory: no
 * counterpart in the MegaMoE pages; it exists for the integration.  Some
 * callers have no way to hand the library scratch: their runtime owns every
 * device allocation (pre-reserved pools, no cudaMalloc after start-up) or the
 * call sits on a latency path where an allocation could synchronise the
 * device.  This entry point takes the same arguments as mm_moe_dispatch minus
 * the scratch and calls no allocator; its per-CTA counts live in one fixed
 * 256 KiB device array inside the library, which every GPU that loads the
 * library holds until the process exits.
 *   - The first call on each device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - The array holds 65536 counts, one per (CTA, expert): the work is
 *     spread over at most min(#SMs, ceil(T*K/512), 65536/E) CTAs (at least
 *     64 for E <= 1024), so every shape mm_moe_dispatch accepts fits and the
 *     routing is the same as mm_moe_dispatch's.
 *   - All calls share the array and each call rewrites the entries it reads,
 *     so calls that may overlap on the GPU (other streams, other host
 *     threads) race with one another: serialise them. */
int mm_moe_dispatch_noalloc(const int32_t* topk_idx, int T, int K, int E, int block_m, int32_t* cnt,
                            int32_t* blk_off, int32_t* slot, int32_t* src, int64_t src_capacity,
                            int32_t* status, void* stream);

/* Copy the routing of the last forward out of a workspace (same shapes as mm_moe_dispatch;
 * block_m is reported through *block_m). */
int mm_moe_read_routing(const void* workspace, const mm_moe_options* opt, int T, int H, int I, int E, int K,
                        int32_t* cnt, int32_t* blk_off, int32_t* slot, int32_t* src, int* block_m,
                        void* stream);

/* Copy the requantised intermediate (step a4) of pool rows [0, rows) out of a
 * workspace: codes u8 [rows, I] and scales (MX: u8 [rows, I/32]; F8: f32
 * [rows, I/128]).  Needs opt->retain_intermediate on the forward call when the
 * fused path recycles its activation ring. */
int mm_moe_read_intermediate(const void* workspace, const mm_moe_options* opt, int T, int H, int I, int E,
                             int K, int64_t rows, uint8_t* codes, void* sf, void* stream);

/* Diagnostics: device address and size of one internal region of a
 * workspace laid out for this shape and these options.  region: 0 status,
 * 1 cnt, 2 blk_off, 3 slot, 4 src, 5 pooled activations, 6 their scales,
 * 7 intermediate codes, 8 intermediate scales, 9 fp32 partials [K, T, H],
 * 10 debug accumulators (debug_flags bit 0 only), 11 per-CTA role timings of the two
 * GEMM kernels (debug_flags bit 1 only: uint64 [2][grid][8] nanoseconds and counts). */
int mm_moe_workspace_region(const void* workspace, const mm_moe_options* opt, int T, int H, int I, int E, int K,
                            int region, void** ptr, size_t* bytes);

/* Synchronise `stream`, then read the device status word of `workspace`.
 * Returns MM_MOE_OK, MM_MOE_ERR_TIMEOUT, MM_MOE_ERR_BAD_ROUTING or
 * MM_MOE_ERR_CUDA; *where (if non-NULL) receives the code of the check that
 * fired.  The word is cleared by the next forward.
 * Wait sites of MM_MOE_ERR_TIMEOUT:
 *   MX GEMM   101 a free pipeline stage, 102 a stage's data, 103 the free
 *             accumulator, 104 the finished accumulator, 105 a pool block's
 *             gathered rows, 106 a pool block's L1 tiles, 107 / 108 the
 *             tile-group queue, 109 an early-combine token's experts, 110 an
 *             early-combine deferred entry;
 *             111 / 112 the exit drain of bulk copies / MMAs (after an earlier
 *             error), 113 a ring slot still read by the L2 tiles of the
 *             block ring_blocks back; swapped and paired kernels 121-152
 *             likewise;
 *   FP8 GEMM  201 a free pipeline stage, 202 a stage's data, 203 a free
 *             partial buffer, 204 a finished partial (the commit waiter), 205
 *             the epilogue's amax rendezvous, 211 / 212 the exit drains;
 *   EP        301 a cross-rank barrier (mm_moe_ep_barrier's own status word). */
int mm_moe_sync_status(const void* workspace, void* stream, int* where);

/* ---------------------------------------------------------------------------
 * Expert parallelism over N ranks: the pages' EP dispatch and combine (llm-infra-
 * atlas "07 · MegaMoE" §7 count -> push metadata -> pull data, §9 combine;
 * DeepGEMM PR #440 "How it works").  Rank r owns experts [r*E/N, (r+1)*E/N)
 * (E % N == 0).  One EP forward, on every rank:
 *   1. mm_moe_ep_count: this rank's pairs per expert -> counts[E] (device).
 *   2. the caller exchanges the counts (an all-gather: counts_all[N][E] on the host),
 *      and mm_moe_ep_plan gives every routed pair its row in the owner's receive
 *      buffer and this rank's receive row count;
 *   3. mm_moe_ep_push_meta: each pair's (source rank, pair index, local expert,
 *      weight) is stored into its owner's receive-metadata buffer;
 *   4. barrier; mm_moe_ep_pull: the owner copies each received row's activations
 *      and scales from the source rank's x into its own receive buffers, and writes
 *      the local routing (one slot a row) that mm_moe_forward then runs on with
 *      E/N experts and K = 1 (the received pairs as tokens);
 *   5. barrier; mm_moe_ep_combine: each rank sums, for each of its tokens, the
 *      bf16 outputs of its pairs' rows at their owners, in k order, in fp32, and
 *      rounds once to bf16: the bf16-partials combine of the pages (each pair's
 *      output reaches the combine as bf16).
 * Peer buffers are reached through device arrays of N device pointers (peer_*[r]
 * is rank r's buffer, [rank] this rank's own), read or written with plain
 * loads and stores from this GPU's kernels; no TMA and no multicast touches a
 * peer's memory.  The barriers between steps are the caller's (host collectives
 * with a timeout), so no kernel waits on another rank.  Every call is
 * stream-ordered and asynchronous; none allocates.
 * Receive-row order on an owner: local expert, then source rank, then the
 * source's pairs in ascending (token, slot): with tokens numbered rank-major, the
 * same order as mm_moe_dispatch's over all ranks' tokens. */

/* counts[e] (device int32 [E], overwritten) = pairs of topk_idx [T, K] (device)
 * with expert e; ids < 0 or >= E are not counted. */
int mm_moe_ep_count(const int32_t* topk_idx, int T, int K, int E, int32_t* counts, void* stream);

/* Host planning (no GPU).  counts_all: host [N][E], counts_all[r][e] = rank r's
 * pairs with expert e (this rank's row must equal its own topk_idx); topk_idx:
 * host [T, K] of this rank.  Writes send_row (host [T*K]): the pair's row in its
 * owner's receive buffer (owner = expert / (E/N)), -1 for masked or out-of-range
 * ids; *recv_rows: the rows this rank receives; recv_expert (host [recv_capacity],
 * optional): each received row's local expert.  MM_MOE_ERR_INVALID_ARG on bad
 * sizes, counts that disagree with topk_idx, or recv_capacity < *recv_rows. */
int mm_moe_ep_plan(const int32_t* counts_all, const int32_t* topk_idx, int T, int K, int E, int N, int rank,
                   int32_t* send_row, int64_t* recv_rows, int32_t* recv_expert, int64_t recv_capacity);

/* Step 3.  topk_idx, topk_w [T, K] and send_row [T*K] are this rank's (device);
 * peer_meta: device array of N pointers to each rank's receive metadata, int32
 * [rows][4] = (source rank, pair index t*K+k, local expert, weight bits). */
int mm_moe_ep_push_meta(const int32_t* topk_idx, const float* topk_w, const int32_t* send_row, int T, int K,
                        int E, int N, int rank, void* const* peer_meta, void* stream);

/* Step 4.  meta: this rank's receive metadata (device int32 [rows][4], written by
 * step 3 on every rank); peer_x / peer_x_sf: device arrays of N pointers to each
 * rank's x [T_r, H] (e4m3 bytes) and x_sf (MX: UE8M0 [T_r, H/32]; F8: fp32
 * [T_r, H/128]); K: slots per token on every rank.  Writes x_recv [rows, H],
 * x_sf_recv (same layout), topk_idx_recv / topk_w_recv [rows] (K = 1 routing over
 * the E/N local experts). */
int mm_moe_ep_pull(const int32_t* meta, int64_t rows, int K, int H, int variant, const void* const* peer_x,
                   const void* const* peer_x_sf, void* x_recv, void* x_sf_recv, int32_t* topk_idx_recv,
                   float* topk_w_recv, void* stream);

/* Step 5.  peer_out: device array of N pointers to each rank's bf16 [rows_r, H]
 * output of its local forward; topk_idx [T, K] and send_row [T*K] this rank's
 * (device).  out [T, H] bf16: the fixed-k-order sum, 0 for a token with no
 * valid slot. */
int mm_moe_ep_combine(const int32_t* topk_idx, const int32_t* send_row, int T, int K, int E, int N, int H,
                      const void* const* peer_out, void* out, void* stream);

/* Push form of step 5 (the pages' combine, Atlas §9): every owner stores each
 * received row's bf16 output (out_recv [rows, H], its local forward's output) into
 * the source rank's partial buffer at the pair's place: peer_partials[r] is rank
 * r's bf16 [T_r * K, H] (row t*K + k).  meta is the owner's receive metadata
 * (step 3).  Rows of masked slots are never written. */
int mm_moe_ep_push_out(const int32_t* meta, int64_t rows, int H, const void* out_recv,
                       void* const* peer_partials, void* stream);

/* After every owner's push (a barrier): out[t] = bf16(sum over k of partials[t*K + k]
 * for the slots with 0 <= topk_idx < E), the sum in fp32 in k order; 0 for a token
 * with no valid slot.  partials: this rank's bf16 [T*K, H]. */
int mm_moe_ep_combine_local(const int32_t* topk_idx, int T, int K, int E, int H, const void* partials,
                            void* out, void* stream);

/* The pages' num_tokens_bound contract (PR #440): with every rank's token count at
 * most num_tokens_bound (the same bound on every rank), a rank receives at most
 * *rows = N * num_tokens_bound * min(K, E/N) rows (each token sends one row to each
 * distinct expert it picks, at most E/N of them on one rank), so receive buffers of
 * that size can be allocated once, alike on every rank.  mm_moe_ep_plan refuses a
 * receive count above the capacity it is given. */
int mm_moe_ep_recv_capacity(int num_tokens_bound, int K, int E, int N, int64_t* rows);

/* Bounded cross-rank barrier for the EP steps (the pages' NVLink barrier,
 * llm-infra-atlas "07 · MegaMoE" §10), an alternative to a host barrier:
 * peer_flags is a device array of N pointers to each rank's uint32 [N] flag array
 * (zeroed once at allocation, peer-accessible); `epoch` must grow by at least one
 * per call.  The kernel stores epoch into slot `rank` of every rank's array, then
 * waits until all N slots of its own array have reached epoch.  After timeout_ms
 * (0: 2000) it records MM_MOE_ERR_TIMEOUT in status (device int32[4]; [1] = 301,
 * [2] = the first rank missing) and returns, so a lost rank never hangs the GPU.
 * N <= 64. */
int mm_moe_ep_barrier(void* const* peer_flags, int N, int rank, uint32_t epoch, unsigned timeout_ms, int32_t* status,
                      void* stream);

/* Every rank's barrier in one cooperative launch on one device (block r is rank
 * r), for a device that holds all ranks' flag arrays; ranks whose bit is set in
 * `absent` skip theirs.  This is how the barrier is exercised on one GPU without
 * separate launches that wait on one another.  MM_MOE_ERR_UNSUPPORTED when the
 * device cannot hold N co-resident blocks. */
int mm_moe_ep_barrier_ranks(void* const* peer_flags, int N, uint32_t epoch, unsigned timeout_ms, uint64_t absent,
                            int32_t* status, void* stream);

/* Human-readable name of a return code. */
const char* mm_moe_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* MM_MOE_H_ */

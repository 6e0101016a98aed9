// Block-scaled grouped GEMMs of the MoE layer on tcgen05 (kind::mxf8f6f4):
// e4m3 activations x e2m1 weights, one UE8M0 scale per 32 contraction elements.
//
// Tile: M = 128 pool rows (the tokens of one pool block of one expert) x
// N = 256 weight rows x K in stages of 128.  On GB300 one M=128, K=32 tcgen05
// MMA takes the same tensor-pipe time for every N up to 256 (measured), so the
// weights are the N operand at its full width and a block with few tokens
// only wastes accumulator rows, not MMA issue slots.
//   L1 task: the 256 rows are 128 gate rows and the matching 128 up rows, so a
//            token's gate and up values for 128 intermediate columns sit in one
//            TMEM lane and SwiGLU, the top-k weight and the per-32 UE8M0
//            requant are thread-local (llm-infra-atlas "07 · MegaMoE" §8).
//   L2 task: 256 output columns; the epilogue writes fp32 partials part[k][t][h].
//
// One kernel, three task streams (mode):
//   1  all L1 tiles, expert by expert (weight tile outer, pool block inner)
//   2  all L2 tiles, same order
//   3  one lag-ordered stream (DeepGEMM PR #440, "How it works"): segment u
//      holds expert u's L1 tiles and then expert (u - lag)'s L2 tiles, so L2
//      trails L1 by `lag` experts.  The pool rows are gathered in the kernel by
//      two gather warps per CTA that publish per-block row counts; the L1
//      epilogue publishes per-block tile counts; a producer waits on them
//      (acquire, bounded) before it loads a block ("07 · MegaMoE" §6: per-block
//      arrival counters instead of kernel boundaries).  Every wait points at a
//      task earlier in the global order and every CTA is resident (one per
//      SM, grid <= #SMs) and works its tasks in that order, so the stream
//      cannot deadlock.
//
// Warps (512 threads in four warpgroups, one CTA per SM):
//   0..3    TMA producers: lane l of warp p owns pipeline stage p + 4 l.  A
//           TMA-issuing thread keeps only about four bulk-tensor copies in
//           flight (measured on GB300), so each stage has its own issuer.  Per stage: one token
//           tile (box of 32, 64 or 128 rows by the block's size), one weight
//           tile (16U4_ALIGN16B, unpacked to 1 byte per element in shared
//           memory; L1 fetches gate and up rows with one 3-D copy) and the
//           scale chunks.
//   4..11   epilogue: one token row per thread, the two warps of a TMEM lane
//           quadrant split the columns.  Each thread copies its 128
//           accumulator columns into registers and releases TMEM at once, so
//           the next tile's MMAs overlap the SwiGLU / requant / stores.
//           setmaxnreg gives these two warpgroups 176 registers a thread and
//           the other two 80; the host refuses to launch unless the kernel
//           starts with exactly the 128 registers a thread the split assumes.
//   12      TMEM allocator + single-thread MMA issuer (tcgen05.cp of the scales
//           into TMEM, 4 MMAs of K=32 per stage).
//   13..14  gather warps (mode 3); warp 15 idles.
// Every wait is bounded: on a deadline the kernel records MM_MOE_ERR_TIMEOUT
// and a site code and returns.
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "sched.cuh"
#include "stream.cuh"

namespace mm {
namespace {

constexpr int kStages = 4;
constexpr int kProducers = 4;          // warps of TMA-issuing threads: thread (warp p, lane l) fills stage p + 4 l
constexpr int kEpiWarp0 = kProducers;  // eight epilogue warps, two per TMEM lane quadrant
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = kEpiWarp0 + kEpiWarps;
constexpr int kGatherWarp0 = kMmaWarp + 1;
constexpr int kGatherWarps = 2;
constexpr int kSchedWarp = kGatherWarp0 + kGatherWarps;   // deals tile groups to this CTA's roles
constexpr int kQueueConsumers = kStages + 1 + kEpiWarps;   // arrivals that free a queue slot
constexpr int kThreads = 512;          // four warpgroups
static_assert((kSchedWarp + 1) * 32 <= kThreads, "warp roles");
constexpr int kLaunchRegs = 128;       // 65536 / 512
constexpr int kSmallRegs = 72;         // WG0 (producers)
constexpr int kMmaRegs = 104;          // WG3 (MMA issuer with its per-stage descriptors, gather, scheduler)
constexpr int kEpiRegs = 168;          // WG1, WG2 (epilogue)
static_assert(128 * kSmallRegs + 128 * kMmaRegs + 2 * 128 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kBN = 256;               // weight rows per tile (MMA N)
constexpr int kTokBytes = kBT * kBK;   // 128 token rows x 128 K
constexpr int kWgtBytes = kBN * kBK;   // 256 weight rows x 128 K, 1 byte per element in smem
// A 16U4_ALIGN16B tile load completes the mbarrier transaction count with the
// PACKED bytes it read from global memory (half a byte per element), not with
// the unpacked bytes it wrote to shared memory (measured on GB300).
constexpr int kWgtTxBytes = kWgtBytes / 2;
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = kBN;           // scale-factor columns after the accumulator
constexpr int kSfColsPerStage = 12;    // 4 (tokens) + 8 (weights)

// wait-site codes reported through the status word
enum : int {
  kSiteEmpty = 101, kSiteFull = 102, kSiteTmemEmpty = 103, kSiteTmemFull = 104,
  kSiteGathered = 105, kSiteL1Done = 106, kSiteQueueEmpty = 108,   // 109, 110: early combine (stream.cuh)
  kSiteDrainCopies = 111, kSiteDrainMma = 112, kSiteRingFree = 113, kSiteRingSize = 114
};

struct Args {
  int T, H, I, E, K;
  int BT, CPB;         // pool rows per block (128) and 128-row scale chunks per block (1)
  int KB1, KB2, NB1, NB2;
  int mode;            // 1, 2 or 3 (see above)
  int per_block;       // deal each (weight tile, pool block) as its own group
  int lag;             // mode 3: experts by which L2 trails L1
  int l1_extra;        // mode 3: extra L1 completions an L2 tile waits for (0; 1 = a wait that cannot end)
  const int* cnt;
  const int* blk_off;
  const int* src;
  const float* topk_w;
  const uint8_t* x;          // mode 3 gather: activations [T, H] and scales [T, H/32], or bf16 [T, H]
  const uint8_t* x_sf;
  int x_bf16;                // the gather quantises bf16 rows (x_sf unused)
  uint8_t* pool_x;           // [P, H]
  uint8_t* pool_x_sf;        // chunks [P/128][H/128][512]
  const uint8_t* sfw1;       // prepared weight scale chunks (two per tile and k-block)
  const uint8_t* sfw2;
  uint8_t* pool2;            // intermediate codes [P, I]
  uint8_t* pool2_sf;         // intermediate scale chunks [P/128][I/128][512]
  float* partials;           // [K, T, H] fp32, or bf16 when pbf16
  int pbf16;                 // partials cast to bf16 (round to nearest even)
  float clamp;               // gate and up clamped to [-clamp, clamp] before the SwiGLU (+inf: none)
  int precise;               // SwiGLU with expf and the IEEE division (else the fast-math form)
  float* dbg;                // raw L1 accumulators [P, 2I] or null
  int* ctr_gather;           // mode 3: rows gathered per pool block
  int* ctr_l1;               // mode 3: L1 epilogue warps finished per pool block
  int* sched;                // tile groups handed out so far (zero at launch)
  int early_combine;         // mode 3: the epilogue warps combine tokens after their last task
  const int32_t* topk_idx;   // early combine: routing [T, K] and the bf16 output [T, H]
  __nv_bfloat16* out;
  int* cmb;                  // early combine counters: tokens taken, deferred, classified, deferred taken
  int* ctr_l2;               // [E] L2 epilogue warps finished per expert (early combine)
  int* deferred;             // [T] tokens pass 1 could not combine yet, as t + 1 (0: not written)
  int ring;                  // mode 3: intermediate slots of a wrapping ring (block b in slot b % ring); 0 = none
  int* ctr_l2r;              // [blocks] L2 tiles that have read a block's intermediate (ring reuse)
  int* status;
  uint64_t timeout_ns;
  unsigned long long* prof;  // per-CTA wait/busy nanoseconds (debug_flags bit 1) or null
  TraceRec* trace;           // per-task records, trace_cap per CTA, or null
  int trace_cap;
};

struct Maps {
  CUtensorMap w1, w2;                       // weights
  CUtensorMap x32, x64, x128;               // pooled activations, boxes of 32/64/128 rows
  CUtensorMap a32, a64, a128;               // intermediate codes
};


struct SmemLayout {
  static constexpr int tok = 0;
  static constexpr int wgt = tok + kStages * kTokBytes;
  static constexpr int sft = wgt + kStages * kWgtBytes;
  static constexpr int sfw = sft + kStages * kSFChunk;
  static constexpr int meta = sfw + kStages * 2 * kSFChunk;   // blk_off[E+1], cnt[E], queue[kQueue]
  static constexpr int meta_ints(int E) { return (E + 1) + E + kQueue; }
  static constexpr int bars_after_meta(int E) { return meta + (meta_ints(E) * 4 + 15) / 16 * 16; }
  // full[S], empty[S], tfull, tempty, qfull[Q], qempty[Q], drain
  static constexpr int nbars = 2 * kStages + 2 + 2 * kQueue + 1;
  static constexpr int total(int E) { return bars_after_meta(E) + nbars * 8 + 16; }
};
static_assert(SmemLayout::total(kMaxE) + 1024 <= 232448, "shared memory budget");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A = e4m3 (0) in
// bits [9:7], B = e2m1 (5) in [12:10], both K-major, N>>3 in [22:17], UE8M0
// scales (bit 23), M>>4 in [28:24]; the scale-factor byte selectors of B and A
// sit in [5:4] and [30:29].
__device__ __forceinline__ uint32_t make_idesc(int sf_id) {
  return (0u << 7) | (5u << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (static_cast<uint32_t>(sf_id) << 29) | (static_cast<uint32_t>(sf_id) << 4);
}

// SwiGLU x top-k weight and UE8M0 requant of one 32-column block c of an L1
// tile for one token row: gate g, up u (fp32 bits, both overwritten).
__device__ __forceinline__ void l1_block(uint32_t (&g)[32], uint32_t (&u)[32], int c, bool live, float w,
                                         size_t row, int n, const Args& args, uint8_t* crow, uint8_t* sfrow) {
  if (!live) return;
  if (args.dbg) {
    float* drow = args.dbg + row * 2 * args.I;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      drow[n * 128 + c * 32 + jj] = __uint_as_float(g[jj]);
      drow[args.I + n * 128 + c * 32 + jj] = __uint_as_float(u[jj]);
    }
  }
  if (args.clamp < INFINITY) {   // the optional activation clamp, a pass of its own
    const float cl = args.clamp;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      g[jj] = __float_as_uint(fminf(fmaxf(__uint_as_float(g[jj]), -cl), cl));
      u[jj] = __float_as_uint(fminf(fmaxf(__uint_as_float(u[jj]), -cl), cl));
    }
  }
  float amax = 0.f;
  if (args.precise) {
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const float av = silu_precise(__uint_as_float(g[jj])) * __uint_as_float(u[jj]) * w;
      g[jj] = __float_as_uint(av);
      amax = fmaxf(amax, fabsf(av));
    }
  } else {
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const float av = silu_fast(__uint_as_float(g[jj])) * __uint_as_float(u[jj]) * w;
      g[jj] = __float_as_uint(av);
      amax = fmaxf(amax, fabsf(av));
    }
  }
  const int ee = ue8m0_exponent_e4m3(amax);   // smallest e with 448 * 2^e >= max(amax, 1e-10)
  const float scale = exp2_neg(ee);
  uint32_t packed[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = cvt_e4m3x2(__uint_as_float(g[4 * i]) * scale, __uint_as_float(g[4 * i + 1]) * scale);
    const uint32_t hi = cvt_e4m3x2(__uint_as_float(g[4 * i + 2]) * scale, __uint_as_float(g[4 * i + 3]) * scale);
    packed[i] = lo | (hi << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(crow + c * 32);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  sfrow[c] = static_cast<uint8_t>(ee + 127);
}

__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSmallRegs)); }
__device__ __forceinline__ void regs_dec_mma() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kMmaRegs)); }
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs)); }

// The lag of a fused stream whose intermediate is a ring of R pool blocks.
// Block b's L1 tiles reuse the slot of block b - R only after the L2 tiles of
// that block have read it.  If every l + 1 consecutive experts own at most R
// blocks, block b - R belongs to an expert at least l + 1 before b's, whose L2
// tiles sit in an earlier segment of the stream: every wait for a free slot
// points at tiles dealt before it, so the stream cannot deadlock.  A window that
// fills the ring leaves no slack, though: b's L1 tiles then wait for L2 tiles
// dealt just before them.  So the lag is the largest l <= lag whose windows own
// at most R / 2 blocks (PR #440 likewise sets the lag near 0.45 of the ring), or
// 0 when one expert alone owns more.  All threads of the CTA call this (barriers
// inside); every CTA reads the same block offsets and takes the same lag.  If
// one expert alone owns more than R blocks (only possible when a token names an
// expert twice) the routing is rejected and the CTA stops at once.
__device__ int ring_lag(const int* blk, int E, int lag, int R, const Status& st, volatile int* s_abort) {
  auto fits = [&](int l, int cap) {
    bool bad = false;
    for (int u = threadIdx.x; u < E; u += blockDim.x) bad |= blk[u + 1] - blk[u - l < 0 ? 0 : u - l] > cap;
    return !__syncthreads_or(bad);
  };
  if (!fits(0, R)) {
    if (threadIdx.x == 0) {
      report_error(st, MM_MOE_ERR_BAD_ROUTING, kSiteRingSize);
      *s_abort = 1;
    }
    __syncthreads();
    return 0;
  }
  const int half = R / 2;
  if (!fits(0, half)) return 0;
  int lo = 0, hi = lag;   // fits(lo, half) holds; the answer lies in [lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (fits(mid, half)) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// kProf: record per-role wait and busy times (debug_flags bit 1) and/or per-task
// trace records (Options.trace_buf).  A separate instantiation, because even
// untaken timing branches slow the MMA issue loop.
template <bool kProf>
__global__ void __launch_bounds__(kThreads, 1) gemm_mx_kernel(const __grid_constant__ Maps maps, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int E = args.E;
  int* s_blk = reinterpret_cast<int*>(smem + SmemLayout::meta);
  int* s_cnt = s_blk + E + 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::bars_after_meta(E));
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 1;
  const Queue q{tempty + 1, tempty + 1 + kQueue, s_cnt + E};
  uint64_t* drain = tempty + 1 + 2 * kQueue;   // the MMA issuer's last commit
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + SmemLayout::nbars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Status st{args.status, args.timeout_ns};
  int lag = args.mode == 3 ? args.lag : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps);
    mbar_init(drain, 1);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&q.full[i], 1);
      mbar_init(&q.empty[i], kQueueConsumers);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp < kProducers && lane == 0) {
    prefetch_tmap(&maps.w1);
    prefetch_tmap(&maps.w2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  // with a programmatic launch the setup above overlaps the routing kernel; everything
  // below reads what that kernel (or earlier work on the stream) wrote
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += kThreads) s_blk[i] = args.blk_off[i];
  for (int i = threadIdx.x; i < E; i += kThreads) s_cnt[i] = args.cnt[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const int nblk = s_blk[E];
  if (args.mode == 3 && args.ring > 0) lag = ring_lag(s_blk, E, lag, args.ring, st, s_abort);
  Sched sch{s_blk, s_cnt, E, args.NB1, args.NB2, args.mode, lag};
  sch.per_block = args.per_block != 0;

  const int wg = warp >> 2;
  // setmaxnreg sits inside each warpgroup's branch: after a join ptxas would
  // have to compile the code below for the smaller budget
  if (wg == 0) {
    regs_dec();
    // ------------------------------------------------------------------ TMA producers
    if (warp + kProducers * lane < kStages) {
      const int p = warp + kProducers * lane;  // this thread fills stage p, phases 0,1,0,...
      const uint64_t pol_w = policy_evict_first();    // a tile group's last pass over its weights
      const uint64_t pol_wk = policy_evict_normal();  // earlier passes: the next block reads them again
      const uint64_t pol_t = policy_evict_last();
      uint8_t* tk = smem + SmemLayout::tok + p * kTokBytes;
      uint8_t* wg = smem + SmemLayout::wgt + p * kWgtBytes;
      uint8_t* st_ = smem + SmemLayout::sft + p * kSFChunk;
      uint8_t* sw = smem + SmemLayout::sfw + p * 2 * kSFChunk;
      uint64_t w_empty = 0;
      int step = 0;                             // global k-block step of this CTA
      bool armed = false;                       // a phase of full[p] was armed: its copies land before exit
      uint32_t armed_parity = 0;
      for (Cursor c; !*s_abort && sch.next(c, q, st, s_abort, false, lane);) {
        const Task& t = c.t;
        const bool l1 = t.type == 1;
        const int KB = l1 ? args.KB1 : args.KB2;
        int kb = ((p - step) % kStages + kStages) % kStages;   // first k-block of this task on stage p
        if (kb < KB && args.mode == 3) {
          // the block's rows must be in the pool before they are loaded
          const bool ok = l1 ? wait_counter_geq(args.ctr_gather + t.b, t.valid, st, s_abort, kSiteGathered)
                             : wait_counter_geq(args.ctr_l1 + t.b, args.NB1 * kEpiWarps + args.l1_extra, st, s_abort,
                                              kSiteL1Done);
          if (!ok) break;
          fence_proxy_async_global();
        }
        const CUtensorMap* tt = t.valid <= 32 ? (l1 ? &maps.x32 : &maps.a32)
                                              : (t.valid <= 64 ? (l1 ? &maps.x64 : &maps.a64)
                                                               : (l1 ? &maps.x128 : &maps.a128));
        const int rows = t.valid <= 32 ? 32 : (t.valid <= 64 ? 64 : 128);
        const uint32_t bytes = rows * kBK + kWgtTxBytes + 2 * kSFChunk + kSFChunk;
        const uint8_t* sfw = (l1 ? args.sfw1 : args.sfw2) +
                             (static_cast<size_t>(t.e) * (l1 ? args.NB1 : args.NB2) + t.n) * KB * 2 * kSFChunk;
        const int tb = (!l1 && args.ring) ? t.b % args.ring : t.b;   // the block's intermediate slot
        const uint8_t* sft = (l1 ? args.pool_x_sf : args.pool2_sf) + static_cast<size_t>(tb) * KB * kSFChunk;
        for (; kb < KB; kb += kStages) {
          const uint32_t phase = ((step + kb) / kStages) & 1;
          const uint64_t t0 = kProf ? globaltimer() : 0;
          if (!mbar_wait(&empty[p], phase ^ 1, st, s_abort, kSiteEmpty)) break;
          if (kProf) w_empty += globaltimer() - t0;
          mbar_arrive_expect_tx(&full[p], bytes);
          armed = true;
          armed_parity = phase;
          const int kbe = t.rev ? KB - 1 - kb : kb;   // the k-block this stage carries
          const int kc = kbe * kBK;
          tma_load_2d(tk, tt, &full[p], kc, tb * kBT, pol_t);
          bulk_load(st_, sft + static_cast<size_t>(kbe) * kSFChunk, kSFChunk, &full[p]);
          const uint64_t pw = t.last ? pol_w : pol_wk;
          if (l1) tma_load_3d(wg, &maps.w1, &full[p], kc, t.e * 2 * args.I + t.n * 128, 0, pw);
          else tma_load_2d(wg, &maps.w2, &full[p], kc, t.e * args.H + t.n * kBN, pw);
          bulk_load(sw, sfw + static_cast<size_t>(kbe) * 2 * kSFChunk, 2 * kSFChunk, &full[p]);
        }
        step += KB;
      }
      // the copies of the last armed phase have landed before the shared memory goes away
      // (at once on a normal exit, where the MMA issuer consumed every phase)
      if (armed) mbar_wait_drain(&full[p], armed_parity, st, kSiteDrainCopies);
      if (kProf && args.prof) atomicAdd(&args.prof[blockIdx.x * 8 + 0], static_cast<unsigned long long>(w_empty));
    }
  } else if (wg == 3) {
    regs_dec_mma();
    if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // The issuing thread, not the tensor pipe, is the limit when every MMA's
      // descriptors are rebuilt after its stage's wait: walk the CTA's k-block
      // stream one round of kStages at a time so that each stage's descriptors
      // and TMEM columns are fixed offsets from values computed once here.
      const uint64_t dtok = make_smem_desc(smem_u32(smem + SmemLayout::tok), 16, 1024, 2);
      const uint64_t dwgt = make_smem_desc(smem_u32(smem + SmemLayout::wgt), 16, 1024, 2);
      const uint64_t dsft = make_smem_desc(smem_u32(smem + SmemLayout::sft), 0, 128, 0);
      const uint64_t dsfw = make_smem_desc(smem_u32(smem + SmemLayout::sfw), 0, 128, 0);
      uint32_t phase = 0;
      int it = 0, kb = 0, KB = 0;
      Cursor cur;
      uint64_t w_full = 0, w_tempty = 0;   // SM cycles (clock64) spent in these waits
      const uint64_t t_start = globaltimer();
      const long long c_start = clock64();
      // start_task: the accumulator must have been drained by the epilogue
      auto start_task = [&]() -> bool {
        if (*s_abort || !sch.next(cur, q, st, s_abort, false, lane)) return false;
        KB = cur.t.type == 1 ? args.KB1 : args.KB2;
        const long long t0 = kProf ? clock64() : 0;
        if (!mbar_wait(tempty, (it & 1) ^ 1, st, s_abort, kSiteTmemEmpty)) return false;
        if (kProf) w_tempty += clock64() - t0;
        tc_fence_after();
        return true;
      };
      bool live = start_task();
      while (live) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
          if (live) {
            const long long t1 = kProf ? clock64() : 0;
            if (!mbar_wait(&full[s], phase, st, s_abort, kSiteFull)) {
              live = false;
            } else {
              if (kProf) {
                w_full += clock64() - t1;
                if (args.trace && kb == 0 && it < args.trace_cap)
                  args.trace[static_cast<size_t>(blockIdx.x) * args.trace_cap + it].t_issue = globaltimer();
              }
              tc_fence_after();
              const uint32_t sft_col = tmem + kSfCol0 + s * kSfColsPerStage;
              const uint32_t sfw_col = sft_col + 4;
              tc_cp_32x128b_warpx4(sft_col, dsft + ((s * kSFChunk) >> 4));
              tc_cp_32x128b_warpx4(sfw_col, dsfw + ((s * 2 * kSFChunk) >> 4));
              tc_cp_32x128b_warpx4(sfw_col + 4, dsfw + (((s * 2 + 1) * kSFChunk) >> 4));
              const uint64_t da = dtok + ((s * kTokBytes) >> 4);
              const uint64_t db = dwgt + ((s * kWgtBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)   // K advances 32 bytes = 2 descriptor units
                tc_mma_mxf8f6f4(tmem, da + 2 * kk, db + 2 * kk, make_idesc(kk), sft_col, sfw_col, (kb | kk) != 0);
              tc_commit(&empty[s]);
              if (++kb == KB) {
                tc_commit(tfull);
                kb = 0;
                ++it;
                live = start_task();
              }
            }
          }
        }
        phase ^= 1;
      }
      // every MMA and scale copy this thread issued has completed before TMEM is freed
      tc_commit(drain);
      mbar_wait_drain(drain, 0, st, kSiteDrainMma);
      if (kProf && args.prof) {
        args.prof[blockIdx.x * 8 + 1] = w_full;
        args.prof[blockIdx.x * 8 + 2] = w_tempty;
        args.prof[blockIdx.x * 8 + 3] = globaltimer() - t_start;
        args.prof[blockIdx.x * 8 + 4] = it;
        args.prof[blockIdx.x * 8 + 7] = clock64() - c_start;   // SM cycles over the span
      }
    }
    __syncwarp();
    } else if (warp < kGatherWarp0 + kGatherWarps && args.mode == 3) {
      gather_rows(args, s_blk, s_cnt, sch, s_abort, warp - kGatherWarp0, kGatherWarps, lane, nblk);
    } else if (warp == kSchedWarp && lane == 0) {
      // ------------------------------------------------------------------ tile-group scheduler
      // Every dependency of a group (the gather and L1 tiles of the blocks an
      // L2 group reads) has a smaller index, so the group with the smallest
      // index not yet finished can always run.
      run_scheduler(sch, q, args.sched, st, s_abort, kSiteQueueEmpty);
    }
  } else {
    regs_inc();
    // ------------------------------------------------------------------ epilogue (8 warps)
    const int quad = warp & 3;             // TMEM lane quadrant this warp may access
    const int half = (warp - kEpiWarp0) >> 2;   // which half of the columns
    const int m = quad * 32 + lane;           // accumulator row = pool row inside the block
    const uint32_t tlane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    int it = 0;
    uint64_t w_tfull = 0, busy = 0;
    for (Cursor c; sch.next(c, q, st, s_abort, true, lane); ++it) {
      const Task& t = c.t;
      const bool live = m < t.valid;
      const size_t row = static_cast<size_t>(t.b) * kBT + m;
      const int s = live ? __ldg(args.src + row) : 0;
      const float w = (t.type == 1 && live) ? __ldg(args.topk_w + s) : 0.f;   // loaded before the wait
      if (t.type == 1 && args.ring && t.b >= args.ring) {
        // the slot's previous block (ring blocks back) must have been read by all of its L2 tiles
        bool ok = true;
        if (lane == 0) ok = wait_counter_geq(args.ctr_l2r + (t.b - args.ring), args.NB2, st, s_abort, kSiteRingFree);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        __syncwarp();
        if (!ok) break;
      }
      const uint64_t t0 = kProf ? globaltimer() : 0;
      if (!mbar_wait(tfull, it & 1, st, s_abort, kSiteTmemFull)) break;
      const uint64_t t1 = kProf ? globaltimer() : 0;
      tc_fence_after();
      // copy this thread's 128 accumulator columns, then hand TMEM back to the MMA warp
      // L1: gate [64h, 64h+64) and up [128+64h, 128+64h+64); L2: [128h, 128h+128)
      uint32_t r0[32], r1[32], r2[32], r3[32];
      {
        const int c0 = t.type == 1 ? 64 * half : 128 * half;
        const int c1 = t.type == 1 ? 128 + 64 * half : 128 * half + 64;
        tmem_ld_32x32b_x32(tlane + c0, r0);
        tmem_ld_32x32b_x32(tlane + c0 + 32, r1);
        tmem_ld_32x32b_x32(tlane + c1, r2);
        tmem_ld_32x32b_x32(tlane + c1 + 32, r3);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      if (t.type == 2 && args.ring && warp == kEpiWarp0 && lane == 0)
        red_release_gpu_add(args.ctr_l2r + t.b, 1);   // the MMAs are done: the slot has been read
      if (t.type == 1) {
        const int sb = args.ring ? t.b % args.ring : t.b;   // the block's intermediate slot
        uint8_t* crow = args.pool2 + (static_cast<size_t>(sb) * kBT + m) * args.I + t.n * 128;
        uint8_t* sfrow = args.pool2_sf + (static_cast<size_t>(sb) * (args.I / 128) + t.n) * kSFChunk +
                         (m & 31) * 16 + (m >> 5) * 4;
        l1_block(r0, r2, 2 * half, live, w, row, t.n, args, crow, sfrow);
        l1_block(r1, r3, 2 * half + 1, live, w, row, t.n, args, crow, sfrow);
        if (args.mode == 3) {
          fence_proxy_async_global();              // the codes are read by TMA later
          __syncwarp();
          if (lane == 0) red_release_gpu_add(args.ctr_l1 + t.b, 1);
        }
      } else {
        const int tt = s / args.K;
        const int k = s - tt * args.K;
        const int col0 = t.n * kBN + 128 * half;
        if (live && col0 < args.H) {
          const size_t off = (static_cast<size_t>(k) * args.T + tt) * args.H + col0;
          if (args.pbf16) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.partials) + off;
            st_bf16x32(dst, r0);
            st_bf16x32(dst + 32, r1);
            st_bf16x32(dst + 64, r2);
            st_bf16x32(dst + 96, r3);
          } else {
            float* dst = args.partials + off;
#pragma unroll
            for (int i = 0; i < 4; ++i) {   // 32-byte stores of the row's 128 columns
              st_global_v8(dst + 8 * i, r0 + 8 * i);
              st_global_v8(dst + 32 + 8 * i, r1 + 8 * i);
              st_global_v8(dst + 64 + 8 * i, r2 + 8 * i);
              st_global_v8(dst + 96 + 8 * i, r3 + 8 * i);
            }
          }
        }
        if (args.early_combine) {
          __syncwarp();   // the warp's partial stores before its release
          if (lane == 0) red_release_gpu_add(args.ctr_l2 + t.e, 1);
        }
      }
      if (kProf) {
        const uint64_t t2 = globaltimer();
        w_tfull += t1 - t0;
        busy += t2 - t1;
        if (args.trace && warp == kEpiWarp0 && lane == 0 && it < args.trace_cap) {
          TraceRec& r = args.trace[static_cast<size_t>(blockIdx.x) * args.trace_cap + it];
          r.cta = blockIdx.x; r.task = it; r.type = t.type; r.expert = t.e; r.tile = t.n; r.block = t.b;
          r.valid = t.valid; r.mode = args.mode;
          r.t_mma_done = t1;
          r.t_epi_done = t2;
        }
      }
    }
    if (args.early_combine) {
      if (args.pbf16) early_combine<__nv_bfloat16>(args, kEpiWarps, args.NB2, s_blk, st, s_abort, lane);
      else early_combine<float>(args, kEpiWarps, args.NB2, s_blk, st, s_abort, lane);
    }
    if (kProf && args.prof && warp == kEpiWarp0 && lane == 0) {
      args.prof[blockIdx.x * 8 + 5] = w_tfull;
      args.prof[blockIdx.x * 8 + 6] = busy;
    }
  }

  // every role has waited for the async work it issued (above), so after this
  // barrier no copy or MMA still targets this CTA's shared or tensor memory
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int mx_lag_auto(int E) {
  // PR #440 picks lag = clamp(round(0.45 x units), 8, 64) with units of up to
  // 8 pool blocks, a rule made for ranks pulling tokens into a bounded ring.  On
  // one GPU with the whole pool the dependency waits of a short lag cost more
  // than the intermediate's L2 locality saves: lag = E, every L1 tile before any
  // L2 tile, measured fastest at flash, decode and pro (lag 29 -> E: 802 -> 791,
  // 553 -> 529 and 4467 -> 4402 us a step).
  return E;
}

cudaError_t launch_gemm_mx(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s) {
  const Layout& L = *g.L;
  const WsPtrs& W = *g.W;
  Maps maps;
  Args a{};
  a.T = L.T; a.H = L.H; a.I = L.I; a.E = L.E; a.K = L.K;
  a.BT = kBT; a.CPB = 1;
  a.KB1 = L.H / 128; a.KB2 = L.I / 128; a.NB1 = L.I / 128; a.NB2 = (L.H + kBN - 1) / kBN;
  a.mode = mode;
  a.per_block = g.per_block ? 1 : 0;
  a.lag = lag < 0 ? 0 : (lag > L.E ? L.E : lag);   // a lag above E orders the stream as E does
  a.l1_extra = l1_extra;
  a.cnt = W.cnt; a.blk_off = W.blk_off; a.src = W.src; a.topk_w = g.topk_w;
  a.x = g.x; a.x_sf = static_cast<const uint8_t*>(g.x_sf); a.x_bf16 = g.x_bf16 ? 1 : 0;
  a.pool_x = W.pool_x; a.pool_x_sf = W.pool_x_sf;
  a.sfw1 = g.w1sfp; a.sfw2 = g.w2sfp;
  a.pool2 = W.pool2; a.pool2_sf = W.pool2_sf;
  a.partials = W.part; a.dbg = g.dbg;
  a.pbf16 = L.part_elem == 2;
  a.clamp = g.clamp;
  a.precise = g.precise;
  a.ctr_gather = W.ctr; a.ctr_l1 = W.ctr + L.nblk_cap;
  a.sched = W.ctr + 2 * L.nblk_cap + mode;
  a.early_combine = (mode == 3 && g.early_combine) ? 1 : 0;
  a.topk_idx = g.topk_idx;
  a.out = static_cast<__nv_bfloat16*>(g.out);
  a.cmb = W.ctr + 2 * L.nblk_cap + kSchedCounters;
  a.ctr_l2 = a.cmb + kCombineCounters;
  a.deferred = a.ctr_l2 + L.E;
  a.ring = mode == 3 ? static_cast<int>(L.ring) : 0;
  a.ctr_l2r = a.deferred + L.T;
  a.status = W.status; a.timeout_ns = g.timeout_ns;
  a.prof = g.prof ? g.prof + (mode == 2 ? 8 * 1024 : 0) : nullptr;
  a.trace = reinterpret_cast<TraceRec*>(g.trace);
  a.trace_cap = g.trace ? g.trace_cap : 0;
  {
    // W1 as (k, row, half): half 1 is I rows below half 0, so one box of
    // {128 k, 128 rows, 2 halves} is 128 gate rows followed by the matching 128 up rows
    const uint64_t dims[3] = {static_cast<uint64_t>(L.H), static_cast<uint64_t>(L.E) * 2 * L.I - L.I, 2};
    const uint64_t strides[2] = {static_cast<uint64_t>(L.H) / 2, static_cast<uint64_t>(L.I) * L.H / 2};
    const uint32_t box[3] = {128, 128, 2};
    if (encode_tmap(&maps.w1, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, g.w1, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (encode_tmap_2d(&maps.w2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w2, L.I, static_cast<uint64_t>(L.E) * L.H,
                     L.I / 2, 128, kBN, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  CUtensorMap* xm[3] = {&maps.x32, &maps.x64, &maps.x128};
  CUtensorMap* am[3] = {&maps.a32, &maps.a64, &maps.a128};
  for (int i = 0; i < 3; ++i) {
    if (encode_tmap_2d(xm[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool_x, L.H, L.P, L.H, 128, 32u << i,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode_tmap_2d(am[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool2, L.I, L.ring ? L.ring * kBT : L.P, L.I, 128, 32u << i,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  using KernelFn = void (*)(Maps, Args);
  const bool prof = a.prof != nullptr || a.trace != nullptr;
  const KernelFn kernels[2] = {gemm_mx_kernel<false>, gemm_mx_kernel<true>};
  const size_t smem = SmemLayout::total(L.E) + 1024;
  // the setmaxnreg split assumes exactly kLaunchRegs registers a thread at launch
  if (cudaError_t e = configure_kernel(reinterpret_cast<const void*>(kernels[prof]), kLaunchRegs,
                                       SmemLayout::total(kMaxE) + 1024))
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (mode == 3) {
    // the fused stream waits across CTAs: launch cooperatively so that every CTA is resident
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (g.pdl) {
    // start during the routing kernel: the setup before pdl_wait() overlaps its tail
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernels[prof], maps, a);
}

}  // namespace mm

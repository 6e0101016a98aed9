// Block-scaled grouped GEMMs of the MoE layer with the operands swapped: the
// weights are the MMA's M operand and the tokens of one pool block its N
// operand, with N = the block's token count rounded up to 16
// (llm-infra-atlas "07 · MegaMoE" §5: the token dimension of each MMA is sized
// to the block's valid rows, aligned to 16, and the block size follows the
// expected tokens per expert).  kind::mxf8f6f4: e2m1 weights (A) x e4m3 tokens
// (B), one UE8M0 scale per 32 contraction elements on both.
//
// On GB300 an M=128, K=32 MMA costs about N/2 cycles for N >= 128 and a floor
// near 55 cycles below that (measured), so a block of 140 tokens costs 144
// columns' work instead of two 128-token tiles, and an expert whose tokens fit
// one block (BT = 160 holds the 128 +- 11 tokens of the pro-shaped workload)
// streams each weight tile once.
//
// Task = (expert e, weight tile n, pool block b of <= BT tokens); per 128-K
// stage two MMAs share the token tile:
//   L1: A0 = 128 gate rows [n*128, +128), A1 = the matching 128 up rows, so
//       TMEM lane j holds gate and up of intermediate column n*128 + j for
//       every token (column), and the per-32 requant block of a token is the 32
//       lanes of one warp (one TMEM lane quadrant);
//   L2: A0, A1 = rows [n*256, +128) and [n*256 + 128, +128) of W2.
//
// Warps (512 threads in four warpgroups, one CTA per SM):
//   0..3    TMA producers: thread (warp p, lane l) owns stage p + 4 l
//   4..11   epilogue: the two warps of a lane quadrant take alternate 16-token
//           column chunks
//   12      TMEM allocator + single-thread MMA issuer
//   13..14  gather warps (fused stream); 15 tile-group scheduler
// Every wait is bounded; on a deadline the kernel records MM_MOE_ERR_TIMEOUT
// with a site code, waits (bounded) for the copies and MMAs it issued, frees
// TMEM and returns.
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "sched.cuh"
#include "stream.cuh"

namespace mm {
namespace {

constexpr int kThreads = 512;
constexpr int kProducers = 4;
constexpr int kEpiWarp0 = kProducers;
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = kEpiWarp0 + kEpiWarps;
constexpr int kGatherWarp0 = kMmaWarp + 1;
constexpr int kGatherWarps = 2;
constexpr int kSchedWarp = kGatherWarp0 + kGatherWarps;
constexpr int kLaunchRegs = 128;
constexpr int kSmallRegs = 72;
constexpr int kMmaRegs = 104;
constexpr int kEpiRegs = 168;
static_assert(128 * kSmallRegs + 128 * kMmaRegs + 2 * 128 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kWgtRows = 256;                 // two M=128 operands per stage
constexpr int kWgtBytes = kWgtRows * kBK;     // unpacked e2m1 in shared memory
constexpr int kWgtTxBytes = kWgtBytes / 2;    // a 16U4_ALIGN16B load counts the packed global bytes
constexpr int kTmemCols = 512;
constexpr int kNumBoxes = 8;
__constant__ int kBoxRows[kNumBoxes] = {16, 32, 48, 64, 80, 96, 128, 160};

enum : int {
  kSiteEmpty = 121, kSiteFull = 122, kSiteTmemEmpty = 123, kSiteTmemFull = 124, kSiteGathered = 125,
  kSiteL1Done = 126, kSiteQueueFull = 127, kSiteQueueEmpty = 128, kSiteDrainCopies = 131, kSiteDrainMma = 132
};

// Compile-time shape of one instantiation (BT = tokens per pool block).
template <int BT>
struct Cfg {
  static constexpr int kStages = 4;
  static constexpr int kAccBufs = BT <= 96 ? 2 : 1;             // accumulator pairs in TMEM
  static constexpr int kAccStride = (BT + 31) / 32 * 32;        // columns of one accumulator
  static constexpr int kCPB = (BT + 127) / 128;                 // 128-row scale chunks per block
  static constexpr int kTokBytes = BT * kBK;
  static constexpr int kSfCol0 = 2 * kAccBufs * kAccStride;
  static constexpr int kSfColsPerStage = 8 + 4 * kCPB;         // A0, A1 (4 each), B (4 per chunk)
  static constexpr int kQueueConsumers = kStages + 1 + kEpiWarps;
  // shared memory: token tiles, weight tiles, weight scales, token scales, meta, barriers
  static constexpr int tok = 0;
  static constexpr int wgt = tok + kStages * kTokBytes;
  static constexpr int sfw = wgt + kStages * kWgtBytes;
  static constexpr int sft = sfw + kStages * 2 * kSFChunk;
  static constexpr int meta = sft + kStages * kCPB * kSFChunk;    // blk_off[E+1], cnt[E], queue[kQueue]
  static constexpr int bars_after_meta(int E) { return meta + (((2 * E + 1) + kQueue) * 4 + 15) / 16 * 16; }
  // full[S], empty[S], tfull[B], tempty[B], qfull[Q], qempty[Q], drain
  static constexpr int nbars = 2 * kStages + 2 * kAccBufs + 2 * kQueue + 1;
  static constexpr int total(int E) { return bars_after_meta(E) + nbars * 8 + 16; }
  static_assert(kTokBytes % 1024 == 0, "token tiles keep the 1024-byte swizzle alignment");
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
};
static_assert(Cfg<160>::total(kMaxE) + 1024 <= 232448, "shared memory budget");
static_assert(Cfg<80>::total(kMaxE) + 1024 <= 232448, "shared memory budget");

struct Args {
  int T, H, I, E, K;
  int BT, CPB;
  int KB1, KB2, NB1, NB2;
  int mode, lag, l1_extra;
  const int* cnt;
  const int* blk_off;
  const int* src;
  const float* topk_w;
  const uint8_t* x;
  const uint8_t* x_sf;
  int x_bf16;
  uint8_t* pool_x;           // [P, H]
  uint8_t* pool_x_sf;        // [blocks][H/128][CPB][512]
  const uint8_t* sfw1;       // prepared weight scale chunks (two per 256-row tile and k-block)
  const uint8_t* sfw2;
  uint8_t* pool2;            // intermediate codes [P, I]
  uint8_t* pool2_sf;         // [blocks][I/128][CPB][512]
  float* partials;           // [K, T, H] fp32, or bf16 when pbf16
  int pbf16;
  float clamp;
  int precise;
  float* dbg;                // raw L1 accumulators [P, 2I] or null
  int* ctr_gather;
  int* ctr_l1;
  int* sched;
  int early_combine;
  const int32_t* topk_idx;
  __nv_bfloat16* out;
  int* cmb;
  int* ctr_l2;
  int* deferred;
  int* status;
  uint64_t timeout_ns;
  unsigned long long* prof;  // per-CTA role timings (kProf instantiation) or null
};

struct Maps {
  CUtensorMap w1, w2;
  CUtensorMap x[kNumBoxes], a[kNumBoxes];   // pool / intermediate rows, boxes of kBoxRows rows
};

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A = e2m1 (5) in
// [9:7], B = e4m3 (0) in [12:10], both K-major, N>>3 in [22:17], UE8M0 scales
// (bit 23), M>>4 in [28:24]; the scale-factor byte selectors of B and A in
// [5:4] and [30:29] (the same K sub-block for both).
__device__ __forceinline__ uint32_t idesc_base(int n) {
  return (5u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_k(uint32_t base, int kk) {
  return base | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
}

__device__ __forceinline__ int box_index(int n16) {   // smallest box of >= n16 rows
  int i = 0;
#pragma unroll
  for (int j = 0; j < kNumBoxes - 1; ++j) i += kBoxRows[j] < n16 ? 1 : 0;
  return i;
}

// 32 lanes x 16 columns of 32-bit: thread i gets columns [c, c+16) of lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Max over the 32 lanes of the warp for each of 16 columns, reduce-scatter
// style: after 4 halving exchanges (16 lanes apart, then 8, 4, 2) lane l holds
// the max over 16 lanes of column l >> 1, and one more exchange with lane l ^ 1
// completes it.  16 shuffles for 16 columns.  Returns the max of column l >> 1.
__device__ __forceinline__ float warp_colmax16(float (&v)[16], int lane) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int half = 8 >> r;            // values kept after this round
    const int mask = 16 >> r;           // lane distance of the exchange
    const bool up = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, mask));
    }
  }
  return fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSmallRegs)); }
__device__ __forceinline__ void regs_dec_mma() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kMmaRegs)); }
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs)); }

// kProf: per-CTA role timings into prof[blockIdx.x * 8 + i]: 0 producers' ns
// waiting for a free stage (summed), 1 / 2 the MMA issuer's SM cycles waiting
// for a stage's data / for a free accumulator, 3 its span in ns, 4 its tasks, 5 /
// 6 epilogue warp 4's ns waiting for an accumulator / working, 7 the issuer's span
// in SM cycles.  A separate instantiation: the timing branches cost issue slots.
template <int BT, bool kProf>
__global__ void __launch_bounds__(kThreads, 1) gemm_mx_sw_kernel(const __grid_constant__ Maps maps, const Args args) {
  using C = Cfg<BT>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int E = args.E;
  int* s_blk = reinterpret_cast<int*>(smem + C::meta);
  int* s_cnt = s_blk + E + 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bars_after_meta(E));
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + C::kAccBufs;
  const Queue q{tempty + C::kAccBufs, tempty + C::kAccBufs + kQueue, s_cnt + E};
  uint64_t* drain = tempty + C::kAccBufs + 2 * kQueue;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::nbars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Status st{args.status, args.timeout_ns};
  const int lag = args.mode == 3 ? args.lag : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&q.full[i], 1);
      mbar_init(&q.empty[i], C::kQueueConsumers);
    }
    mbar_init(drain, 1);
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
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += kThreads) s_blk[i] = args.blk_off[i];
  for (int i = threadIdx.x; i < E; i += kThreads) s_cnt[i] = args.cnt[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int nblk = s_blk[E];
  Sched sch{s_blk, s_cnt, E, args.NB1, args.NB2, args.mode, lag};
  sch.BT = BT;

  const int wg = warp >> 2;
  if (wg == 0) {
    regs_dec();
    // ------------------------------------------------------------------ TMA producers
    if (warp + kProducers * lane < S) {
      const int p = warp + kProducers * lane;
      const uint64_t pol_w = policy_evict_first();    // a tile group's last pass over its weights
      const uint64_t pol_wk = policy_evict_normal();  // earlier passes: the next block reads them again
      const uint64_t pol_t = policy_evict_last();
      uint8_t* tk = smem + C::tok + p * C::kTokBytes;
      uint8_t* wt = smem + C::wgt + p * kWgtBytes;
      uint8_t* sw = smem + C::sfw + p * 2 * kSFChunk;
      uint8_t* stk = smem + C::sft + p * C::kCPB * kSFChunk;
      int step = 0;
      bool armed = false;
      uint32_t armed_parity = 0;
      uint64_t w_empty = 0;
      for (Cursor c; !*s_abort && sch.next(c, q, st, s_abort, false, lane, kSiteQueueFull);) {
        const Task& t = c.t;
        const bool l1 = t.type == 1;
        const int KB = l1 ? args.KB1 : args.KB2;
        int kb = ((p - step) % S + S) % S;   // first k-block of this task on stage p
        if (kb < KB && args.mode == 3) {
          const bool ok = l1 ? wait_counter_geq(args.ctr_gather + t.b, t.valid, st, s_abort, kSiteGathered)
                             : wait_counter_geq(args.ctr_l1 + t.b, args.NB1 * kEpiWarps + args.l1_extra, st,
                                                s_abort, kSiteL1Done);
          if (!ok) break;
          fence_proxy_async_global();
        }
        const int n16 = (t.valid + 15) & ~15;
        const int bi = box_index(n16);
        const CUtensorMap* tt = l1 ? &maps.x[bi] : &maps.a[bi];
        const int chunks = n16 > 128 ? 2 : 1;
        const uint32_t bytes = kBoxRows[bi] * kBK + kWgtTxBytes + 2 * kSFChunk + chunks * kSFChunk;
        const uint8_t* sfw = (l1 ? args.sfw1 : args.sfw2) +
                             (static_cast<size_t>(t.e) * (l1 ? args.NB1 : args.NB2) + t.n) * KB * 2 * kSFChunk;
        const uint8_t* sft = (l1 ? args.pool_x_sf : args.pool2_sf) + static_cast<size_t>(t.b) * KB * C::kCPB * kSFChunk;
        for (; kb < KB; kb += S) {
          const uint32_t phase = ((step + kb) / S) & 1;
          const uint64_t t0 = kProf ? globaltimer() : 0;
          if (!mbar_wait(&empty[p], phase ^ 1, st, s_abort, kSiteEmpty)) break;
          if (kProf) w_empty += globaltimer() - t0;
          mbar_arrive_expect_tx(&full[p], bytes);
          armed = true;
          armed_parity = phase;
          const int kbe = t.rev ? KB - 1 - kb : kb;   // the k-block this stage carries
          const int kc = kbe * kBK;
          tma_load_2d(tk, tt, &full[p], kc, t.b * BT, pol_t);
          bulk_load(stk, sft + static_cast<size_t>(kbe) * C::kCPB * kSFChunk, chunks * kSFChunk, &full[p]);
          const uint64_t pw = t.last ? pol_w : pol_wk;
          if (l1) tma_load_3d(wt, &maps.w1, &full[p], kc, t.e * 2 * args.I + t.n * 128, 0, pw);
          else tma_load_2d(wt, &maps.w2, &full[p], kc, t.e * args.H + t.n * kWgtRows, pw);
          bulk_load(sw, sfw + static_cast<size_t>(kbe) * 2 * kSFChunk, 2 * kSFChunk, &full[p]);
        }
        step += KB;
      }
      if (armed) mbar_wait_drain(&full[p], armed_parity, st, kSiteDrainCopies);
      if (kProf) atomicAdd(&args.prof[blockIdx.x * 8 + 0], static_cast<unsigned long long>(w_empty));
    }
  } else if (wg == 3) {
    regs_dec_mma();
    if (warp == kMmaWarp) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint64_t dtok = make_smem_desc(smem_u32(smem + C::tok), 16, 1024, 2);
        const uint64_t dwgt = make_smem_desc(smem_u32(smem + C::wgt), 16, 1024, 2);
        const uint64_t dsfw = make_smem_desc(smem_u32(smem + C::sfw), 0, 128, 0);
        const uint64_t dsft = make_smem_desc(smem_u32(smem + C::sft), 0, 128, 0);
        uint32_t phase = 0;
        int it = 0, kb = 0, KB = 0;
        uint32_t idb = 0, acc0 = 0;
        bool two = false;   // the token scales span two chunks (N > 128)
        Cursor cur;
        uint64_t w_full = 0, w_tempty = 0;
        const uint64_t t_start = kProf ? globaltimer() : 0;
        const long long c_start = kProf ? clock64() : 0;
        auto start_task = [&]() -> bool {
          if (*s_abort || !sch.next(cur, q, st, s_abort, false, lane, kSiteQueueFull)) return false;
          KB = cur.t.type == 1 ? args.KB1 : args.KB2;
          const int n16 = (cur.t.valid + 15) & ~15;
          idb = idesc_base(n16);
          two = n16 > 128;
          const int buf = it % C::kAccBufs;
          acc0 = tmem + buf * 2 * C::kAccStride;
          const long long t0 = kProf ? clock64() : 0;
          if (!mbar_wait(&tempty[buf], ((it / C::kAccBufs) & 1) ^ 1, st, s_abort, kSiteTmemEmpty)) return false;
          if (kProf) w_tempty += clock64() - t0;
          tc_fence_after();
          return true;
        };
        bool live = start_task();
        while (live) {
#pragma unroll
          for (int s = 0; s < S; ++s) {
            if (live) {
              const long long t1 = kProf ? clock64() : 0;
              if (!mbar_wait(&full[s], phase, st, s_abort, kSiteFull)) {
                live = false;
              } else {
                if (kProf) w_full += clock64() - t1;
                tc_fence_after();
                const uint32_t sf = tmem + C::kSfCol0 + s * C::kSfColsPerStage;
                tc_cp_32x128b_warpx4(sf, dsfw + ((s * 2 * kSFChunk) >> 4));
                tc_cp_32x128b_warpx4(sf + 4, dsfw + (((s * 2 + 1) * kSFChunk) >> 4));
                tc_cp_32x128b_warpx4(sf + 8, dsft + ((s * C::kCPB * kSFChunk) >> 4));
                if (C::kCPB > 1 && two) tc_cp_32x128b_warpx4(sf + 12, dsft + (((s * C::kCPB + 1) * kSFChunk) >> 4));
                const uint64_t da0 = dwgt + ((s * kWgtBytes) >> 4);
                const uint64_t da1 = da0 + ((kWgtBytes / 2) >> 4);
                const uint64_t db = dtok + ((s * C::kTokBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {   // K advances 32 bytes = 2 descriptor units
                  const uint32_t id = idesc_k(idb, kk);
                  tc_mma_mxf8f6f4(acc0, da0 + 2 * kk, db + 2 * kk, id, sf, sf + 8, (kb | kk) != 0);
                  tc_mma_mxf8f6f4(acc0 + C::kAccStride, da1 + 2 * kk, db + 2 * kk, id, sf + 4, sf + 8,
                                  (kb | kk) != 0);
                }
                tc_commit(&empty[s]);
                if (++kb == KB) {
                  tc_commit(&tfull[it % C::kAccBufs]);
                  kb = 0;
                  ++it;
                  live = start_task();
                }
              }
            }
          }
          phase ^= 1;
        }
        tc_commit(drain);
        mbar_wait_drain(drain, 0, st, kSiteDrainMma);
        if (kProf) {
          args.prof[blockIdx.x * 8 + 1] = w_full;
          args.prof[blockIdx.x * 8 + 2] = w_tempty;
          args.prof[blockIdx.x * 8 + 3] = globaltimer() - t_start;
          args.prof[blockIdx.x * 8 + 4] = it;
          args.prof[blockIdx.x * 8 + 7] = clock64() - c_start;
        }
      }
      __syncwarp();
    } else if (warp < kGatherWarp0 + kGatherWarps && args.mode == 3) {
      gather_rows(args, s_blk, s_cnt, sch, s_abort, warp - kGatherWarp0, kGatherWarps, lane, nblk);
    } else if (warp == kSchedWarp && lane == 0) {
      run_scheduler(sch, q, args.sched, st, s_abort, kSiteQueueEmpty);
    }
  } else {
    regs_inc();
    // ------------------------------------------------------------------ epilogue (8 warps)
    const int quad = warp & 3;                   // TMEM lane quadrant: weight rows 32 quad + lane
    const int half = (warp - kEpiWarp0) >> 2;    // this warp takes 16-token chunks half, half + 2, ...
    const uint32_t qoff = static_cast<uint32_t>(quad * 32) << 16;
    int it = 0;
    uint64_t w_tfull = 0, busy = 0, t_mark = 0;
    for (Cursor c; sch.next(c, q, st, s_abort, true, lane, kSiteQueueFull); ++it) {
      const Task& t = c.t;
      const int buf = it % C::kAccBufs;
      const uint32_t a0 = tmem + qoff + buf * 2 * C::kAccStride;
      const uint32_t a1 = a0 + C::kAccStride;
      const int nch = (t.valid + 15) >> 4;
      const uint64_t t0 = kProf ? globaltimer() : 0;
      if (kProf && it > 0) busy += t0 - t_mark;
      if (!mbar_wait(&tfull[buf], (it / C::kAccBufs) & 1, st, s_abort, kSiteTmemFull)) break;
      if (kProf) {
        t_mark = globaltimer();
        w_tfull += t_mark - t0;
      }
      tc_fence_after();
      const size_t row0 = static_cast<size_t>(t.b) * BT;
      if (t.type == 1) {
        const int j = t.n * 128 + quad * 32 + lane;   // intermediate column of this lane
        for (int ch = half; ch < nch; ch += 2) {
          uint32_t g[16], u[16];
          tmem_ld_32x32b_x16(a0 + ch * 16, g);
          tmem_ld_32x32b_x16(a1 + ch * 16, u);
          // lane i < 16 fetches token 16 ch + i's router weight while the loads land
          const int ti = ch * 16 + (lane & 15);
          const bool lv = ti < t.valid;
          const float wl = lv ? __ldg(args.topk_w + __ldg(args.src + row0 + ti)) : 0.f;
          tmem_ld_wait();
          float a[16], v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float gi = __uint_as_float(g[i]), ui = __uint_as_float(u[i]);
            if (args.dbg && ch * 16 + i < t.valid) {
              float* drow = args.dbg + (row0 + ch * 16 + i) * 2 * args.I;
              drow[j] = gi;
              drow[args.I + j] = ui;
            }
            if (args.clamp < INFINITY) {
              gi = fminf(fmaxf(gi, -args.clamp), args.clamp);
              ui = fminf(fmaxf(ui, -args.clamp), args.clamp);
            }
            const float wi = __shfl_sync(0xffffffffu, wl, i);
            a[i] = (args.precise ? silu_precise(gi) : silu_fast(gi)) * ui * wi;
            v[i] = fabsf(a[i]);
          }
          // per-token amax over this warp's 32 columns j (one requant block)
          const float am = warp_colmax16(v, lane);
          const int ee = ue8m0_exponent_e4m3(am);      // lane l: token l >> 1
          const float sc = exp2_neg(ee);
          const int tl = ch * 16 + (lane >> 1);
          if ((lane & 1) == 0 && tl < t.valid)
            args.pool2_sf[pool_sf_word(t.b, t.n, args.KB2, args.CPB, tl) + quad] = static_cast<uint8_t>(ee + 127);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float si = __shfl_sync(0xffffffffu, sc, 2 * i);
            const uint16_t code = cvt_e4m3x2(a[i] * si, 0.f);
            if (ch * 16 + i < t.valid) args.pool2[(row0 + ch * 16 + i) * args.I + j] = static_cast<uint8_t>(code & 0xff);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (args.mode == 3) {
          fence_proxy_async_global();              // the codes are read by TMA later
          __syncwarp();
          if (lane == 0) red_release_gpu_add(args.ctr_l1 + t.b, 1);
        }
      } else {
        const int h = t.n * kWgtRows + quad * 32 + lane;   // output column of acc0; acc1 is h + 128
        const bool h1 = h + 128 < args.H;
        for (int ch = half; ch < nch; ch += 2) {
          uint32_t y0[16], y1[16];
          tmem_ld_32x32b_x16(a0 + ch * 16, y0);
          tmem_ld_32x32b_x16(a1 + ch * 16, y1);
          // lane i < 16 resolves token 16 ch + i's partial row (k * T + t) * H
          const int ti = ch * 16 + (lane & 15);
          long long off = -1;
          if (ti < t.valid) {
            const int s = __ldg(args.src + row0 + ti);
            const int tt = s / args.K;
            off = (static_cast<long long>(s - tt * args.K) * args.T + tt) * args.H;
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const long long oi = __shfl_sync(0xffffffffu, off, i);
            if (oi < 0) continue;
            if (args.pbf16) {
              __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.partials) + oi + h;
              dst[0] = __float2bfloat16_rn(__uint_as_float(y0[i]));
              if (h1) dst[128] = __float2bfloat16_rn(__uint_as_float(y1[i]));
            } else {
              float* dst = args.partials + oi + h;
              dst[0] = __uint_as_float(y0[i]);
              if (h1) dst[128] = __uint_as_float(y1[i]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (args.early_combine) {
          __syncwarp();   // the warp's partial stores before its release
          if (lane == 0) red_release_gpu_add(args.ctr_l2 + t.e, 1);
        }
      }
    }
    if (kProf && it > 0) busy += globaltimer() - t_mark;
    if (kProf && warp == kEpiWarp0 && lane == 0) {
      args.prof[blockIdx.x * 8 + 5] = w_tfull;
      args.prof[blockIdx.x * 8 + 6] = busy;
    }
    if (args.early_combine) {
      if (args.pbf16) early_combine<__nv_bfloat16>(args, kEpiWarps, args.NB2, s_blk, st, s_abort, lane);
      else early_combine<float>(args, kEpiWarps, args.NB2, s_blk, st, s_abort, lane);
    }
  }

  // every role has waited for the async work it issued, so after this barrier
  // no copy or MMA still targets this CTA's shared or tensor memory
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BT>
cudaError_t launch_impl(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s) {
  using C = Cfg<BT>;
  const Layout& L = *g.L;
  const WsPtrs& W = *g.W;
  Maps maps;
  Args a{};
  a.T = L.T; a.H = L.H; a.I = L.I; a.E = L.E; a.K = L.K;
  a.BT = BT; a.CPB = C::kCPB;
  a.KB1 = L.H / 128; a.KB2 = L.I / 128; a.NB1 = L.I / 128; a.NB2 = (L.H + kWgtRows - 1) / kWgtRows;
  a.mode = mode;
  a.lag = lag < 0 ? 0 : (lag > L.E ? L.E : lag);
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
  a.status = W.status; a.timeout_ns = g.timeout_ns;
  a.prof = g.prof ? g.prof + (mode == 2 ? 8 * 1024 : 0) : nullptr;
  {
    // W1 as (k, row, half): one box of {128 k, 128 rows, 2 halves} is 128 gate
    // rows followed by the matching 128 up rows (A0, then A1)
    const uint64_t dims[3] = {static_cast<uint64_t>(L.H), static_cast<uint64_t>(L.E) * 2 * L.I - L.I, 2};
    const uint64_t strides[2] = {static_cast<uint64_t>(L.H) / 2, static_cast<uint64_t>(L.I) * L.H / 2};
    const uint32_t box[3] = {128, 128, 2};
    if (encode_tmap(&maps.w1, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, g.w1, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (encode_tmap_2d(&maps.w2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w2, L.I, static_cast<uint64_t>(L.E) * L.H,
                     L.I / 2, 128, kWgtRows, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  static const int rows[kNumBoxes] = {16, 32, 48, 64, 80, 96, 128, 160};
  for (int i = 0; i < kNumBoxes; ++i) {
    const uint32_t r = static_cast<uint32_t>(rows[i] <= BT ? rows[i] : BT);   // boxes past BT are never picked
    if (encode_tmap_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool_x, L.H, L.P, L.H, 128, r,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode_tmap_2d(&maps.a[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool2, L.I, L.P, L.I, 128, r,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kernel = a.prof ? gemm_mx_sw_kernel<BT, true> : gemm_mx_sw_kernel<BT, false>;
  if (cudaError_t e = configure_kernel(reinterpret_cast<const void*>(kernel), kLaunchRegs, C::total(kMaxE) + 1024))
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::total(L.E) + 1024;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (mode == 3) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (g.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, maps, a);
}

}  // namespace

bool mx_sw_block_supported(int bt) { return bt == 80 || bt == 160; }

cudaError_t launch_gemm_mx_sw(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s) {
  switch (g.L->BT) {
    case 80: return launch_impl<80>(g, mode, lag, l1_extra, s);
    case 160: return launch_impl<160>(g, mode, lag, l1_extra, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mm

// Block-scaled grouped GEMMs of the MoE layer on CTA pairs (tcgen05
// cta_group::2): the weights are the MMA's M operand, 256 rows per MMA split
// over the two CTAs of a cluster, and each pool block's tokens are its N
// operand (N = the block's token count rounded up to 16, half of the rows in
// each CTA).  This is the pages' SM100 form: a 2x1-SM block-scaled MMA issued
// by one thread of the leader CTA, with the token dimension sized to the
// block's valid rows (llm-infra-atlas "07 · MegaMoE" §2 and §5).
//
// Why pairs: on GB300 a tcgen05 instruction costs its issuing thread about as
// long as an M=128 MMA of N = 128 takes the tensor pipe (measured: 51 cycles
// for N <= 80, N/2 above), and an M=256 cta_group::2 MMA costs the same issue
// time while both SMs' tensor pipes work.  With single-CTA MMAs the swapped
// operand order needs twice the instructions per weight byte of the token-M
// form and the issuing thread becomes the limit; a pair halves that per SM,
// and halves each CTA's share of the token tile, so 5 pipeline stages fit.
//
// Task = (expert e, pair tile n, pool block b).  CTA r of the pair owns the
// weight rows of single-CTA tile 2n + r:
//   L1: gate rows [256n + 128r, +128) and the matching up rows (A0, A1), so its
//       TMEM lane j holds gate and up of intermediate column 256n + 128r + j;
//   L2: W2 rows [512n + 256r, +128) and [512n + 256r + 128, +128).
// A half-tile past I (L1) or H (L2) is a ghost: its CTA loads the last real
// tile again and its epilogue stores nothing.  CTA r holds token rows
// [r N/2, (r+1) N/2) of the block; both CTAs hold the block's token scales.
//
// Every copy of both CTAs completes on the leader's stage barrier
// (cp.async.bulk.tensor ... .cta_group::2); the leader's MMA commits release
// both CTAs' stages and accumulators.  Warp roles per CTA as in the single-CTA
// kernels (gemm_mx_sw.cu); the peer's MMA warp only allocates TMEM, and the
// tile-group scheduler runs in the leader and fills both CTAs' queues.
// Every wait is bounded.  Before TMEM is freed the leader waits for every
// phase either CTA armed or loaded (the peer records its loads in the
// leader's shared memory) and for its last MMA commit, behind two cluster
// barriers.
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
constexpr int kEpiWarps = 8;                  // per CTA; a pair task has 16
constexpr int kMmaWarp = kEpiWarp0 + kEpiWarps;
constexpr int kGatherWarp0 = kMmaWarp + 1;
constexpr int kGatherWarps = 2;
constexpr int kSchedWarp = kGatherWarp0 + kGatherWarps;
constexpr int kLaunchRegs = 128;
constexpr int kSmallRegs = 72;
constexpr int kMmaRegs = 104;
constexpr int kEpiRegs = 168;
static_assert(128 * kSmallRegs + 128 * kMmaRegs + 2 * 128 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kWgtRows = 256;                 // weight rows per CTA and stage (two M=128 halves of two pair MMAs)
constexpr int kWgtBytes = kWgtRows * kBK;
constexpr int kWgtTxBytes = kWgtBytes / 2;    // packed e2m1 bytes a 16U4_ALIGN16B load counts
constexpr int kTmemCols = 512;
constexpr int kNumBoxes = 8;                  // token boxes of N/2 rows
__constant__ int kBoxRows[kNumBoxes] = {8, 16, 24, 32, 40, 48, 64, 80};

enum : int {
  kSiteEmpty = 141, kSiteFull = 142, kSiteTmemEmpty = 143, kSiteTmemFull = 144, kSiteGathered = 145,
  kSiteL1Done = 146, kSiteQueueFull = 147, kSiteQueueEmpty = 148, kSiteDrainCopies = 151, kSiteDrainMma = 152
};

template <int BT>
struct Cfg {
  static constexpr int kStages = 5;
  static constexpr int kHalfRows = BT / 2;                       // token rows per CTA at most
  static constexpr int kAccStride = (BT + 31) / 32 * 32;
  static constexpr int kCPB = (BT + 127) / 128;
  static constexpr int kSfColsPerStage = 8 + 4 * kCPB;
  static constexpr int kAccBufs = 4 * kAccStride + kStages * kSfColsPerStage <= kTmemCols ? 2 : 1;
  static constexpr int kSfCol0 = 2 * kAccBufs * kAccStride;
  static constexpr int kTokBytes = kHalfRows * kBK;
  static constexpr int kSftBytes = kCPB * kSFChunk;
  static constexpr int kQueueConsumers = kStages + kEpiWarps;   // per CTA, plus the leader's MMA thread
  static constexpr int tok = 0;
  static constexpr int wgt = tok + kStages * kTokBytes;
  static constexpr int sfw = wgt + kStages * kWgtBytes;
  static constexpr int sft = sfw + kStages * 2 * kSFChunk;
  // queue[kQueue]; per stage: phases the leader armed, phases the peer loaded, the peer's bytes
  static constexpr int meta = sft + kStages * kSftBytes;
  static constexpr int bars = meta + ((kQueue + 3 * kStages) * 4 + 15) / 16 * 16;
  // full[S], empty[S], tfull[B], tempty[B], qfull[Q], qempty[Q], drain
  static constexpr int nbars = 2 * kStages + 2 * kAccBufs + 2 * kQueue + 1;
  static constexpr int total = bars + nbars * 8 + 16;
  static_assert(kTokBytes % 1024 == 0, "token tiles keep the 1024-byte swizzle alignment");
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
};
static_assert(Cfg<160>::total + 1024 <= 232448, "shared memory budget");
static_assert(Cfg<80>::total + 1024 <= 232448, "shared memory budget");

struct Args {
  int T, H, I, E, K;
  int BT, CPB;
  int KB1, KB2, NB1, NB2;     // single-CTA tile counts (128 intermediate columns, 256 rows of H)
  int PB1, PB2;               // pair tiles: ceil(NB1 / 2), ceil(NB2 / 2)
  int mode, lag, l1_extra;
  const int* cnt;
  const int* blk_off;
  const int* src;
  const float* topk_w;
  const uint8_t* x;
  const uint8_t* x_sf;
  int x_bf16;
  uint8_t* pool_x;
  uint8_t* pool_x_sf;
  uint8_t* pool2;
  uint8_t* pool2_sf;
  float* partials;
  int pbf16;
  float clamp;
  int precise;
  float* dbg;
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
  unsigned long long* prof;
};

struct Maps {
  CUtensorMap w1, w2;                         // weights (as in the single-CTA kernels)
  CUtensorMap sw1, sw2;                       // prepared weight scales viewed as [*, 256 B], boxes of 4 rows (1 KB)
  CUtensorMap sx, sa;                         // pool / intermediate scales, boxes of one block's chunks
  CUtensorMap x[kNumBoxes], a[kNumBoxes];     // pool / intermediate rows, boxes of kBoxRows rows
};

// ------------------------------------------------------------------ cluster / pair helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// both CTAs, every thread: prior work of each CTA (shared memory, remote arrivals) is visible to the other
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster(uint32_t caddr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(caddr), "r"(v) : "memory");
}
__device__ __forceinline__ void arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// TMA tile loads into this CTA's shared memory completing on a barrier of either CTA of the pair
__device__ __forceinline__ void tma2d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int c0, int c1,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma3d_pair(void* dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int c2,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}
// Bounded wait with cluster-scope acquire, for barriers the other CTA of the pair
// arrives on (its writes before the arrival are visible afterwards).
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, const Status& st, volatile int* abort,
                                      int where) {
  const uint32_t a = smem_u32(bar);
  if (try_wait_cluster(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (try_wait_cluster(a, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > st.timeout_ns) {
      report_error(st, 4 /*MM_MOE_ERR_TIMEOUT*/, where);
      *abort = 1;
      return false;
    }
  }
}

// tcgen05 on the pair: TMEM allocation (a warp of each CTA), copies and MMAs (one leader thread), commits
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst, uint32_t n) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(n)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t t, uint32_t n) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(t), "r"(n) : "memory");
}
// each CTA's 512-byte chunk at the descriptor's offset goes to the same TMEM columns of that CTA
__device__ __forceinline__ void tc_cp2(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma2(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
          "r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit2(uint32_t bar_cluster) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_cluster)
               : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling, M = 256: A = e2m1 (5)
// in [9:7], B = e4m3 (0) in [12:10], both K-major, N>>3 in [22:17], UE8M0 scales
// (bit 23), M>>4 in [28:24]; scale-factor byte selectors in [30:29] and [5:4].
__device__ __forceinline__ uint32_t idesc_base(int n) {
  return (5u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | ((256u >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_k(uint32_t base, int kk) {
  return base | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
}
__device__ __forceinline__ int box_index(int rows) {   // smallest box of >= rows rows
  int i = 0;
#pragma unroll
  for (int j = 0; j < kNumBoxes - 1; ++j) i += kBoxRows[j] < rows ? 1 : 0;
  return i;
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Max over the warp's 32 lanes of each of 16 columns, reduce-scatter style (see gemm_mx_sw.cu);
// returns the max of column lane >> 1.
__device__ __forceinline__ float warp_colmax16(float (&v)[16], int lane) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int half = 8 >> r;
    const int mask = 16 >> r;
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

// The pair's queue reader: both CTAs wait on their own slot; every consumer releases the
// slot on the leader's barrier.
__device__ __forceinline__ bool pair_next(const Sched& sch, Cursor& c, const Queue& q, uint32_t rank,
                                          const Status& st, volatile int* abort, bool warp_wide, int lane) {
  if (c.bl + 1 < c.nb) {
    ++c.bl;
    sch.block(c);
    return true;
  }
  const int slot = c.i % kQueue;
  const uint32_t parity = (c.i / kQueue) & 1;
  ++c.i;
  int g = -1;
  if (!warp_wide || lane == 0) {
    if (pwait(&q.full[slot], parity, st, abort, kSiteQueueFull)) {
      g = q.g[slot];
      if (rank == 0) mbar_arrive(&q.empty[slot]);
      else arrive_cluster(cl_map(&q.empty[slot], 0));
    }
  }
  if (warp_wide) g = __shfl_sync(0xffffffffu, g, 0);
  c.nb = 0;
  if (g < 0) return false;
  int bl;
  sch.group(g, c.t, &bl);
  c.nb = sch.blk[c.t.e + 1] - sch.blk[c.t.e];
  c.bl = 0;
  sch.block(c);
  return true;
}

// The leader's scheduler thread: tile groups from the device-wide counter into both CTAs' queues.
__device__ __forceinline__ void pair_scheduler(const Sched& sch, const Queue& q, int* counter, const Status& st,
                                               volatile int* abort) {
  const int ng = sch.groups();
  for (int i = 0;; ++i) {
    const int slot = i % kQueue;
    if (!pwait(&q.empty[slot], ((i / kQueue) & 1) ^ 1, st, abort, kSiteQueueEmpty)) break;
    int g = -1;
    for (;;) {
      const int x = atomicAdd(counter, 1);
      if (x >= ng) break;
      if (sch.group_blocks(x) > 0) {
        g = x;
        break;
      }
    }
    q.g[slot] = g;
    st_cluster(cl_map(const_cast<int*>(&q.g[slot]), 1), g);
    arrive_cluster(cl_map(&q.full[slot], 1));   // release: the peer's copy of the slot first
    mbar_arrive(&q.full[slot]);
    if (g < 0) break;
  }
}

template <int BT, bool kProf>
__global__ void __launch_bounds__(kThreads, 1) gemm_mx_pair_kernel(const __grid_constant__ Maps maps, const Args args) {
  using C = Cfg<BT>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int E = args.E;
  int* s_q = reinterpret_cast<int*>(smem + C::meta);
  int* s_armed = s_q + kQueue;                 // leader: phases it armed per stage
  int* s_peer = s_armed + S;                   // leader: phases the peer loaded per stage
  int* s_peer_bytes = s_peer + S;              // leader: the peer's bytes in its last loaded phase
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + C::kAccBufs;
  const Queue q{tempty + C::kAccBufs, tempty + C::kAccBufs + kQueue, s_q};
  uint64_t* drain = tempty + C::kAccBufs + 2 * kQueue;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::nbars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const Status st{args.status, args.timeout_ns};
  const int lag = args.mode == 3 ? args.lag : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      s_armed[i] = 0;
      s_peer[i] = 0;
      s_peer_bytes[i] = 0;
    }
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * kEpiWarps);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&q.full[i], 1);
      mbar_init(&q.empty[i], 2 * C::kQueueConsumers + 1);
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
    tmem_alloc2(s_tmem, kTmemCols);
    tmem_relinquish2();
  }
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  cluster_sync();              // both CTAs' barriers exist before anything targets them
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // the block offsets and counts are read from global memory (they stay in L1)
  Sched sch{args.blk_off, args.cnt, E, args.PB1, args.PB2, args.mode, lag};
  sch.BT = BT;
  const int nblk = __ldg(args.blk_off + E);

  const int wg = warp >> 2;
  if (wg == 0) {
    regs_dec();
    // ------------------------------------------------------------------ TMA producers (both CTAs)
    if (warp + kProducers * lane < S) {
      const int p = warp + kProducers * lane;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_wk = policy_evict_normal();
      const uint64_t pol_t = policy_evict_last();
      uint8_t* tk = smem + C::tok + p * C::kTokBytes;
      uint8_t* wt = smem + C::wgt + p * kWgtBytes;
      uint8_t* sw = smem + C::sfw + p * 2 * kSFChunk;
      uint8_t* stk = smem + C::sft + p * C::kSftBytes;
      const uint32_t fullp = cl_map(&full[p], 0);        // the leader's barrier of this stage
      const uint32_t peer_slot = cl_map(&s_peer[p], 0);
      const uint32_t peer_bytes_slot = cl_map(&s_peer_bytes[p], 0);
      int step = 0;
      bool armed = false;
      uint32_t armed_parity = 0;
      for (Cursor c; !*s_abort && pair_next(sch, c, q, rank, st, s_abort, false, lane);) {
        const Task& t = c.t;
        const bool l1 = t.type == 1;
        const int KB = l1 ? args.KB1 : args.KB2;
        int kb = ((p - step) % S + S) % S;
        if (kb < KB && args.mode == 3) {
          const bool ok = l1 ? wait_counter_geq(args.ctr_gather + t.b, t.valid, st, s_abort, kSiteGathered)
                             : wait_counter_geq(args.ctr_l1 + t.b, args.PB1 * 2 * kEpiWarps + args.l1_extra, st,
                                                s_abort, kSiteL1Done);
          if (!ok) break;
          fence_proxy_async_global();
        }
        const int n16 = (t.valid + 15) & ~15;
        const int half = n16 >> 1;                       // token rows of each CTA
        const int bi = box_index(half);
        const CUtensorMap* tt = l1 ? &maps.x[bi] : &maps.a[bi];
        const CUtensorMap* ts = l1 ? &maps.sx : &maps.sa;
        // this CTA's single-CTA tile; a ghost half (past I or H) reloads the last real tile
        const int nt = l1 ? args.NB1 : args.NB2;
        int ne = 2 * t.n + static_cast<int>(rank);
        ne = ne < nt ? ne : nt - 1;
        const uint32_t pair_bytes = 2 * (kBoxRows[bi] * kBK + kWgtTxBytes + 2 * kSFChunk + C::kSftBytes);
        for (; kb < KB; kb += S) {
          const uint32_t phase = ((step + kb) / S) & 1;
          if (!pwait(&empty[p], phase ^ 1, st, s_abort, kSiteEmpty)) break;
          if (leader) {
            mbar_arrive_expect_tx(&full[p], pair_bytes);
            armed = true;
            armed_parity = phase;
            s_armed[p] = (step + kb) / S + 1;
          } else {
            // recorded before the loads: the leader's exit waits for any phase it never armed
            st_cluster(peer_bytes_slot, static_cast<int>(pair_bytes / 2));
            st_cluster(peer_slot, (step + kb) / S + 1);
          }
          const int kbe = t.rev ? KB - 1 - kb : kb;
          const int kc = kbe * kBK;
          tma2d_pair(tk, tt, fullp, kc, t.b * BT + static_cast<int>(rank) * half, pol_t);
          tma2d_pair(stk, ts, fullp, 0, (t.b * KB + kbe) * 2 * C::kCPB, pol_t);
          const uint64_t pw = t.last ? pol_w : pol_wk;
          if (l1) tma3d_pair(wt, &maps.w1, fullp, kc, t.e * 2 * args.I + ne * 128, 0, pw);
          else tma2d_pair(wt, &maps.w2, fullp, kc, t.e * args.H + ne * kWgtRows, pw);
          tma2d_pair(sw, l1 ? &maps.sw1 : &maps.sw2, fullp, 0, ((t.e * nt + ne) * KB + kbe) * 4, pw);
        }
        step += KB;
      }
      // leader: the copies of the last phase this CTA armed have landed (the peer's too)
      if (leader && armed) mbar_wait_drain(&full[p], armed_parity, st, kSiteDrainCopies);
    }
  } else if (wg == 3) {
    regs_dec_mma();
    if (warp == kMmaWarp) {
      // ------------------------------------------------------------------ MMA issuer (leader)
      if (leader && lane == 0) {
        const uint64_t dtok = make_smem_desc(smem_u32(smem + C::tok), 16, 1024, 2);
        const uint64_t dwgt = make_smem_desc(smem_u32(smem + C::wgt), 16, 1024, 2);
        const uint64_t dsfw = make_smem_desc(smem_u32(smem + C::sfw), 0, 128, 0);
        const uint64_t dsft = make_smem_desc(smem_u32(smem + C::sft), 0, 128, 0);
        uint32_t phase = 0;
        int it = 0, kb = 0, KB = 0;
        uint32_t idb = 0, acc0 = 0;
        bool two = false;
        Cursor cur;
        uint64_t w_full = 0, w_tempty = 0;
        const uint64_t t_start = kProf ? globaltimer() : 0;
        const long long c_start = kProf ? clock64() : 0;
        auto start_task = [&]() -> bool {
          if (*s_abort || !pair_next(sch, cur, q, rank, st, s_abort, false, lane)) return false;
          KB = cur.t.type == 1 ? args.KB1 : args.KB2;
          const int n16 = (cur.t.valid + 15) & ~15;
          idb = idesc_base(n16);
          two = n16 > 128;
          const int buf = it % C::kAccBufs;
          acc0 = tmem + buf * 2 * C::kAccStride;
          const long long t0 = kProf ? clock64() : 0;
          if (!pwait(&tempty[buf], ((it / C::kAccBufs) & 1) ^ 1, st, s_abort, kSiteTmemEmpty)) return false;
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
                tc_cp2(sf, dsfw + ((s * 2 * kSFChunk) >> 4));
                tc_cp2(sf + 4, dsfw + (((s * 2 + 1) * kSFChunk) >> 4));
                tc_cp2(sf + 8, dsft + ((s * C::kSftBytes) >> 4));
                if (C::kCPB > 1 && two) tc_cp2(sf + 12, dsft + ((s * C::kSftBytes + kSFChunk) >> 4));
                const uint64_t da0 = dwgt + ((s * kWgtBytes) >> 4);
                const uint64_t da1 = da0 + ((kWgtBytes / 2) >> 4);
                const uint64_t db = dtok + ((s * C::kTokBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint32_t id = idesc_k(idb, kk);
                  tc_mma2(acc0, da0 + 2 * kk, db + 2 * kk, id, sf, sf + 8, (kb | kk) != 0);
                  tc_mma2(acc0 + C::kAccStride, da1 + 2 * kk, db + 2 * kk, id, sf + 4, sf + 8, (kb | kk) != 0);
                }
                tc_commit2(smem_u32(&empty[s]));
                tc_commit2(cl_map(&empty[s], 1));
                if (++kb == KB) {
                  const int buf = it % C::kAccBufs;
                  tc_commit2(smem_u32(&tfull[buf]));
                  tc_commit2(cl_map(&tfull[buf], 1));
                  kb = 0;
                  ++it;
                  live = start_task();
                }
              }
            }
          }
          phase ^= 1;
        }
        tc_commit2(smem_u32(drain));
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
      gather_rows(args, args.blk_off, args.cnt, sch, s_abort, warp - kGatherWarp0, kGatherWarps, lane, nblk);
    } else if (warp == kSchedWarp && lane == 0 && leader) {
      pair_scheduler(sch, q, args.sched, st, s_abort);
    }
  } else {
    regs_inc();
    // ------------------------------------------------------------------ epilogue (8 warps per CTA)
    const int quad = warp & 3;
    const int half = (warp - kEpiWarp0) >> 2;     // 16-token chunks half, half + 2, ...
    const uint32_t qoff = static_cast<uint32_t>(quad * 32) << 16;
    int it = 0;
    uint64_t w_tfull = 0, busy = 0, t_mark = 0, t_rel = 0;
    uint64_t hold1 = 0, post1 = 0, hold2 = 0, post2 = 0;   // profiling build: per task type
    for (Cursor c; pair_next(sch, c, q, rank, st, s_abort, true, lane); ++it) {
      const Task& t = c.t;
      const bool l1 = t.type == 1;
      const int buf = it % C::kAccBufs;
      const uint32_t a0 = tmem + qoff + buf * 2 * C::kAccStride;
      const uint32_t a1 = a0 + C::kAccStride;
      const int nch = (t.valid + 15) >> 4;
      const int ne = 2 * t.n + static_cast<int>(rank);       // this CTA's single-CTA tile
      const bool ghost = ne >= (l1 ? args.NB1 : args.NB2);
      const size_t row0 = static_cast<size_t>(t.b) * BT;
      // per-token data of this warp's chunks, fetched before the accumulator is ready:
      // chunk i of the warp is column chunk half + 2 i; lane l < 16 holds its token l
      constexpr int kMaxCh = (BT / 16 + 1) / 2;
      float wv[kMaxCh];
      long long ov[kMaxCh];
#pragma unroll
      for (int i = 0; i < kMaxCh; ++i) {
        const int ti = (half + 2 * i) * 16 + (lane & 15);
        wv[i] = 0.f;
        ov[i] = -1;
        if (ti < t.valid && !ghost) {
          const int s = __ldg(args.src + row0 + ti);
          if (l1) {
            wv[i] = __ldg(args.topk_w + s);
          } else {
            const int tt = s / args.K;
            ov[i] = (static_cast<long long>(s - tt * args.K) * args.T + tt) * args.H;
          }
        }
      }
      const uint64_t t0 = kProf ? globaltimer() : 0;
      if (kProf && it > 0) busy += t0 - t_mark;
      if (!pwait(&tfull[buf], (it / C::kAccBufs) & 1, st, s_abort, kSiteTmemFull)) break;
      if (kProf) {
        t_mark = globaltimer();
        w_tfull += t_mark - t0;
      }
      tc_fence_after();
      // software pipeline: the next chunk's TMEM loads are in flight while this one is processed,
      // and the accumulator is handed back as soon as the last load has landed
      uint32_t g[2][16], u[2][16];
      const int mine = nch > half ? (nch - half + 1) / 2 : 0;   // chunks of this warp
      if (mine > 0) {
        tmem_ld_32x32b_x16(a0 + half * 16, g[0]);
        tmem_ld_32x32b_x16(a1 + half * 16, u[0]);
      }
      tmem_ld_wait();
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&tempty[buf]);
          else arrive_cluster(cl_map(&tempty[buf], 0));
        }
        if (kProf) t_rel = globaltimer();
      };
      if (mine <= 1) release();
#pragma unroll
      for (int i = 0; i < kMaxCh; ++i) {
        if (i >= mine) break;
        const int ch = half + 2 * i;
        const int cur = i & 1;
        if (i + 1 < mine) {
          tmem_ld_32x32b_x16(a0 + (ch + 2) * 16, g[cur ^ 1]);
          tmem_ld_32x32b_x16(a1 + (ch + 2) * 16, u[cur ^ 1]);
        }
        if (!ghost) {
          if (l1) {
            const int j = ne * 128 + quad * 32 + lane;
            float a[16], v[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float gk = __uint_as_float(g[cur][k]), uk = __uint_as_float(u[cur][k]);
              if (args.dbg && ch * 16 + k < t.valid) {
                float* drow = args.dbg + (row0 + ch * 16 + k) * 2 * args.I;
                drow[j] = gk;
                drow[args.I + j] = uk;
              }
              if (args.clamp < INFINITY) {
                gk = fminf(fmaxf(gk, -args.clamp), args.clamp);
                uk = fminf(fmaxf(uk, -args.clamp), args.clamp);
              }
              const float wk = __shfl_sync(0xffffffffu, wv[i], k);
              a[k] = (args.precise ? silu_precise(gk) : silu_fast(gk)) * uk * wk;
              v[k] = fabsf(a[k]);
            }
            const float am = warp_colmax16(v, lane);
            const int ee = ue8m0_exponent_e4m3(am);
            const float sc = exp2_neg(ee);
            const int tl = ch * 16 + (lane >> 1);
            if ((lane & 1) == 0 && tl < t.valid)
              args.pool2_sf[pool_sf_word(t.b, ne, args.KB2, args.CPB, tl) + quad] = static_cast<uint8_t>(ee + 127);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float sk = __shfl_sync(0xffffffffu, sc, 2 * k);
              const uint16_t code = cvt_e4m3x2(a[k] * sk, 0.f);
              if (ch * 16 + k < t.valid)
                args.pool2[(row0 + ch * 16 + k) * args.I + j] = static_cast<uint8_t>(code & 0xff);
            }
          } else {
            const int h = ne * kWgtRows + quad * 32 + lane;
            const bool h1 = h + 128 < args.H;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const long long ok = __shfl_sync(0xffffffffu, ov[i], k);
              if (ok < 0) continue;
              if (args.pbf16) {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.partials) + ok + h;
                dst[0] = __float2bfloat16_rn(__uint_as_float(g[cur][k]));
                if (h1) dst[128] = __float2bfloat16_rn(__uint_as_float(u[cur][k]));
              } else {
                float* dst = args.partials + ok + h;
                dst[0] = __uint_as_float(g[cur][k]);
                if (h1) dst[128] = __uint_as_float(u[cur][k]);
              }
            }
          }
        }
        if (i + 1 < mine) {
          tmem_ld_wait();
          if (i + 2 >= mine) release();   // the warp's last loads have landed
        }
      }
      if (kProf) {   // hold = accumulator ready -> released, post = released -> task done
        const uint64_t t_end = globaltimer();
        (l1 ? hold1 : hold2) += t_rel - t_mark;
        (l1 ? post1 : post2) += t_end - t_rel;
      }
      if (l1 && args.mode == 3) {
        fence_proxy_async_global();              // the codes are read by TMA later
        __syncwarp();
        if (lane == 0) red_release_gpu_add(args.ctr_l1 + t.b, 1);
      }
      if (!l1 && args.early_combine) {
        __syncwarp();
        if (lane == 0) red_release_gpu_add(args.ctr_l2 + t.e, 1);
      }
    }
    if (kProf && it > 0) busy += globaltimer() - t_mark;
    if (kProf && warp == kEpiWarp0 && lane == 0) {
      args.prof[blockIdx.x * 8 + 5] = w_tfull;
      args.prof[blockIdx.x * 8 + 6] = busy;
      args.prof[4096 + blockIdx.x] = hold1;
      args.prof[4096 + 1024 + blockIdx.x] = post1;
      args.prof[4096 + 2048 + blockIdx.x] = hold2;
      args.prof[4096 + 3072 + blockIdx.x] = post2;
    }
    if (args.early_combine) {
      if (args.pbf16) early_combine<__nv_bfloat16>(args, 2 * kEpiWarps, args.PB2, args.blk_off, st, s_abort, lane);
      else early_combine<float>(args, 2 * kEpiWarps, args.PB2, args.blk_off, st, s_abort, lane);
    }
  }

  // The leader's producers waited for the last phase each armed (both CTAs' copies).
  // After this barrier the peer has issued its last copy; a phase it loaded that the
  // leader never armed (the leader stopped first, on a timeout) is armed now with the
  // peer's share and waited for, bounded.  After the second barrier no copy or MMA
  // targets either CTA any more.
  __syncthreads();
  cluster_sync();
  if (leader && threadIdx.x < S) {
    const int p = threadIdx.x;
    const int loaded = s_peer[p];
    if (loaded > s_armed[p]) {
      mbar_arrive_expect_tx(&full[p], static_cast<uint32_t>(s_peer_bytes[p]));
      mbar_wait_drain(&full[p], (loaded - 1) & 1, st, kSiteDrainCopies);
    }
  }
  __syncthreads();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc2(tmem, kTmemCols);
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
  a.PB1 = (a.NB1 + 1) / 2; a.PB2 = (a.NB2 + 1) / 2;
  a.mode = mode;
  a.lag = lag < 0 ? 0 : (lag > L.E ? L.E : lag);
  a.l1_extra = l1_extra;
  a.cnt = W.cnt; a.blk_off = W.blk_off; a.src = W.src; a.topk_w = g.topk_w;
  a.x = g.x; a.x_sf = static_cast<const uint8_t*>(g.x_sf); a.x_bf16 = g.x_bf16 ? 1 : 0;
  a.pool_x = W.pool_x; a.pool_x_sf = W.pool_x_sf;
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
  // scale regions viewed as rows of 256 bytes
  const uint64_t sw1_rows = static_cast<uint64_t>(L.E) * a.NB1 * a.KB1 * 4;
  const uint64_t sw2_rows = static_cast<uint64_t>(L.E) * a.NB2 * a.KB2 * 4;
  const uint64_t sx_rows = static_cast<uint64_t>(L.nblk_cap) * a.KB1 * C::kCPB * 2;
  const uint64_t sa_rows = static_cast<uint64_t>(L.nblk_cap) * a.KB2 * C::kCPB * 2;
  if (encode_tmap_2d(&maps.sw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w1sfp, 256, sw1_rows, 256, 256, 4,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
      encode_tmap_2d(&maps.sw2, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w2sfp, 256, sw2_rows, 256, 256, 4,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
      encode_tmap_2d(&maps.sx, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool_x_sf, 256, sx_rows, 256, 256, 2 * C::kCPB,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
      encode_tmap_2d(&maps.sa, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool2_sf, 256, sa_rows, 256, 256, 2 * C::kCPB,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  static const int rows[kNumBoxes] = {8, 16, 24, 32, 40, 48, 64, 80};
  for (int i = 0; i < kNumBoxes; ++i) {
    const uint32_t r = static_cast<uint32_t>(rows[i] <= C::kHalfRows ? rows[i] : C::kHalfRows);
    if (encode_tmap_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool_x, L.H, L.P, L.H, 128, r,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode_tmap_2d(&maps.a[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool2, L.I, L.P, L.I, 128, r,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kernel = a.prof ? gemm_mx_pair_kernel<BT, true> : gemm_mx_pair_kernel<BT, false>;
  if (cudaError_t e = configure_kernel(reinterpret_cast<const void*>(kernel), kLaunchRegs, C::total + 1024))
    return e;
  // pairs of co-resident CTAs: the grid is even and every cluster fits at once
  int clusters = 0;
  if (cudaError_t e = max_pair_clusters(reinterpret_cast<const void*>(kernel), kThreads, C::total + 1024, &clusters))
    return e;
  int grid = g.grid & ~1;
  if (grid > 2 * clusters) grid = 2 * clusters;
  if (grid < 2) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::total + 1024;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = 2; attr[na].val.clusterDim.y = 1; attr[na].val.clusterDim.z = 1;
  ++na;
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

bool mx_pair_block_supported(int bt) { return bt == 80 || bt == 160; }

cudaError_t launch_gemm_mx_pair(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s) {
  switch (g.L->BT) {
    case 80: return launch_impl<80>(g, mode, lag, l1_extra, s);
    case 160: return launch_impl<160>(g, mode, lag, l1_extra, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mm

// Block-scaled grouped GEMMs of the MoE layer on tcgen05 (kind::mxf8f6f4):
// e4m3 activations x e2m1 weights, one UE8M0 scale per 32 contraction elements.
//
// Tile: M = 128 pool rows (the tokens of one pool block of one expert) x
// N = 256 weight rows x K in stages of 128.  On GB300 one M=128, K=32 tcgen05
// MMA takes the same ~143 cycles of tensor-pipe time for every N up to 256
// (measured), so the weights are the N operand at its full width and a block
// with few tokens only wastes accumulator rows, not MMA issue slots.
//   L1: the 256 rows are 128 gate rows and the matching 128 up rows, so a
//       token's gate and up values for 128 intermediate columns sit in one
//       TMEM lane and SwiGLU, the top-k weight and the per-32 UE8M0 requant
//       are thread-local (llm-infra-atlas "07 · MegaMoE" §8).
//   L2: 256 output columns; the epilogue writes fp32 partials part[k][t][h].
//
// Persistent, warp-specialised, one CTA per SM (416 threads):
//   warps 0..3   TMA producers, warp p owns pipeline stage p.  A TMA-issuing
//                thread keeps only about four bulk-tensor copies in flight
//                (measured on GB300), so each stage has its own issuer.  Per
//                stage: one token tile (box of 32, 64 or 128 rows by the
//                block's size), one weight tile (16U4_ALIGN16B, unpacked to
//                1 byte per element in shared memory; L1 fetches the gate and
//                the up rows with one 3-D copy) and the scale chunks.
//   warps 4..11  epilogue: tcgen05.ld of the fp32 accumulator, one token row
//                per thread; the two warps of a TMEM lane quadrant split the
//                columns, so the accumulator is drained (and released to the
//                next tile's MMAs) sooner.
//   warp 12      TMEM allocator + single-thread MMA issuer (tcgen05.cp of the
//                scales into TMEM, 4 MMAs of K=32 per stage).
// The 128 x 256 fp32 accumulator takes half the TMEM; while the epilogue
// drains it the producers keep filling the stages of the next tile.  Every
// wait is bounded: on a deadline the kernel records MM_MOE_ERR_TIMEOUT and a
// site code and returns.
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"

namespace mm {
namespace {

constexpr int kStages = 4;
constexpr int kProducers = kStages;    // one issuing warp per stage
constexpr int kEpiWarp0 = kProducers;  // eight epilogue warps, two per TMEM lane quadrant
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
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
enum : int { kSiteEmpty = 101, kSiteFull = 102, kSiteTmemEmpty = 103, kSiteTmemFull = 104 };

struct Args {
  int T, H, I, E, K;
  int kblocks;        // contraction / 128
  int nblocks;        // weight tiles per expert
  const int* cnt;
  const int* blk_off;
  const int* src;
  const float* topk_w;
  const uint8_t* sfw;   // prepared weight scale chunks (two per tile and k-block)
  const uint8_t* sft;   // token scale chunks (one per pool block and k-block)
  uint8_t* out_codes;   // L1: intermediate codes [P, I]
  uint8_t* out_sf;      // L1: intermediate scale chunks
  float* partials;      // L2: [K, T, H]
  float* dbg;           // L1: raw gate|up accumulators [P, 2I] or null
  int* status;
  uint64_t timeout_ns;
  unsigned long long* prof;   // per-CTA wait/busy nanoseconds (debug_flags bit 1) or null
};

struct TokenMaps {
  CUtensorMap b32, b64, b128;   // pool rows, boxes of 32 / 64 / 128 rows x 128 K
};

struct SmemLayout {
  static constexpr int tok = 0;
  static constexpr int wgt = tok + kStages * kTokBytes;
  static constexpr int sft = wgt + kStages * kWgtBytes;
  static constexpr int sfw = sft + kStages * kSFChunk;
  static constexpr int meta = sfw + kStages * 2 * kSFChunk;           // blk_off[E+1], cnt[E]
  static constexpr int bars_after_meta(int E) { return meta + ((2 * E + 1) * 4 + 15) / 16 * 16; }
  // barriers: full[S], empty[S], tfull, tempty
  static constexpr int nbars = 2 * kStages + 2;
  static constexpr int total(int E) { return bars_after_meta(E) + nbars * 8 + 16; }
};
static_assert(SmemLayout::total(kMaxE) + 1024 <= 232448, "shared memory budget");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");

__device__ __forceinline__ void decode_tile(int tile, int nblocks, const int* blk_off, const int* cnt, int E,
                                            int& e, int& n, int& b, int& valid) {
  // tiles run expert by expert; inside an expert weight tile n outer, pool block inner
  int lo = 0, hi = E - 1;                      // largest e with blk_off[e] * nblocks <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (blk_off[mid] * nblocks <= tile) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int nb = blk_off[e + 1] - blk_off[e];
  const int local = tile - blk_off[e] * nblocks;
  n = local / nb;
  const int bl = local - n * nb;
  b = blk_off[e] + bl;
  const int rem = cnt[e] - bl * kBT;
  valid = rem < kBT ? rem : kBT;
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A = e4m3 (0) in
// bits [9:7], B = e2m1 (5) in [12:10], both K-major, N>>3 in [22:17], UE8M0
// scales (bit 23), M>>4 in [28:24]; the scale-factor byte selectors of B and A
// sit in [5:4] and [30:29].
__device__ __forceinline__ uint32_t make_idesc(int sf_id) {
  return (0u << 7) | (5u << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (static_cast<uint32_t>(sf_id) << 29) | (static_cast<uint32_t>(sf_id) << 4);
}

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ TokenMaps tmT, const Args args) {
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
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + SmemLayout::nbars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Status st{args.status, args.timeout_ns};

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp < kProducers && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmT.b32);
    prefetch_tmap(&tmT.b64);
    prefetch_tmap(&tmT.b128);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i <= E; i += kThreads) s_blk[i] = args.blk_off[i];
  for (int i = threadIdx.x; i < E; i += kThreads) s_cnt[i] = args.cnt[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const int total = s_blk[E] * args.nblocks;
  const int KB = args.kblocks;

  if (warp < kProducers) {
    // ------------------------------------------------------------------ TMA producers
    if (lane == 0) {
      const int p = warp;                       // this warp fills stage p, phases 0,1,0,...
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_t = policy_evict_last();
      uint8_t* tk = smem + SmemLayout::tok + p * kTokBytes;
      uint8_t* wg = smem + SmemLayout::wgt + p * kWgtBytes;
      uint8_t* st_ = smem + SmemLayout::sft + p * kSFChunk;
      uint8_t* sw = smem + SmemLayout::sfw + p * 2 * kSFChunk;
      uint64_t w_empty = 0;
      int step = 0;                             // global k-block step of this CTA
      for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x) {
        int e, n, b, valid;
        decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
        const CUtensorMap* tt = valid <= 32 ? &tmT.b32 : (valid <= 64 ? &tmT.b64 : &tmT.b128);
        const int rows = valid <= 32 ? 32 : (valid <= 64 ? 64 : 128);
        const uint32_t bytes = rows * kBK + kWgtTxBytes + 3 * kSFChunk;
        const uint8_t* sfw = args.sfw + (static_cast<size_t>(e) * args.nblocks + n) * KB * 2 * kSFChunk;
        const uint8_t* sft = args.sft + static_cast<size_t>(b) * KB * kSFChunk;
        int kb = ((p - step) % kStages + kStages) % kStages;   // first k-block of this tile on stage p
        for (; kb < KB; kb += kStages) {
          const uint32_t phase = ((step + kb) / kStages) & 1;
          const uint64_t t0 = args.prof ? globaltimer() : 0;
          if (!mbar_wait(&empty[p], phase ^ 1, st, s_abort, kSiteEmpty)) break;
          if (args.prof) w_empty += globaltimer() - t0;
          mbar_arrive_expect_tx(&full[p], bytes);
          const int kc = kb * kBK;
          tma_load_2d(tk, tt, &full[p], kc, b * kBT, pol_t);
          if (PHASE == 1) tma_load_3d(wg, &tmW, &full[p], kc, e * 2 * args.I + n * 128, 0, pol_w);
          else tma_load_2d(wg, &tmW, &full[p], kc, e * args.H + n * kBN, pol_w);
          bulk_load(st_, sft + static_cast<size_t>(kb) * kSFChunk, kSFChunk, &full[p]);
          bulk_load(sw, sfw + static_cast<size_t>(kb) * 2 * kSFChunk, 2 * kSFChunk, &full[p]);
        }
        step += KB;
      }
      if (args.prof) atomicAdd(&args.prof[blockIdx.x * 8 + 0], static_cast<unsigned long long>(w_empty));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      uint64_t w_full = 0, w_tempty = 0;
      const uint64_t t_start = globaltimer();
      for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x, ++it) {
        const uint64_t t0 = args.prof ? globaltimer() : 0;
        if (!mbar_wait(tempty, (it & 1) ^ 1, st, s_abort, kSiteTmemEmpty)) break;
        if (args.prof) w_tempty += globaltimer() - t0;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          const uint64_t t1 = args.prof ? globaltimer() : 0;
          if (!mbar_wait(&full[stage], phase, st, s_abort, kSiteFull)) { ok = false; break; }
          if (args.prof) w_full += globaltimer() - t1;
          tc_fence_after();
          const uint32_t sft_col = tmem + kSfCol0 + stage * kSfColsPerStage;
          const uint32_t sfw_col = sft_col + 4;
          const uint32_t sf_t = smem_u32(smem + SmemLayout::sft + stage * kSFChunk);
          const uint32_t sf_w = smem_u32(smem + SmemLayout::sfw + stage * 2 * kSFChunk);
          tc_cp_32x128b_warpx4(sft_col, make_smem_desc(sf_t, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfw_col, make_smem_desc(sf_w, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfw_col + 4, make_smem_desc(sf_w + kSFChunk, 0, 128, 0));
          const uint32_t a0 = smem_u32(smem + SmemLayout::tok + stage * kTokBytes);
          const uint32_t b0 = smem_u32(smem + SmemLayout::wgt + stage * kWgtBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = make_smem_desc(a0 + kk * 32, 16, 1024, 2);
            const uint64_t bdesc = make_smem_desc(b0 + kk * 32, 16, 1024, 2);
            tc_mma_mxf8f6f4(tmem, adesc, bdesc, make_idesc(kk), sft_col, sfw_col, (kb | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(tfull);
      }
      if (args.prof) {
        args.prof[blockIdx.x * 8 + 1] = w_full;
        args.prof[blockIdx.x * 8 + 2] = w_tempty;
        args.prof[blockIdx.x * 8 + 3] = globaltimer() - t_start;
        args.prof[blockIdx.x * 8 + 4] = it;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (8 warps)
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    const int half = (warp - kEpiWarp0) >> 2;   // which half of the columns
    const int m = q * 32 + lane;           // accumulator row = pool row inside the block
    const uint32_t tlane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int it = 0;
    uint64_t w_tfull = 0, busy = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, n, b, valid;
      decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
      const bool live = m < valid;
      const size_t row = static_cast<size_t>(b) * kBT + m;
      const int s = live ? __ldg(args.src + row) : 0;
      const float w = (PHASE == 1 && live) ? __ldg(args.topk_w + s) : 0.f;   // loaded before the wait
      const uint64_t t0 = args.prof ? globaltimer() : 0;
      if (!mbar_wait(tfull, it & 1, st, s_abort, kSiteTmemFull)) break;
      const uint64_t t1 = args.prof ? globaltimer() : 0;
      tc_fence_after();
      if (PHASE == 1) {
        uint8_t* crow = args.out_codes + row * args.I + n * 128;
        uint8_t* sfrow = args.out_sf + (static_cast<size_t>(b) * (args.I / 128) + n) * kSFChunk +
                         (m & 31) * 16 + (m >> 5) * 4;
#pragma unroll 1
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tlane + c * 32, g);
          tmem_ld_32x32b_x32(tlane + 128 + c * 32, u);
          tmem_ld_wait();
          if (live) {
            if (args.dbg) {
              float* drow = args.dbg + row * 2 * args.I;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                drow[n * 128 + c * 32 + j] = __uint_as_float(g[j]);
                drow[args.I + n * 128 + c * 32 + j] = __uint_as_float(u[j]);
              }
            }
            float a[32];
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float gv = __uint_as_float(g[j]);
              const float sv = gv * __frcp_rn(1.0f + __expf(-gv));   // silu(g) = g * sigmoid(g)
              a[j] = sv * __uint_as_float(u[j]) * w;
              amax = fmaxf(amax, fabsf(a[j]));
            }
            // UE8M0: smallest e with 448 * 2^e >= max(amax, 1e-10)
            const uint32_t bits = __float_as_uint(fmaxf(amax, 1e-10f));
            const int ex = static_cast<int>((bits >> 23) & 0xFF) - 126;
            int ee = ex - 9 + ((bits & 0x7FFFFF) > 0x600000 ? 1 : 0);
            ee = ee < -127 ? -127 : (ee > 126 ? 126 : ee);
            const float scale = __uint_as_float(static_cast<uint32_t>(127 - ee) << 23);
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t lo = cvt_e4m3x2(a[4 * i] * scale, a[4 * i + 1] * scale);
              const uint32_t hi = cvt_e4m3x2(a[4 * i + 2] * scale, a[4 * i + 3] * scale);
              packed[i] = lo | (hi << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(crow + c * 32);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            sfrow[c] = static_cast<uint8_t>(ee + 127);
          }
        }
      } else {
        const int t = s / args.K;
        const int k = s - t * args.K;
        float* prow = args.partials + (static_cast<size_t>(k) * args.T + t) * args.H + n * kBN;
        const int cols = args.H - n * kBN < kBN ? args.H - n * kBN : kBN;
#pragma unroll 1
        for (int c = half * (kBN / 64); c < (half + 1) * (kBN / 64); ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tlane + c * 32, v);
          tmem_ld_wait();
          if (live && c * 32 < cols) {
            float4* dst = reinterpret_cast<float4*>(prow + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                   __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      if (args.prof) { w_tfull += t1 - t0; busy += globaltimer() - t1; }
    }
    if (args.prof && warp == kEpiWarp0 && lane == 0) {
      args.prof[blockIdx.x * 8 + 5] = w_tfull;
      args.prof[blockIdx.x * 8 + 6] = busy;
    }
  }

  __syncthreads();
  if (*s_abort) {
    // let in-flight bulk copies and MMAs land before the TMEM and smem go away
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 200000) {}
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int PHASE>
cudaError_t launch_impl(const GemmLaunch& g, cudaStream_t s) {
  const Layout& L = *g.L;
  const WsPtrs& W = *g.W;
  CUtensorMap tmW;
  TokenMaps tmT;
  Args a{};
  a.T = L.T; a.H = L.H; a.I = L.I; a.E = L.E; a.K = L.K;
  a.cnt = W.cnt; a.blk_off = W.blk_off; a.src = W.src; a.topk_w = g.topk_w;
  a.sfw = g.wsfp; a.status = W.status; a.timeout_ns = g.timeout_ns;
  a.dbg = PHASE == 1 ? g.dbg : nullptr;
  a.prof = g.prof ? g.prof + (PHASE - 1) * 8 * 1024 : nullptr;
  const uint8_t* pool;
  int kdim;
  if (PHASE == 1) {
    a.kblocks = L.H / 128;
    a.nblocks = L.I / 128;
    a.sft = W.pool_x_sf;
    a.out_codes = W.pool2;
    a.out_sf = W.pool2_sf;
    // W1 as (k, row, half): half 1 is I rows below half 0, so one box of
    // {128 k, 128 rows, 2 halves} is 128 gate rows followed by the matching 128 up rows
    const uint64_t dims[3] = {static_cast<uint64_t>(L.H), static_cast<uint64_t>(L.E) * 2 * L.I - L.I, 2};
    const uint64_t strides[2] = {static_cast<uint64_t>(L.H) / 2, static_cast<uint64_t>(L.I) * L.H / 2};
    const uint32_t box[3] = {128, 128, 2};
    if (encode_tmap(&tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, g.w, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    pool = W.pool_x;
    kdim = L.H;
  } else {
    a.kblocks = L.I / 128;
    a.nblocks = (L.H + kBN - 1) / kBN;
    a.sft = W.pool2_sf;
    a.partials = W.part;
    if (encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w, L.I, static_cast<uint64_t>(L.E) * L.H,
                       L.I / 2, 128, kBN, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    pool = W.pool2;
    kdim = L.I;
  }
  CUtensorMap* maps[3] = {&tmT.b32, &tmT.b64, &tmT.b128};
  for (int i = 0; i < 3; ++i)
    if (encode_tmap_2d(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, pool, kdim, L.P, kdim, 128, 32u << i,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  const int smem = SmemLayout::total(L.E) + 1024;
  static int configured[2] = {-1, -1};
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured[PHASE - 1] != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_mx_kernel<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SmemLayout::total(kMaxE) + 1024);
    if (e != cudaSuccess) return e;
    configured[PHASE - 1] = dev;
  }
  gemm_mx_kernel<PHASE><<<g.grid, kThreads, smem, s>>>(tmW, tmT, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_mx_l1(const GemmLaunch& g, cudaStream_t s) { return launch_impl<1>(g, s); }
cudaError_t launch_gemm_mx_l2(const GemmLaunch& g, cudaStream_t s) { return launch_impl<2>(g, s); }

}  // namespace mm

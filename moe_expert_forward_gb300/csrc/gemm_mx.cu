// Block-scaled grouped GEMMs of the MoE layer on tcgen05 (kind::mxf8f6f4):
// e2m1 weights x e4m3 activations, one UE8M0 scale per 32 contraction elements.
//
// Orientation ("swap-AB"): the MMA's M operand is 128 weight rows, its N operand
// the tokens of one pool block (N = valid tokens rounded up to 16, <= 128), so a
// block with few tokens costs few MMA columns (the pages' small-M problem:
// llm-infra-atlas "07 · MegaMoE" §5 on get_valid_m and UMMA_N).
//
// Persistent, warp-specialised, one CTA per SM (192 threads):
//   warp 0      TMA producer: weights (16U4_ALIGN16B, unpacked to 1 byte per
//               element in shared memory), token rows, both 512-byte scale chunks
//   warp 1      TMEM allocator + single-thread MMA issuer (tcgen05.cp of the
//               scales into TMEM, 4 MMAs of K=32 per 128-K stage)
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator;
//               L1: SwiGLU x top-k weight, UE8M0 requant to e4m3 into the
//                   intermediate pool (llm-infra-atlas "07 · MegaMoE" §8);
//               L2: fp32 partials part[k][t][h].
// Accumulators are double-buffered in TMEM (2 x 128 columns) so the epilogue of
// one tile overlaps the main loop of the next.  Every wait is bounded: on a
// deadline the kernel records MM_MOE_ERR_TIMEOUT and a site code and returns.
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"

namespace mm {
namespace {

constexpr int kStages = 5;
constexpr int kThreads = 192;
constexpr int kABytes = 128 * kBK;     // 128 weight rows x 128 K, 1 byte per element in smem
// A 16U4_ALIGN16B tile load completes the mbarrier transaction count with the
// PACKED bytes it read from global memory (half a byte per element), not with
// the unpacked bytes it wrote to shared memory (measured on GB300).
constexpr int kATxBytes = kABytes / 2;
constexpr int kBBytes = kBT * kBK;     // 128 token rows x 128 K
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = 2 * kBT;       // scale-factor columns after the two accumulators
constexpr int kGuStride = 33;          // padded row of the L1 gate/up staging buffer

// wait-site codes reported through the status word
enum : int { kSiteEmpty = 101, kSiteFull = 102, kSiteTmemEmpty = 103, kSiteTmemFull = 104, kSiteEpiBar = 105 };

struct Args {
  int T, H, I, E, K;
  int kblocks;        // contraction / 128
  int nblocks;        // weight-row tiles per expert
  const int* cnt;
  const int* blk_off;
  const int* src;
  const float* topk_w;
  const uint8_t* sfa;   // prepared weight scale chunks
  const uint8_t* sfb;   // token scale chunks
  uint8_t* out_codes;   // L1: intermediate codes [P, I]
  uint8_t* out_sf;      // L1: intermediate scale chunks
  float* partials;      // L2: [K, T, H]
  float* dbg;           // L1: raw gate|up accumulators [P, 2I] or null
  int* status;
  uint64_t timeout_ns;
  int a_tx_bytes;       // transaction bytes the weight tile's TMA reports (kATxBytes)
};

struct SmemLayout {
  static constexpr int a = 0;
  static constexpr int b = a + kStages * kABytes;
  static constexpr int sfa = b + kStages * kBBytes;
  static constexpr int sfb = sfa + kStages * kSFChunk;
  static constexpr int gu = sfb + kStages * kSFChunk;                 // L1 only: G[64][33], U[64][33] fp32
  static constexpr int srcs = gu + 2 * 64 * kGuStride * 4;            // [2][128] int
  static constexpr int meta = srcs + 2 * kBT * 4;                     // blk_off[E+1], cnt[E]
  static constexpr int bars_after_meta(int E) { return meta + ((2 * E + 1) * 4 + 15) / 16 * 16; }
  // barriers: full[S], empty[S], tfull[2], tempty[2], epi
  static constexpr int nbars = 2 * kStages + 5;
  static constexpr int total(int E) { return bars_after_meta(E) + nbars * 8 + 16; }
};

__device__ __forceinline__ void decode_tile(int tile, int nblocks, const int* blk_off, const int* cnt, int E,
                                            int& e, int& n, int& b, int& valid) {
  // largest e with blk_off[e] * nblocks <= tile
  int lo = 0, hi = E - 1;
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

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A = e2m1 (5) in
// bits [9:7], B = e4m3 (0) in [12:10], both K-major, N>>3 in [22:17], UE8M0
// scales (bit 23), M>>4 in [28:24]; the scale-factor byte selectors of B and A
// sit in [5:4] and [30:29].
__device__ __forceinline__ uint32_t make_idesc(int n, int sf_id) {
  return (5u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (static_cast<uint32_t>(sf_id) << 29) | (static_cast<uint32_t>(sf_id) << 4);
}

// Bounded 128-thread rendezvous of the epilogue warps on an mbarrier.
struct EpiBar {
  uint64_t* bar;
  uint32_t phase;
  __device__ __forceinline__ bool sync(const Status& st, volatile int* abort) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, st, abort, kSiteEpiBar);
    phase ^= 1;
    return ok;
  }
};

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int E = args.E;
  int* s_blk = reinterpret_cast<int*>(smem + SmemLayout::meta);
  int* s_cnt = s_blk + E + 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::bars_after_meta(E));
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* epibar = tempty + 2;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(epibar, 128);
    *s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
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

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x) {
        int e, n, b, valid;
        decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
        const int boxes = (valid + 31) >> 5;
        const uint32_t bytes = args.a_tx_bytes + boxes * 32 * kBK + 2 * kSFChunk;
        const uint8_t* sfa = args.sfa + (static_cast<size_t>(e) * args.nblocks + n) * KB * kSFChunk;
        const uint8_t* sfb = args.sfb + static_cast<size_t>(b) * KB * kSFChunk;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, st, s_abort, kSiteEmpty)) break;
          mbar_arrive_expect_tx(&full[stage], bytes);
          uint8_t* a = smem + SmemLayout::a + stage * kABytes;
          uint8_t* bb = smem + SmemLayout::b + stage * kBBytes;
          const int kc = kb * kBK;
          if (PHASE == 1) {
            tma_load_2d(a, &tmA, &full[stage], kc, e * 2 * args.I + n * 64, pol_w);
            tma_load_2d(a + 64 * kBK, &tmA, &full[stage], kc, e * 2 * args.I + args.I + n * 64, pol_w);
          } else {
            tma_load_2d(a, &tmA, &full[stage], kc, e * args.H + n * 128, pol_w);
          }
          for (int r = 0; r < boxes; ++r) tma_load_2d(bb + r * 32 * kBK, &tmB, &full[stage], kc, b * kBT + r * 32, pol_x);
          bulk_load(smem + SmemLayout::sfa + stage * kSFChunk, sfa + static_cast<size_t>(kb) * kSFChunk, kSFChunk,
                    &full[stage]);
          bulk_load(smem + SmemLayout::sfb + stage * kSFChunk, sfb + static_cast<size_t>(kb) * kSFChunk, kSFChunk,
                    &full[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x, ++it) {
        int e, n, b, valid;
        decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
        const int N = ((valid + 15) >> 4) << 4;
        const int acc = it & 1;
        if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, st, s_abort, kSiteTmemEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * kBT;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, st, s_abort, kSiteFull)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sfa_col = tmem + kSfCol0 + stage * 8;
          const uint32_t sfb_col = sfa_col + 4;
          tc_cp_32x128b_warpx4(sfa_col, make_smem_desc(smem_u32(smem + SmemLayout::sfa + stage * kSFChunk), 0, 128, 0));
          tc_cp_32x128b_warpx4(sfb_col, make_smem_desc(smem_u32(smem + SmemLayout::sfb + stage * kSFChunk), 0, 128, 0));
          const uint32_t a0 = smem_u32(smem + SmemLayout::a + stage * kABytes);
          const uint32_t b0 = smem_u32(smem + SmemLayout::b + stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = make_smem_desc(a0 + kk * 32, 16, 1024, 2);
            const uint64_t bdesc = make_smem_desc(b0 + kk * 32, 16, 1024, 2);
            tc_mma_mxf8f6f4(d, adesc, bdesc, make_idesc(N, kk), sfa_col, sfb_col, (kb | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    const int m = q * 32 + lane;           // accumulator row = weight row of the tile
    const int et = (warp - 2) * 32 + lane; // 0..127
    EpiBar eb{epibar, 0};
    float* G = reinterpret_cast<float*>(smem + SmemLayout::gu);
    float* U = G + 64 * kGuStride;
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, n, b, valid;
      decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
      int* srcs = reinterpret_cast<int*>(smem + SmemLayout::srcs) + (it & 1) * kBT;
      srcs[et] = et < valid ? args.src[static_cast<size_t>(b) * kBT + et] : -1;
      const int acc = it & 1;
      if (!mbar_wait(&tfull[acc], (it >> 1) & 1, st, s_abort, kSiteTmemFull)) break;
      tc_fence_after();
      if (!eb.sync(st, s_abort)) break;    // srcs visible to all epilogue threads
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * kBT;
      const int chunks = (valid + 31) >> 5;
      bool ok = true;
      if (PHASE == 2) {
        float* prow = args.partials + static_cast<size_t>(n) * 128 + m;
        for (int c = 0; c < chunks; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = c * 32 + j;
            if (col < valid) {
              const int s = srcs[col];
              const int t = s / args.K;
              const int k = s - t * args.K;
              prow[(static_cast<size_t>(k) * args.T + t) * args.H] = __uint_as_float(v[j]);
            }
          }
        }
      } else {
        const int token = et >> 2;          // 0..31 within the chunk
        const int jq = et & 3;              // 16 intermediate columns each
        for (int c = 0; c < chunks && ok; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, v);
          tmem_ld_wait();
          if (args.dbg) {
            const int wrow = (m < 64) ? n * 64 + m : args.I + n * 64 + (m - 64);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j < valid)
                args.dbg[(static_cast<size_t>(b) * kBT + c * 32 + j) * 2 * args.I + wrow] = __uint_as_float(v[j]);
          }
          float* dst = (m < 64 ? G : U) + (m & 63) * kGuStride;
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[j] = __uint_as_float(v[j]);
          if (!eb.sync(st, s_abort)) { ok = false; break; }
          const int col = c * 32 + token;
          const bool live = col < valid;
          float a[16];
          float amax = 0.f;
          if (live) {
            const float w = __ldg(args.topk_w + srcs[col]);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int jj = jq * 16 + i;
              const float g = G[jj * kGuStride + token];
              const float u = U[jj * kGuStride + token];
              const float s = g / (1.0f + expf(-g));
              a[i] = s * u * w;
              amax = fmaxf(amax, fabsf(a[i]));
            }
          }
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          if (live) {
            // UE8M0: smallest e with 448 * 2^e >= max(amax, 1e-10)
            const uint32_t bits = __float_as_uint(fmaxf(amax, 1e-10f));
            int ex = static_cast<int>((bits >> 23) & 0xFF) - 126;
            int ee = ex - 9 + ((bits & 0x7FFFFF) > 0x600000 ? 1 : 0);
            ee = ee < -127 ? -127 : (ee > 126 ? 126 : ee);
            const float scale = __uint_as_float(static_cast<uint32_t>(127 - ee) << 23);
            uint32_t packed[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t lo = cvt_e4m3x2(a[4 * i] * scale, a[4 * i + 1] * scale);
              const uint32_t hi = cvt_e4m3x2(a[4 * i + 2] * scale, a[4 * i + 3] * scale);
              packed[i] = lo | (hi << 16);
            }
            const size_t row = static_cast<size_t>(b) * kBT + col;
            *reinterpret_cast<uint4*>(args.out_codes + row * args.I + n * 64 + jq * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            if ((jq & 1) == 0) {
              const int kb32 = n * 2 + (jq >> 1);
              args.out_sf[(static_cast<size_t>(b) * (args.I / 128) + (kb32 >> 2)) * kSFChunk +
                          (col & 31) * 16 + (col >> 5) * 4 + (kb32 & 3)] = static_cast<uint8_t>(ee + 127);
            }
          }
          if (!eb.sync(st, s_abort)) { ok = false; break; }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (!ok) break;
    }
  }

  __syncthreads();
  if (*s_abort) {
    // let in-flight bulk copies and MMAs land before the TMEM and smem go away
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 200000) {}
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int PHASE>
cudaError_t launch_impl(const GemmLaunch& g, cudaStream_t s) {
  const Layout& L = *g.L;
  const WsPtrs& W = *g.W;
  CUtensorMap tmA, tmB;
  Args a{};
  a.T = L.T; a.H = L.H; a.I = L.I; a.E = L.E; a.K = L.K;
  a.cnt = W.cnt; a.blk_off = W.blk_off; a.src = W.src; a.topk_w = g.topk_w;
  a.sfa = g.wsfp; a.status = W.status; a.timeout_ns = g.timeout_ns;
  a.dbg = PHASE == 1 ? g.dbg : nullptr;
  a.a_tx_bytes = kATxBytes;
  CUresult r;
  if (PHASE == 1) {
    a.kblocks = L.H / 128;
    a.nblocks = L.I / 64;
    a.sfb = W.pool_x_sf;
    a.out_codes = W.pool2;
    a.out_sf = W.pool2_sf;
    r = encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w, L.H, static_cast<uint64_t>(L.E) * 2 * L.I,
                       L.H / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    r = encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool_x, L.H, L.P, L.H, 128, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    a.kblocks = L.I / 128;
    a.nblocks = L.H / 128;
    a.sfb = W.pool2_sf;
    a.partials = W.part;
    r = encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w, L.I, static_cast<uint64_t>(L.E) * L.H,
                       L.I / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    r = encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.pool2, L.I, L.P, L.I, 128, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
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
  gemm_mx_kernel<PHASE><<<g.grid, kThreads, smem, s>>>(tmA, tmB, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_mx_l1(const GemmLaunch& g, cudaStream_t s) { return launch_impl<1>(g, s); }
cudaError_t launch_gemm_mx_l2(const GemmLaunch& g, cudaStream_t s) { return launch_impl<2>(g, s); }

int gemm_mx_smem_bytes(int E) { return SmemLayout::total(E) + 1024; }

}  // namespace mm

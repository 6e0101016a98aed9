// Dispatch (routing histogram, segment offsets, stable slots), gather into the
// pool, fixed-order combine, weight-scale relayout and intermediate read-back.
#include <cuda_bf16.h>

#include "combine.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mm {

// Byte offset of (row r, 32-element scale block kk in 0..3) inside a 512-byte
// scale chunk that covers 128 rows x 128 contraction elements.  The chunk is the
// source of one tcgen05.cp.32x128b.warpx4: 16-byte line (r % 32) holds the four
// words of rows r%32, r%32+32, r%32+64, r%32+96; word byte kk is the scale of
// contraction block kk.
__host__ __device__ __forceinline__ int sf_chunk_offset(int r, int kk) {
  return (r & 31) * 16 + (r >> 5) * 4 + kk;
}

// ----------------------------------------------------------------------------- dispatch
// Two kernels over G CTAs; CTA g owns the contiguous flat pairs
// p = t*K + k in [g*CH, (g+1)*CH).
//   count:  per-CTA expert histogram cc[g][e] (shared-memory atomics).
//   assign: every CTA rebuilds, from cc, the totals cnt[e], the segment offsets
//           blk_off (exclusive scan of ceil(cnt/BT)) and its own starting rank
//           inside each expert (sum of cc over earlier CTAs); its 8 warps then
//           count their sub-ranges, take exclusive offsets over warps, and rank
//           equal experts inside each 32-pair step with __match_any_sync.  The
//           slot order is therefore ascending p (= ascending token, then k).
//           CTA 0 publishes cnt/blk_off; padding rows are spread over CTAs.
constexpr int kDispatchThreads = 256;
constexpr int kDispatchWarps = kDispatchThreads / 32;

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_count_kernel(const int32_t* __restrict__ idx, int64_t TK, int E, int64_t CH, int32_t* __restrict__ cc,
                          int32_t* __restrict__ status) {
  extern __shared__ int sc[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sc[e] = 0;
  __syncthreads();
  const int64_t beg = static_cast<int64_t>(blockIdx.x) * CH;
  const int64_t end = beg + CH < TK ? beg + CH : TK;
  bool bad = false;
  for (int64_t p = beg + threadIdx.x; p < end; p += blockDim.x) {
    const int e = __ldg(idx + p);
    if (e >= 0 && e < E) atomicAdd(&sc[e], 1);
    else if (e >= E || e < -1) bad = true;
  }
  if (bad) atomicCAS(status, 0, MM_MOE_ERR_BAD_ROUTING);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) cc[static_cast<int64_t>(blockIdx.x) * E + e] = sc[e];
}

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_assign_kernel(const int32_t* __restrict__ idx, int64_t TK, int E, int BT, int64_t CH,
                           const int32_t* __restrict__ cc, int32_t* __restrict__ cnt, int32_t* __restrict__ blk_off,
                           int32_t* __restrict__ slot, int32_t* __restrict__ src) {
  extern __shared__ int sm[];
  pdl_trigger();                             // the GEMM may start its setup meanwhile
  int* wc = sm;                              // [8][E] per-warp counts, then offsets
  int* s_base = wc + kDispatchWarps * E;     // [E] rank of this CTA's first pair inside each expert
  int* s_cnt = s_base + E;                   // [E]
  int* s_blk = s_cnt + E;                    // [E+1]
  __shared__ int s_wsum[kDispatchWarps];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, G = gridDim.x;

  for (int i = tid; i < kDispatchWarps * E; i += blockDim.x) wc[i] = 0;
  for (int e = tid; e < E; e += blockDim.x) {
    int base = 0, tot = 0;
    for (int h = 0; h < G; ++h) {
      const int c = __ldg(cc + static_cast<int64_t>(h) * E + e);
      base += (h < g) ? c : 0;
      tot += c;
    }
    s_base[e] = base;
    s_cnt[e] = tot;
    s_blk[e] = (tot + BT - 1) / BT;
  }
  __syncthreads();

  // exclusive scan of blocks per expert: each thread owns up to 4 consecutive experts
  {
    constexpr int kPer = (kMaxE + kDispatchThreads - 1) / kDispatchThreads;
    int v[kPer];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = tid * kPer + j;
      v[j] = e < E ? s_blk[e] : 0;
      sum += v[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[w] = incl;
    __syncthreads();
    int wpre = 0;
    for (int i = 0; i < w; ++i) wpre += s_wsum[i];
    int run = wpre + incl - sum;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = tid * kPer + j;
      if (e < E) s_blk[e] = run;
      run += v[j];
    }
    if (tid == kDispatchThreads - 1) s_blk[E] = run;
    __syncthreads();
  }
  if (g == 0) {
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = s_cnt[e];
    for (int e = tid; e <= E; e += blockDim.x) blk_off[e] = s_blk[e];
  }

  const int64_t per = CH / kDispatchWarps;   // multiple of 32
  const int64_t beg = static_cast<int64_t>(g) * CH + w * per;
  const int64_t end = beg + per < TK ? beg + per : TK;
  int* my = wc + w * E;
  constexpr int kBatch = 8;                  // independent idx loads in flight per lane
  for (int64_t base0 = beg; base0 < end; base0 += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t p = base0 + j * 32 + lane;
      ev[j] = (p < end) ? __ldg(idx + p) : -1;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (base0 + j * 32 >= end) break;      // warp-uniform
      const int e = ev[j];
      const bool valid = (e >= 0) && (e < E);
      const unsigned m = __match_any_sync(0xffffffffu, valid ? e : -1);
      if (valid && lane == __ffs(m) - 1) my[e] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = s_base[e];
    for (int ww = 0; ww < kDispatchWarps; ++ww) {
      const int c = wc[ww * E + e];
      wc[ww * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int64_t base0 = beg; base0 < end; base0 += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t p = base0 + j * 32 + lane;
      ev[j] = (p < end) ? __ldg(idx + p) : -1;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t p = base0 + j * 32 + lane;
      if (base0 + j * 32 >= end) break;      // warp-uniform
      const int e = ev[j];
      const bool valid = (e >= 0) && (e < E);
      const unsigned m = __match_any_sync(0xffffffffu, valid ? e : -1);
      int before = 0;
      if (valid) before = my[e];
      __syncwarp();
      if (valid) {
        const int rank = __popc(m & ((1u << lane) - 1u));
        const int64_t pos = static_cast<int64_t>(s_blk[e]) * BT + before + rank;
        slot[p] = static_cast<int32_t>(pos);
        src[pos] = static_cast<int32_t>(p);
        if (lane == __ffs(m) - 1) my[e] = before + __popc(m);
      } else if (p < end) {
        slot[p] = -1;
      }
      __syncwarp();
    }
  }
  // padding rows of every segment: expert e is padded by CTA e % G, one warp per expert
  for (int e = g + w * G; e < E; e += G * kDispatchWarps) {
    const int64_t lo = static_cast<int64_t>(s_blk[e]) * BT + s_cnt[e];
    const int64_t hi = static_cast<int64_t>(s_blk[e + 1]) * BT;
    for (int64_t r = lo + lane; r < hi; r += 32) src[r] = -1;
  }
}

int dispatch_ctas(int64_t TK, int E, int64_t scratch_ints) {
  int64_t g = (TK + 511) / 512;
  const int64_t cap_sm = dev_info().sms;
  if (g > cap_sm) g = cap_sm;
  if (g > scratch_ints / E) g = scratch_ints / E;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int K, int E, int block_m, int32_t* cnt,
                            int32_t* blk_off, int32_t* slot, int32_t* src, int32_t* status, int32_t* scratch,
                            int64_t scratch_ints, cudaStream_t s) {
  const int64_t TK = static_cast<int64_t>(T) * K;
  const int G = dispatch_ctas(TK, E, scratch_ints);
  int64_t CH = (TK + G - 1) / G;
  CH = (CH + 32 * kDispatchWarps - 1) / (32 * kDispatchWarps) * (32 * kDispatchWarps);
  if (CH == 0) CH = 32 * kDispatchWarps;
  const size_t smem_assign = static_cast<size_t>(kDispatchWarps + 3) * E * sizeof(int) + 16;
  if (cudaError_t e = configure_kernel(reinterpret_cast<const void*>(dispatch_assign_kernel), 0,
                                       (kDispatchWarps + 3) * kMaxE * static_cast<int>(sizeof(int)) + 16))
    return e;
  dispatch_count_kernel<<<G, kDispatchThreads, E * sizeof(int), s>>>(topk_idx, TK, E, CH, scratch, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dispatch_assign_kernel<<<G, kDispatchThreads, smem_assign, s>>>(topk_idx, TK, E, block_m, CH, scratch, cnt,
                                                                   blk_off, slot, src);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- gather
// Token-major: one warp per token reads the token's row once and writes it to
// each of its pool rows slot[t*K + k] (masked slots are skipped; padding rows
// are never written, the GEMM epilogues ignore them).  MX scales go to the
// 512-byte chunk layout the MMA consumes; F8 scales to a plain [P, H/128] fp32
// array (a GEMM epilogue thread reads four k-blocks of its row with one load).
// Every lane holds the token's K pool rows; the shuffles that spread them run
// with the warp converged.
__device__ __forceinline__ void token_rows(const int32_t* __restrict__ slot, int64_t t, int K, int lane,
                                           int (&rows)[kMaxK]) {
  const int myrow = lane < K ? __ldg(slot + t * K + lane) : -1;
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) rows[k] = __shfl_sync(0xffffffffu, myrow, k);
}

// x holds e4m3 codes [T, H] and their scales (MX: UE8M0 bytes [T, H/32]; F8: fp32 [T, H/128]).
__global__ void __launch_bounds__(256)
    gather_kernel(const int32_t* __restrict__ slot, int T, int K, int H, int BT, int CPB, int variant,
                  const uint8_t* __restrict__ x, const void* __restrict__ x_sf, uint8_t* __restrict__ pool_x,
                  uint8_t* __restrict__ pool_x_sf) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int KB = H / 128;
  for (int64_t t = warp0; t < T; t += nwarps) {
    int rows[kMaxK];
    token_rows(slot, t, K, lane, rows);
    const uint4* srow = reinterpret_cast<const uint4*>(x + t * H);
#pragma unroll 4
    for (int i = lane; i < H / 16; i += 32) {
      const uint4 v = __ldg(srow + i);
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        const int r = k < K ? rows[k] : -1;
        if (r >= 0) reinterpret_cast<uint4*>(pool_x + static_cast<int64_t>(r) * H)[i] = v;
      }
    }
    for (int kb = lane; kb < KB; kb += 32) {
      if (variant == MM_MOE_VARIANT_MX) {
        // the four UE8M0 bytes of one 128-element block, one 32-bit word in either layout
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(x_sf) + t * (H / 32)) + kb);
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          const int r = k < K ? rows[k] : -1;
          if (r >= 0) *reinterpret_cast<uint32_t*>(pool_x_sf + pool_sf_word(r / BT, kb, KB, CPB, r % BT)) = w;
        }
      } else {
        const float sc = __ldg(static_cast<const float*>(x_sf) + t * KB + kb);
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          const int r = k < K ? rows[k] : -1;
          if (r >= 0) reinterpret_cast<float*>(pool_x_sf)[static_cast<int64_t>(r) * KB + kb] = sc;
        }
      }
    }
  }
}

// x holds bf16 activations [T, H]: each token's row is quantised once
// (quant.cuh) and every chunk written to each of the token's pool rows, so the
// division-heavy F8 rule runs once per token rather than once per slot.
__global__ void __launch_bounds__(256)
    gather_quant_kernel(const int32_t* __restrict__ slot, int T, int K, int H, int BT, int CPB, int variant,
                        const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ pool_x,
                        uint8_t* __restrict__ pool_x_sf) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = warp0; t < T; t += nwarps) {
    int rows[kMaxK];
    token_rows(slot, t, K, lane, rows);
    const __nv_bfloat16* brow = x + t * H;
    if (variant == MM_MOE_VARIANT_MX) {
      quant_row_mx_bf16(brow, H, lane, [&](int j, const uint4 (&c)[2], uint8_t sfb, bool) {
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          const int r = k < K ? rows[k] : -1;
          if (r < 0) continue;
          uint4* d = reinterpret_cast<uint4*>(pool_x + static_cast<int64_t>(r) * H) + 2 * j;
          d[0] = c[0];
          d[1] = c[1];
          pool_x_sf[pool_sf_word(r / BT, j >> 2, H / 128, CPB, r % BT) + (j & 3)] = sfb;
        }
      });
    } else {
      quant_row_f8_bf16(brow, H, lane, [&](int c, const uint4 (&cd)[2], float sc, bool lead) {
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          const int r = k < K ? rows[k] : -1;
          if (r < 0) continue;
          uint4* d = reinterpret_cast<uint4*>(pool_x + static_cast<int64_t>(r) * H) + 2 * c;
          d[0] = cd[0];
          d[1] = cd[1];
          if (lead) reinterpret_cast<float*>(pool_x_sf)[static_cast<int64_t>(r) * (H / 128) + (c >> 2)] = sc;
        }
      });
    }
  }
}

cudaError_t launch_gather(const Layout& L, const WsPtrs& W, const uint8_t* x, const void* x_sf, bool x_bf16,
                          cudaStream_t s) {
  const int grid = dev_info().sms * 4;
  if (x_bf16)
    gather_quant_kernel<<<grid, 256, 0, s>>>(W.slot, L.T, L.K, L.H, L.BT, L.CPB, L.variant,
                                             reinterpret_cast<const __nv_bfloat16*>(x), W.pool_x, W.pool_x_sf);
  else
    gather_kernel<<<grid, 256, 0, s>>>(W.slot, L.T, L.K, L.H, L.BT, L.CPB, L.variant, x, x_sf, W.pool_x,
                                       W.pool_x_sf);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- combine
// out[t, h] = bf16(sum over k = 0..K-1 of part[k][t][h]), the sum in fp32 in
// fixed k order; slots with a masked or out-of-range expert are skipped.  Each
// thread takes 8 consecutive columns of one token (combine.cuh).
template <typename PartT>
__global__ void __launch_bounds__(256)
    combine_kernel(const PartT* __restrict__ part, const int32_t* __restrict__ idx, int T, int K, int E, int H,
                   __nv_bfloat16* __restrict__ out) {
  pdl_wait();                                // the partials of the GEMM before this launch
  const int64_t groups = static_cast<int64_t>(T) * (H / 8);
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = g / (H / 8);
    const int h = static_cast<int>(g % (H / 8)) * 8;
    combine8(part, t, h, T, H, K,
             [&](int k) {
               const int e = __ldg(idx + t * K + k);
               return e >= 0 && e < E;
             },
             out);
  }
}

cudaError_t launch_combine(const Layout& L, const WsPtrs& W, const int32_t* topk_idx, void* out, bool pdl,
                           cudaStream_t s) {
  const int64_t groups = static_cast<int64_t>(L.T) * (L.H / 8);
  int64_t blocks = (groups + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev_info().sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  if (L.part_elem == 2)
    return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, reinterpret_cast<const __nv_bfloat16*>(W.part),
                              topk_idx, L.T, L.K, L.E, L.H, o);
  return cudaLaunchKernelEx(&cfg, combine_kernel<float>, static_cast<const float*>(W.part), topk_idx, L.T, L.K, L.E,
                            L.H, o);
}

// ----------------------------------------------------------------------------- weight scales (MX)
// The GEMMs stream weights in tiles of 256 rows x 128 K; each tile's scales are
// two 512-byte chunks (rows 0..127, rows 128..255), stored tile after tile:
//   W1 tile ((e*(I/128) + n)*(H/128) + kb): chunk 0 = gate rows n*128 + r,
//                                          chunk 1 = up rows I + n*128 + r;
//   W2 tile ((e*ceil(H/256) + n)*(I/128) + kb): chunk c = rows n*256 + c*128 + r
//                                          (rows past H are zero).
// One thread moves one 4-byte word (the 4 scale blocks of one row in one tile).
__global__ void prepare_sf_mx_kernel(const uint8_t* __restrict__ w1_sf, const uint8_t* __restrict__ w2_sf,
                                     int H, int I, int E, uint8_t* __restrict__ w1_sfp,
                                     uint8_t* __restrict__ w2_sfp) {
  const int NB1 = I / 128, KB1 = H / 128, NB2 = (H + 255) / 256, KB2 = I / 128;
  const int64_t n1 = static_cast<int64_t>(E) * NB1 * KB1 * 256;
  const int64_t n2 = static_cast<int64_t>(E) * NB2 * KB2 * 256;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < n1 + n2;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (g < n1) {
      const int r = static_cast<int>(g & 255);
      const int64_t tile = g >> 8;
      const int kb = static_cast<int>(tile % KB1);
      const int n = static_cast<int>((tile / KB1) % NB1);
      const int64_t e = tile / (static_cast<int64_t>(KB1) * NB1);
      const int row = (r < 128) ? n * 128 + r : I + n * 128 + (r - 128);
      const uint32_t word =
          *reinterpret_cast<const uint32_t*>(w1_sf + (e * 2 * I + row) * (H / 32) + kb * 4);
      *reinterpret_cast<uint32_t*>(w1_sfp + tile * 2 * kSFChunk + (r >> 7) * kSFChunk + sf_chunk_offset(r & 127, 0)) =
          word;
    } else {
      const int64_t h = g - n1;
      const int r = static_cast<int>(h & 255);
      const int64_t tile = h >> 8;
      const int kb = static_cast<int>(tile % KB2);
      const int n = static_cast<int>((tile / KB2) % NB2);
      const int64_t e = tile / (static_cast<int64_t>(KB2) * NB2);
      const int row = n * 256 + r;
      const uint32_t word =
          row < H ? *reinterpret_cast<const uint32_t*>(w2_sf + (e * H + row) * (I / 32) + kb * 4) : 0u;
      *reinterpret_cast<uint32_t*>(w2_sfp + tile * 2 * kSFChunk + (r >> 7) * kSFChunk + sf_chunk_offset(r & 127, 0)) =
          word;
    }
  }
}

cudaError_t launch_prepare_sf_mx(const uint8_t* w1_sf, const uint8_t* w2_sf, int H, int I, int E,
                                 uint8_t* w1_sfp, uint8_t* w2_sfp, cudaStream_t s) {
  prepare_sf_mx_kernel<<<dev_info().sms * 8, 256, 0, s>>>(w1_sf, w2_sf, H, I, E, w1_sfp, w2_sfp);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- intermediate read-back
// Shared experts: every token's routing grows by S slots naming experts
// E .. E+S-1 with weight 1, after its K routed slots.  A routed id in [E, E+S)
// would otherwise name a shared expert, so it becomes -2, which the routing
// kernels mask and flag like any other id out of range.
__global__ void extend_routing_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int K,
                                      int E, int S, int32_t* __restrict__ xidx, float* __restrict__ xw) {
  const int KS = K + S;
  const int64_t n = static_cast<int64_t>(T) * KS;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / KS;
    const int j = static_cast<int>(i - t * KS);
    if (j < K) {
      const int e = idx[t * K + j];
      xidx[i] = (e >= E && e < E + S) ? -2 : e;
      xw[i] = w[t * K + j];
    } else {
      xidx[i] = E + (j - K);
      xw[i] = 1.0f;
    }
  }
}

cudaError_t launch_extend_routing(const int32_t* topk_idx, const float* topk_w, int T, int K, int E, int S,
                                  int32_t* ext_idx, float* ext_w, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(T) * (K + S);
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > dev_info().sms * 8) blocks = dev_info().sms * 8;
  if (blocks < 1) blocks = 1;
  extend_routing_kernel<<<blocks, 256, 0, s>>>(topk_idx, topk_w, T, K, E, S, ext_idx, ext_w);
  return cudaGetLastError();
}

__global__ void read_sf_mx_kernel(const uint8_t* __restrict__ pool2_sf, int64_t rows, int I, int BT, int CPB,
                                  uint8_t* __restrict__ sf) {
  const int KB32 = I / 32;
  const int KB = I / 128;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < rows * KB32;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / KB32;
    const int j = static_cast<int>(g % KB32);
    const int64_t blk = r / BT;
    const int rr = static_cast<int>(r % BT);
    sf[g] = pool2_sf[pool_sf_word(blk, j / 4, KB, CPB, rr) + (j & 3)];
  }
}

cudaError_t launch_read_intermediate(const Layout& L, const WsPtrs& W, int64_t rows, uint8_t* codes,
                                     void* sf, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(codes, W.pool2, static_cast<size_t>(rows) * L.I, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return e;
  if (L.variant == MM_MOE_VARIANT_MX) {
    read_sf_mx_kernel<<<dev_info().sms * 4, 256, 0, s>>>(W.pool2_sf, rows, L.I, L.BT, L.CPB,
                                                         static_cast<uint8_t*>(sf));
    return cudaGetLastError();
  }
  return cudaMemcpyAsync(sf, W.pool2_sf, static_cast<size_t>(rows) * (L.I / L.act_gran) * sizeof(float),
                         cudaMemcpyDeviceToDevice, s);
}

}  // namespace mm

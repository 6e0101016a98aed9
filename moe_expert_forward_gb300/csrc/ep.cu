// Expert parallelism over N ranks (llm-infra-atlas "07 · MegaMoE" §7 and §9;
// DeepGEMM PR #440 "How it works"): per-expert counts, the host plan of every
// pair's row at its owner, the metadata push, the pull of the activation rows
// into the owner's receive buffers, and the combine that reads each pair's bf16
// output back from its owner.  Peers' buffers are plain device pointers read or
// written with ordinary loads and stores; the barriers between the steps are the
// caller's, so no kernel here waits on another rank.
#include <cuda_bf16.h>

#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace mm {
namespace {

constexpr int kCombinePart = 128;   // 16-byte chunks (1024 bf16 columns) a warp sums
constexpr int kSiteEpBarrier = 301;  // status site of a cross-rank barrier that ran out

__global__ void ep_count_kernel(const int32_t* __restrict__ idx, int64_t n, int E, int32_t* __restrict__ counts) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = idx[i];
    if (e >= 0 && e < E) atomicAdd(counts + e, 1);
  }
}

// One thread per pair: its metadata row at its owner.
__global__ void ep_push_meta_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w,
                                    const int32_t* __restrict__ send_row, int64_t n, int E, int Eloc, int rank,
                                    void* const* __restrict__ peer_meta) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = idx[i];
    const int row = send_row[i];
    if (e < 0 || e >= E || row < 0) continue;
    const int owner = e / Eloc;
    int4* meta = static_cast<int4*>(peer_meta[owner]);
    meta[row] = make_int4(rank, static_cast<int>(i), e - owner * Eloc, __float_as_int(w[i]));
  }
}

// One warp per received row: the source token's activations and scales, copied
// 16 bytes a lane (H is a multiple of 128, so every row and scale row is too).
__global__ void ep_pull_kernel(const int4* __restrict__ meta, int64_t rows, int K, int H, int sf_bytes,
                               const void* const* __restrict__ peer_x, const void* const* __restrict__ peer_x_sf,
                               uint8_t* __restrict__ x_recv, uint8_t* __restrict__ x_sf_recv,
                               int32_t* __restrict__ idx_recv, float* __restrict__ w_recv) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t j = warp0; j < rows; j += nwarps) {
    const int4 m = meta[j];
    const int64_t t = m.y / K;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(peer_x[m.x]) + t * H);
    uint4* dst = reinterpret_cast<uint4*>(x_recv + j * H);
    for (int i = lane; i < H / 16; i += 32) dst[i] = src[i];
    const uint8_t* ssrc = static_cast<const uint8_t*>(peer_x_sf[m.x]) + t * sf_bytes;
    uint8_t* sdst = x_sf_recv + j * sf_bytes;
    for (int i = lane; i < sf_bytes / 4; i += 32)
      reinterpret_cast<uint32_t*>(sdst)[i] = reinterpret_cast<const uint32_t*>(ssrc)[i];
    if (lane == 0) {
      idx_recv[j] = m.z;
      w_recv[j] = __int_as_float(m.w);
    }
  }
}

// One warp per (token, 1024-column part): out[t] = bf16(sum over k of its pairs'
// bf16 outputs at their owners), the sum in fp32 in k order; 8 bf16 (16 bytes) a
// lane a step.  Lane k < K resolves slot k's source row once; the row addresses
// are then broadcast, so every step issues its K independent loads back to back.
__global__ void ep_combine_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ send_row, int T,
                                  int K, int E, int Eloc, int H, const void* const* __restrict__ peer_out,
                                  __nv_bfloat16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int parts = (H / 8 + kCombinePart - 1) / kCombinePart;
  for (int64_t w = warp0; w < static_cast<int64_t>(T) * parts; w += nwarps) {
    const int64_t t = w / parts;
    const int c0 = static_cast<int>(w - t * parts) * kCombinePart;
    const int c1 = c0 + kCombinePart < H / 8 ? c0 + kCombinePart : H / 8;
    const uint4* mine = nullptr;
    if (lane < K) {
      const int e = idx[t * K + lane];
      const int row = send_row[t * K + lane];
      if (e >= 0 && e < E && row >= 0)
        mine = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(peer_out[e / Eloc]) +
                                              static_cast<int64_t>(row) * H);
    }
    const uint4* src[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
      src[k] = reinterpret_cast<const uint4*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(mine), k));
    for (int c = c0 + lane; c < c1; c += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        if (k >= K || !src[k]) continue;
        const uint4 v = src[k][c];
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(p[i]);
          acc[2 * i] += f.x;
          acc[2 * i + 1] += f.y;
        }
      }
      uint4 o;
      __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      reinterpret_cast<uint4*>(out + t * H)[c] = o;
    }
  }
}

// One warp per received row: its bf16 output to the pair's row of the source
// rank's partial buffer.
__global__ void ep_push_out_kernel(const int4* __restrict__ meta, int64_t rows, int H,
                                   const __nv_bfloat16* __restrict__ out_recv, void* const* __restrict__ peer_partials) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t j = warp0; j < rows; j += nwarps) {
    const int4 m = meta[j];
    const uint4* src = reinterpret_cast<const uint4*>(out_recv + j * H);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(peer_partials[m.x]) +
                                          static_cast<int64_t>(m.y) * H);
    for (int i = lane; i < H / 8; i += 32) dst[i] = src[i];
  }
}

// One warp per (token, 1024-column part): the token's K bf16 partials summed in
// fp32 in k order, rounded once to bf16.
__global__ void ep_combine_local_kernel(const int32_t* __restrict__ idx, int T, int K, int E, int H,
                                        const __nv_bfloat16* __restrict__ part, __nv_bfloat16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int parts = (H / 8 + kCombinePart - 1) / kCombinePart;
  for (int64_t w = warp0; w < static_cast<int64_t>(T) * parts; w += nwarps) {
    const int64_t t = w / parts;
    const int c0 = static_cast<int>(w - t * parts) * kCombinePart;
    const int c1 = c0 + kCombinePart < H / 8 ? c0 + kCombinePart : H / 8;
    const int e_mine = lane < K ? idx[t * K + lane] : -1;
    const uint32_t valid = __ballot_sync(0xffffffffu, e_mine >= 0 && e_mine < E);
    for (int c = c0 + lane; c < c1; c += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        if (k >= K || !((valid >> k) & 1u)) continue;
        const uint4 v = reinterpret_cast<const uint4*>(part + (t * K + k) * H)[c];
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(p[i]);
          acc[2 * i] += f.x;
          acc[2 * i + 1] += f.y;
        }
      }
      uint4 o;
      __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      reinterpret_cast<uint4*>(out + t * H)[c] = o;
    }
  }
}

// Cross-rank barrier (the pages' NVLink barrier, llm-infra-atlas "07 · MegaMoE"
// §10), bounded: rank `rank` stores `epoch` into slot `rank` of every rank's flag
// array (system-scope release), then waits until every slot of its own array has
// reached `epoch` (system-scope acquire) or the deadline passes, which it records
// as MM_MOE_ERR_TIMEOUT with site 301 and the first missing rank.  Epochs only
// grow, so the flags are never reset.  One thread does the work.
__device__ bool ep_barrier_body(uint32_t* const* peer_flags, int N, int rank, uint32_t epoch, uint64_t timeout_ns,
                                int32_t* status) {
  for (int r = 0; r < N; ++r)
    asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(peer_flags[r] + rank), "r"(epoch) : "memory");
  const uint32_t* mine = peer_flags[rank];
  const uint64_t t0 = globaltimer();
  for (int r = 0; r < N; ++r) {
    for (;;) {
      uint32_t v;
      asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(mine + r) : "memory");
      if (static_cast<int32_t>(v - epoch) >= 0) break;
      if (globaltimer() - t0 > timeout_ns) {
        if (atomicCAS(status, 0, MM_MOE_ERR_TIMEOUT) == 0) {
          status[1] = kSiteEpBarrier;
          status[2] = r;
        }
        return false;
      }
    }
  }
  return true;
}

__global__ void ep_barrier_kernel(uint32_t* const* peer_flags, int N, int rank, uint32_t epoch, uint64_t timeout_ns,
                                  int32_t* status) {
  if (threadIdx.x == 0) ep_barrier_body(peer_flags, N, rank, epoch, timeout_ns, status);
}

// All ranks' barriers in one launch on one device: block r runs rank r's barrier
// (the blocks are co-resident: a cooperative launch).  Ranks set in `absent`
// skip theirs, which makes the others' waits run out.
__global__ void ep_barrier_ranks_kernel(uint32_t* const* peer_flags, int N, uint32_t epoch, uint64_t timeout_ns,
                                        uint64_t absent, int32_t* status) {
  const int rank = blockIdx.x;
  if (threadIdx.x == 0 && !((absent >> rank) & 1)) ep_barrier_body(peer_flags, N, rank, epoch, timeout_ns, status);
}

int grid_for(int64_t items, int per_block) {
  int64_t b = (items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(dev_info().sms) * 8;
  if (b > cap) b = cap;
  return b < 1 ? 1 : static_cast<int>(b);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int ep_shape(int T, int K, int E, int N) {
  if (T < 0 || K <= 0 || K > kMaxK || E <= 0 || N <= 0 || E % N != 0 || K > E) return MM_MOE_ERR_INVALID_ARG;
  return MM_MOE_OK;
}

}  // namespace
}  // namespace mm

using namespace mm;

extern "C" {

int mm_moe_ep_count(const int32_t* topk_idx, int T, int K, int E, int32_t* counts, void* stream) {
  if (T < 0 || K <= 0 || E <= 0 || !counts || (T > 0 && !topk_idx)) return MM_MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess) return MM_MOE_ERR_CUDA;
  const int64_t n = static_cast<int64_t>(T) * K;
  if (n > 0) ep_count_kernel<<<grid_for(n, 256), 256, 0, s>>>(topk_idx, n, E, counts);
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_plan(const int32_t* counts_all, const int32_t* topk_idx, int T, int K, int E, int N, int rank,
                   int32_t* send_row, int64_t* recv_rows, int32_t* recv_expert, int64_t recv_capacity) {
  if (ep_shape(T, K, E, N) || rank < 0 || rank >= N || !counts_all || !recv_rows || (T > 0 && (!topk_idx || !send_row)))
    return MM_MOE_ERR_INVALID_ARG;
  const int Eloc = E / N;
  // this rank's own counts must be the ones it published
  std::vector<int64_t> own(E, 0);
  for (int64_t i = 0; i < static_cast<int64_t>(T) * K; ++i) {
    const int e = topk_idx[i];
    if (e >= 0 && e < E) ++own[e];
  }
  for (int e = 0; e < E; ++e)
    if (counts_all[static_cast<int64_t>(rank) * E + e] != own[e] || own[e] < 0) return MM_MOE_ERR_INVALID_ARG;
  for (int64_t i = 0; i < static_cast<int64_t>(N) * E; ++i)
    if (counts_all[i] < 0) return MM_MOE_ERR_INVALID_ARG;
  // base[e]: the first row of this rank's pairs with expert e at e's owner.  On owner
  // o the rows run by local expert, then source rank, then the source's pairs.
  std::vector<int64_t> base(E, 0);
  for (int o = 0; o < N; ++o) {
    int64_t row = 0;
    for (int e = o * Eloc; e < (o + 1) * Eloc; ++e) {
      for (int r = 0; r < N; ++r) {
        if (r == rank) base[e] = row;
        row += counts_all[static_cast<int64_t>(r) * E + e];
      }
    }
    if (o == rank) {
      if (row > (int64_t(1) << 31) - 1) return MM_MOE_ERR_INVALID_ARG;
      *recv_rows = row;
    }
  }
  if (recv_expert) {
    if (recv_capacity < *recv_rows) return MM_MOE_ERR_INVALID_ARG;
    int64_t row = 0;
    for (int e = rank * Eloc; e < (rank + 1) * Eloc; ++e) {
      int64_t n = 0;
      for (int r = 0; r < N; ++r) n += counts_all[static_cast<int64_t>(r) * E + e];
      for (int64_t i = 0; i < n; ++i) recv_expert[row++] = e - rank * Eloc;
    }
  }
  // this rank's pairs in ascending (token, slot) take consecutive rows from base[e]
  std::vector<int64_t> next(base);
  for (int64_t i = 0; i < static_cast<int64_t>(T) * K; ++i) {
    const int e = topk_idx[i];
    send_row[i] = (e >= 0 && e < E) ? static_cast<int32_t>(next[e]++) : -1;
  }
  return MM_MOE_OK;
}

int mm_moe_ep_push_meta(const int32_t* topk_idx, const float* topk_w, const int32_t* send_row, int T, int K,
                        int E, int N, int rank, void* const* peer_meta, void* stream) {
  if (ep_shape(T, K, E, N) || rank < 0 || rank >= N || !peer_meta) return MM_MOE_ERR_INVALID_ARG;
  if (T == 0) return MM_MOE_OK;
  if (!topk_idx || !topk_w || !send_row) return MM_MOE_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(T) * K;
  ep_push_meta_kernel<<<grid_for(n, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      topk_idx, topk_w, send_row, n, E, E / N, rank, peer_meta);
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_pull(const int32_t* meta, int64_t rows, int K, int H, int variant, const void* const* peer_x,
                   const void* const* peer_x_sf, void* x_recv, void* x_sf_recv, int32_t* topk_idx_recv,
                   float* topk_w_recv, void* stream) {
  if (rows < 0 || K <= 0 || K > kMaxK || H <= 0 || H % 128) return MM_MOE_ERR_INVALID_ARG;
  if (variant != MM_MOE_VARIANT_MX && variant != MM_MOE_VARIANT_F8) return MM_MOE_ERR_INVALID_ARG;
  if (rows == 0) return MM_MOE_OK;
  if (!meta || !peer_x || !peer_x_sf || !x_recv || !x_sf_recv || !topk_idx_recv || !topk_w_recv)
    return MM_MOE_ERR_INVALID_ARG;
  if (!aligned16(meta) || !aligned16(x_recv) || (reinterpret_cast<uintptr_t>(x_sf_recv) & 3))
    return MM_MOE_ERR_INVALID_ARG;
  const int sf_bytes = variant == MM_MOE_VARIANT_MX ? H / 32 : (H / 128) * 4;
  ep_pull_kernel<<<grid_for(rows, 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const int4*>(meta), rows, K, H, sf_bytes, peer_x, peer_x_sf, static_cast<uint8_t*>(x_recv),
      static_cast<uint8_t*>(x_sf_recv), topk_idx_recv, topk_w_recv);
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_combine(const int32_t* topk_idx, const int32_t* send_row, int T, int K, int E, int N, int H,
                      const void* const* peer_out, void* out, void* stream) {
  if (ep_shape(T, K, E, N) || H <= 0 || H % 128 || !peer_out) return MM_MOE_ERR_INVALID_ARG;
  if (T == 0) return MM_MOE_OK;
  if (!topk_idx || !send_row || !out || !aligned16(out)) return MM_MOE_ERR_INVALID_ARG;
  const int64_t warps = static_cast<int64_t>(T) * ((H / 8 + 127) / 128);
  ep_combine_kernel<<<grid_for(warps, 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      topk_idx, send_row, T, K, E, E / N, H, peer_out, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_push_out(const int32_t* meta, int64_t rows, int H, const void* out_recv,
                       void* const* peer_partials, void* stream) {
  if (rows < 0 || H <= 0 || H % 128) return MM_MOE_ERR_INVALID_ARG;
  if (rows == 0) return MM_MOE_OK;
  if (!meta || !out_recv || !peer_partials || !aligned16(meta) || !aligned16(out_recv)) return MM_MOE_ERR_INVALID_ARG;
  ep_push_out_kernel<<<grid_for(rows, 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const int4*>(meta), rows, H, static_cast<const __nv_bfloat16*>(out_recv), peer_partials);
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_combine_local(const int32_t* topk_idx, int T, int K, int E, int H, const void* partials,
                            void* out, void* stream) {
  if (T < 0 || K <= 0 || K > kMaxK || E <= 0 || H <= 0 || H % 128) return MM_MOE_ERR_INVALID_ARG;
  if (T == 0) return MM_MOE_OK;
  if (!topk_idx || !partials || !out || !aligned16(partials) || !aligned16(out)) return MM_MOE_ERR_INVALID_ARG;
  const int64_t warps = static_cast<int64_t>(T) * ((H / 8 + kCombinePart - 1) / kCombinePart);
  ep_combine_local_kernel<<<grid_for(warps, 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      topk_idx, T, K, E, H, static_cast<const __nv_bfloat16*>(partials), static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_recv_capacity(int num_tokens_bound, int K, int E, int N, int64_t* rows) {
  if (!rows || num_tokens_bound < 0 || ep_shape(0, K, E, N)) return MM_MOE_ERR_INVALID_ARG;
  const int per = K < E / N ? K : E / N;
  *rows = static_cast<int64_t>(N) * num_tokens_bound * per;
  return MM_MOE_OK;
}

int mm_moe_ep_barrier(void* const* peer_flags, int N, int rank, uint32_t epoch, unsigned timeout_ms, int32_t* status,
                      void* stream) {
  if (!peer_flags || !status || N <= 0 || N > 64 || rank < 0 || rank >= N) return MM_MOE_ERR_INVALID_ARG;
  const uint64_t ns = static_cast<uint64_t>(timeout_ms ? timeout_ms : 2000) * 1000000ull;
  ep_barrier_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<uint32_t* const*>(peer_flags), N, rank, epoch, ns, status);
  return cudaGetLastError() == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_ep_barrier_ranks(void* const* peer_flags, int N, uint32_t epoch, unsigned timeout_ms, uint64_t absent,
                            int32_t* status, void* stream) {
  if (!peer_flags || !status || N <= 0 || N > 64) return MM_MOE_ERR_INVALID_ARG;
  int coop = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop || N > dev_info().sms)
    return MM_MOE_ERR_UNSUPPORTED;
  const uint64_t ns = static_cast<uint64_t>(timeout_ms ? timeout_ms : 2000) * 1000000ull;
  uint32_t* const* flags = reinterpret_cast<uint32_t* const*>(peer_flags);
  void* kargs[] = {const_cast<uint32_t* const**>(&flags), &N, &epoch, const_cast<uint64_t*>(&ns), &absent, &status};
  const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(ep_barrier_ranks_kernel), dim3(N),
                                                    dim3(32), kargs, 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

}  // extern "C"

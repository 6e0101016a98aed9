// The top-k combine, shared by the combine kernel and the fused stream's early
// combine so that both give the same bits: out[t, h] = bf16_rn(sum over valid
// k, in k order, of part[k][t][h]), the sum in fp32 ("07 · MegaMoE" §9: the
// router weight was applied in the SwiGLU, so the combine is a plain sum).
// PartT: float, or bf16 when the L2 epilogue cast its partials (widened
// exactly).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace mm {

// acc[0..8) += part values p[0..8)
template <typename PartT>
__device__ __forceinline__ void add_partials8(const PartT* __restrict__ p, float (&acc)[8]) {
  if constexpr (sizeof(PartT) == 4) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p)), b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  } else {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // bf16 -> fp32 is exact: the bits move up 16 places
      acc[2 * i] += __uint_as_float(w[i] << 16);
      acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// out[0..8) = bf16_rn(acc[0..8))
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* __restrict__ out, const float (&acc)[8]) {
  uint4 o;
  __nv_bfloat162 v0 = __floats2bfloat162_rn(acc[0], acc[1]);
  __nv_bfloat162 v1 = __floats2bfloat162_rn(acc[2], acc[3]);
  __nv_bfloat162 v2 = __floats2bfloat162_rn(acc[4], acc[5]);
  __nv_bfloat162 v3 = __floats2bfloat162_rn(acc[6], acc[7]);
  o.x = *reinterpret_cast<uint32_t*>(&v0);
  o.y = *reinterpret_cast<uint32_t*>(&v1);
  o.z = *reinterpret_cast<uint32_t*>(&v2);
  o.w = *reinterpret_cast<uint32_t*>(&v3);
  *reinterpret_cast<uint4*>(out) = o;
}

// One thread, 8 consecutive columns h..h+8 of token t; valid(k) tells whether slot k counts.
template <typename PartT, typename Valid>
__device__ __forceinline__ void combine8(const PartT* __restrict__ part, int64_t t, int h, int T, int H, int K,
                                         Valid valid, __nv_bfloat16* __restrict__ out) {
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int k = 0; k < K; ++k)
    if (valid(k)) add_partials8(part + ((static_cast<int64_t>(k) * T + t) * H + h), acc);
  store_bf16x8(out + t * H + h, acc);
}

// One warp, all of token t: lane l takes the 8-column groups l, l + 32, ...,
// kU of them per step, so every slot's loads of a step are kU x 32 bytes a
// lane in flight at once.  Bit k of vmask marks slot k valid.  Each element
// gets the same fp32 additions in the same k order as in combine8.
template <typename PartT, int kU>
__device__ __forceinline__ void combine_token_warp(const PartT* __restrict__ part, int64_t t, int T, int H, int K,
                                                   uint32_t vmask, __nv_bfloat16* __restrict__ out, int lane) {
  const int G = H / 8;
  for (int g0 = lane; g0 < G; g0 += 32 * kU) {
    float acc[kU][8];
#pragma unroll
    for (int u = 0; u < kU; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
    for (int k = 0; k < K; ++k) {
      if (!((vmask >> k) & 1u)) continue;
      const PartT* base = part + (static_cast<int64_t>(k) * T + t) * H;
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (g0 + 32 * u < G) add_partials8(base + 8 * (g0 + 32 * u), acc[u]);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (g0 + 32 * u < G) store_bf16x8(out + t * H + 8 * (g0 + 32 * u), acc[u]);
  }
}

}  // namespace mm

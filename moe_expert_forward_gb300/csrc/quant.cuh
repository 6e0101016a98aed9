// FP8 quantisation of bf16 activation rows inside the gather.  The pages'
// layer takes x already in FP8 with its scales (llm-infra-atlas "07 · MegaMoE"
// §3: the buffer's input region holds x and x_sf), so a caller holding bf16
// activations runs a quantisation pass first; here the gather warps may
// instead quantise bf16 rows on the way into the pool.
//   MX: e4m3 codes with one UE8M0 scale per 32 elements, the scale the
//       smallest power of two 2^e with 448 * 2^e >= max(amax, 1e-10) and the
//       codes RNE_e4m3(x * 2^-e) (the same rule as the intermediate requant).
//   F8: e4m3 codes with one fp32 scale s = max(amax, 1e-10) / 448 per 128
//       elements (IEEE division) and the codes RNE_e4m3(x / s).
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mm {

// Smallest e with 448 * 2^e >= max(amax, 1e-10), read exactly from the fp32
// bit pattern: amax = m * 2^ex with m in [0.5, 1), and 448 = 0.875 * 2^9, so
// e = ex - 9 when m <= 0.875 (mantissa field <= 0x600000), else ex - 8.
// Clamped to [-127, 126]; amax >= 1e-10 keeps e >= -42.
__device__ __forceinline__ int ue8m0_exponent_e4m3(float amax) {
  const uint32_t bits = __float_as_uint(fmaxf(amax, 1e-10f));
  const int ex = static_cast<int>((bits >> 23) & 0xFF) - 126;
  const int e = ex - 9 + ((bits & 0x7FFFFF) > 0x600000 ? 1 : 0);
  return e < -127 ? -127 : (e > 126 ? 126 : e);
}

// 2^-e as an fp32 (e in [-127, 126]).
__device__ __forceinline__ float exp2_neg(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

// The 32 bf16 values of four 16-byte words, as fp32 (exact).
__device__ __forceinline__ void unpack_bf16x32(const uint4 (&v)[4], float (&f)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
      f[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// 32 e4m3 codes of f * scale (RNE, saturating), as two 16-byte words.
__device__ __forceinline__ void pack_e4m3x32(const float (&f)[32], float scale, uint4 (&c)[2]) {
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    p[i] = static_cast<uint32_t>(cvt_e4m3x2(f[4 * i] * scale, f[4 * i + 1] * scale)) |
           (static_cast<uint32_t>(cvt_e4m3x2(f[4 * i + 2] * scale, f[4 * i + 3] * scale)) << 16);
  c[0] = make_uint4(p[0], p[1], p[2], p[3]);
  c[1] = make_uint4(p[4], p[5], p[6], p[7]);
}

// Rows are taken in 32-element chunks, one chunk per lane and step, and two
// steps' loads (eight 16-byte words a lane) are issued before any arithmetic,
// so a warp keeps 4 KB of the row in flight.  Each quantised chunk goes to
// sink(chunk, codes, scale, lead): the fused gather writes it to one pool row,
// the token-major gather to each pool row of the token.
constexpr int kQuantSteps = 2;

// One warp quantises one bf16 row of H elements (H a multiple of 32) to MX
// codes.  A chunk is a 32-element block, so its amax is thread-local;
// sink(j, codes, ue8m0_byte, true) receives block j.
template <typename Sink>
__device__ __forceinline__ void quant_row_mx_bf16(const __nv_bfloat16* __restrict__ src, int H, int lane, Sink sink) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  const int nb = H / 32;
  for (int j0 = 0; j0 < nb; j0 += 32 * kQuantSteps) {
    uint4 v[kQuantSteps][4];
#pragma unroll
    for (int u = 0; u < kQuantSteps; ++u) {
      const int j = j0 + 32 * u + lane;
#pragma unroll
      for (int q = 0; q < 4; ++q) v[u][q] = j < nb ? __ldg(s4 + 4 * j + q) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantSteps; ++u) {
      const int j = j0 + 32 * u + lane;
      if (j < nb) {
        float f[32];
        unpack_bf16x32(v[u], f);
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(f[i]));
        const int e = ue8m0_exponent_e4m3(am);
        uint4 c[2];
        pack_e4m3x32(f, exp2_neg(e), c);
        sink(j, c, static_cast<uint8_t>(e + 127), true);
      }
    }
  }
}

// One warp quantises one bf16 row of H elements (H a multiple of 128) to F8
// codes.  The four lanes holding the chunks of a 128-element block exchange
// their amax by shuffles (all 32 lanes take every step, so the shuffles see
// converged lanes); sink(c, codes, s, lead) receives chunk c with its block's
// scale s, lead on the block's first lane.
template <typename Sink>
__device__ __forceinline__ void quant_row_f8_bf16(const __nv_bfloat16* __restrict__ src, int H, int lane, Sink sink) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  const int nc = H / 32;
  for (int c0 = 0; c0 < nc; c0 += 32 * kQuantSteps) {
    uint4 v[kQuantSteps][4];
#pragma unroll
    for (int u = 0; u < kQuantSteps; ++u) {
      const int c = c0 + 32 * u + lane;
#pragma unroll
      for (int q = 0; q < 4; ++q) v[u][q] = c < nc ? __ldg(s4 + 4 * c + q) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantSteps; ++u) {
      const int c = c0 + 32 * u + lane;   // whole 4-lane groups are in or out: nc is a multiple of 4
      float f[32];
      unpack_bf16x32(v[u], f);
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(f[i]));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      if (c < nc) {
        const float s = __fdiv_rn(fmaxf(am, 1e-10f), 448.0f);
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __fdiv_rn(f[i], s);
        uint4 cd[2];
        pack_e4m3x32(f, 1.0f, cd);
        sink(c, cd, s, (lane & 3) == 0);
      }
    }
  }
}

}  // namespace mm

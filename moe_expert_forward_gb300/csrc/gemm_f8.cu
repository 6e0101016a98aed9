// Grouped GEMMs of the FP8 x FP8 variant on tcgen05 (kind::f8f6f4): e4m3
// activations with one fp32 scale per 1x128, e4m3 weights with one fp32 scale
// per 128x128 block, intermediate requantised per 128 or per 64 with the raw
// scale amax/448 (DeepGEMM PR #440, "Why the order and not the pool size" and
// "Ring sizing, recycling, and why that granularity"; MEGAMOE_SM90_DESIGN.md
// §10.1).
//
// fp32 scales cannot ride the MMA, so each promotion unit (a 128-K block, or a
// 64-K half of one when L2 reads a per-64 intermediate: the design doc's
// dual-half scaling, §5.4) is multiplied into a fresh TMEM partial and the
// epilogue promotes it: acc += partial * sx[row,unit] * sw[rows,kb] (the
// design doc's register-side scale application, §5.3).
// Tile: 128 pool rows x 256 weight rows (L1: 128 gate + 128 up rows).
//
// One CTA per SM, 512 threads in four warpgroups:
//   WG0 (warps 0..3)   TMA producers, warp p owns pipeline stage p
//   WG1, WG2 (4..11)   epilogue: two warps per TMEM lane quadrant, each thread
//                      one pool row and 128 fp32 running sums in registers
//                      (L1: gate and up columns of the same 64 intermediate
//                      columns, so SwiGLU stays thread-local)
//   WG3 (warps 12..15) warps 12 and 13: one MMA-issuing thread each, taking
//                      alternate promotion units (warp 12 also allocates TMEM);
//                      warp 14: waits for each unit's partial and passes it on
//
// While the tensor core streams its operands, every shared-memory access of
// another warp (an mbarrier wait included) takes hundreds of cycles.  So the
// epilogue learns that a unit's partial is complete through a named barrier
// (barriers 1, 2), which touches no shared memory: warp 14 waits on the unit's
// commit and arrives, the eight epilogue warps sync.  The release of a buffer
// back to its issuer stays an mbarrier, whose wait is bounded: a named barrier
// between two single-warp parties cannot be made safe on the abort path (one
// side running two phases ahead completes a phase without the other).  The
// activation and weight scales of a unit reach registers a group of units ahead.
// setmaxnreg moves registers from WG0/WG3 (40 each) to WG1/WG2 (216 each);
// the host refuses to launch unless the kernel was built with exactly 128
// registers per thread, the total the split assumes.
// TMEM: two 256-column partial buffers, one per issuing thread, so the MMAs of
// block kb+1 overlap the promotion of block kb.  Every wait is bounded.
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"

namespace mm {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 512;
constexpr int kLaunchRegs = 128;       // 65536 / 512
constexpr int kSmallRegs = 40;         // producers
constexpr int kMmaRegs = 40;           // MMA warpgroup
constexpr int kEpiRegs = 216;          // epilogue warpgroups
static_assert(128 * kSmallRegs + 128 * kMmaRegs + 2 * 128 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kBN = 256;
constexpr int kTokBytes = kBT * kBK;
constexpr int kWgtBytes = kBN * kBK;
constexpr int kTmemCols = 512;
constexpr int kEpiThreads = 256;       // the two epilogue warpgroups
constexpr int kBarDone0 = 1;           // named barriers 1, 2: the partial of a unit in buffer 0 / 1 is complete
constexpr int kBarThreads = kEpiThreads + 32;   // the epilogue and warp 14

enum : int {
  kSiteEmpty = 201, kSiteFull = 202, kSitePEmpty = 203, kSitePFull = 204, kSiteAmax = 205,
  kSiteDrainCopies = 211, kSiteDrainMma = 212
};

struct Args {
  int T, H, I, E, K;
  int kblocks;
  int nblocks;
  const int* cnt;
  const int* blk_off;
  const int* src;
  const float* topk_w;
  const float* sw;      // weight scales [E, rows/128, kdim/128]
  const float* sx;      // token scales [P, units per row]
  uint8_t* out_codes;   // L1: intermediate codes [P, I]
  float* out_sf;        // L1: intermediate scales [P, I/gran]
  int gran;             // L1: intermediate scale block along I, 128 or 64
  int units;            // promotion units per 128-K stage: 1, or 2 when L2 reads per-64 scales
  int exact_div;        // L1: every requant code from the IEEE quotient (no fast path)
  int unreachable;      // the last stage of this CTA's last task is never loaded (a wait that cannot end)
  float* partials;      // L2: [K, T, H] fp32, or bf16 when pbf16
  int pbf16;
  float clamp;          // gate and up clamped to [-clamp, clamp] before the SwiGLU (+inf: none)
  int precise;          // SwiGLU with expf and the IEEE division (else the fast-math form)
  int* status;
  uint64_t timeout_ns;
  unsigned long long* prof;   // per-CTA role cycles (debug_flags bit 1) or null
};

struct TokenMaps {
  CUtensorMap b32, b64, b128;
};

struct SmemLayout {
  static constexpr int tok = 0;
  static constexpr int wgt = tok + kStages * kTokBytes;
  static constexpr int amax = wgt + kStages * kWgtBytes;              // [2 tasks][2 halves][128] fp32
  static constexpr int meta = amax + 2 * 2 * 128 * 4;
  static constexpr int bars_after_meta(int E) { return meta + ((2 * E + 1) * 4 + 15) / 16 * 16; }
  // full[S], empty[S] (one commit per promotion unit: stage free and partial complete), pempty[2], epi, drain[2]
  static constexpr int nbars = 2 * kStages + 5;
  static constexpr int total(int E) { return bars_after_meta(E) + nbars * 8 + 16; }
};
static_assert(SmemLayout::total(kMaxE) + 1024 <= 232448, "shared memory budget");

__device__ __forceinline__ void decode_tile(int tile, int nblocks, const int* blk_off, const int* cnt, int E,
                                            int& e, int& n, int& b, int& valid) {
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

// kind::f8f6f4 instruction descriptor: fp32 accumulator (bits [5:4] = 1),
// A = B = e4m3 (0), both K-major, N>>3 in [22:17], M>>4 in [28:24].
__device__ __forceinline__ uint32_t make_idesc() {
  return (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) | ((128u >> 4) << 24);
}

// The e4m3 codes RNE_e4m3(fp32(a0 / s)), RNE_e4m3(fp32(a1 / s)) with IEEE
// quotients, r = 1/s correctly rounded.  q = a * r is within 2^-23 |a/s| of the
// exact quotient, so the IEEE quotient lies within 4 fp32 ulps of q; e4m3
// rounding is monotonic, so when q - 4 ulps and q + 4 ulps give the same code,
// that is the code of the IEEE quotient.  Only otherwise (a quotient next to an
// e4m3 rounding boundary) are the divisions done.  exact: always divide.
__device__ __forceinline__ float ulps_toward(float q, int d) {   // |q| moved by d ulps, sign kept, not past 0
  const uint32_t b = __float_as_uint(q);
  const uint32_t m = b & 0x7fffffffu;
  const uint32_t mm = d < 0 ? (m > static_cast<uint32_t>(-d) ? m + d : 0u) : m + d;
  return __uint_as_float((b & 0x80000000u) | mm);
}
__device__ __forceinline__ uint32_t quot_e4m3x2(float a0, float a1, float s, float r, bool exact) {
  if (!exact) {
    const float q0 = a0 * r, q1 = a1 * r;
    const uint16_t lo = cvt_e4m3x2(ulps_toward(q0, -4), ulps_toward(q1, -4));
    const uint16_t hi = cvt_e4m3x2(ulps_toward(q0, 4), ulps_toward(q1, 4));
    if (lo == hi) return lo;
  }
  return cvt_e4m3x2(__fdiv_rn(a0, s), __fdiv_rn(a1, s));
}

__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSmallRegs)); }
__device__ __forceinline__ void regs_dec_mma() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kMmaRegs)); }
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs)); }

// kProf: record per-role SM cycles into args.prof[blockIdx.x * 8 + i]: 0 MMA
// issuer span, 1 its waits for a free partial buffer, 2 its waits for data, 3
// epilogue (warp 4) waits for a partial, 4 promotion, 5 per-task SwiGLU /
// requant / stores, 6 k-blocks, 7 epilogue span; args.prof[4096 + blockIdx.x]:
// the epilogue's per-task setup, [5120 + blockIdx.x] the L1 tail's SwiGLU and
// amax, [6144 + blockIdx.x] its amax rendezvous.  A separate instantiation.
template <int PHASE, bool kProf>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ TokenMaps tmT, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int E = args.E;
  int* s_blk = reinterpret_cast<int*>(smem + SmemLayout::meta);
  int* s_cnt = s_blk + E + 1;
  float* s_amax = reinterpret_cast<float*>(smem + SmemLayout::amax);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmemLayout::bars_after_meta(E));
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* pempty = bars + 2 * kStages;   // [2]: buffer read by all eight epilogue warps
  uint64_t* epibar = pempty + 2;
  uint64_t* drain = epibar + 1;   // [2]: each MMA issuer's last commit
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + SmemLayout::nbars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  const Status st{args.status, args.timeout_ns};
  const int U = args.units;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], U);                  // one commit per promotion unit of the stage
    }
    for (int i = 0; i < 2; ++i) mbar_init(&pempty[i], 8);
    mbar_init(epibar, 256);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp < kStages && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmT.b32);
    prefetch_tmap(&tmT.b64);
    prefetch_tmap(&tmT.b128);
  }
  if (warp == 12) {
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

  if (wg == 0) {
    regs_dec();
    // ------------------------------------------------------------------ TMA producers
    if (lane == 0) {
      const int p = warp;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_t = policy_evict_last();
      uint8_t* tk = smem + SmemLayout::tok + p * kTokBytes;
      uint8_t* wgp = smem + SmemLayout::wgt + p * kWgtBytes;
      int step = 0;
      bool armed = false;                       // a phase of full[p] was armed: its copies land before exit
      uint32_t armed_parity = 0;
      for (int tile = blockIdx.x; tile < total && !*s_abort; tile += gridDim.x) {
        int e, n, b, valid;
        decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
        const CUtensorMap* tt = valid <= 32 ? &tmT.b32 : (valid <= 64 ? &tmT.b64 : &tmT.b128);
        const int rows = valid <= 32 ? 32 : (valid <= 64 ? 64 : 128);
        const uint32_t bytes = rows * kBK + kWgtBytes;
        int kb = ((p - step) % kStages + kStages) % kStages;
        for (; kb < KB; kb += kStages) {
          const uint32_t phase = ((step + kb) / kStages) & 1;
          if (args.unreachable && kb == KB - 1 && tile + static_cast<int>(gridDim.x) >= total) break;
          if (!mbar_wait(&empty[p], phase ^ 1, st, s_abort, kSiteEmpty)) break;
          mbar_arrive_expect_tx(&full[p], bytes);
          armed = true;
          armed_parity = phase;
          const int kc = kb * kBK;
          tma_load_2d(tk, tt, &full[p], kc, b * kBT, pol_t);
          if (PHASE == 1) tma_load_3d(wgp, &tmW, &full[p], kc, e * 2 * args.I + n * 128, 0, pol_w);
          else tma_load_2d(wgp, &tmW, &full[p], kc, e * args.H + n * kBN, pol_w);
        }
        step += KB;
      }
      if (armed) mbar_wait_drain(&full[p], armed_parity, st, kSiteDrainCopies);
    }
  } else if (wg == 3) {
    regs_dec_mma();
    // ------------------------------------------------------------------ MMA issuers
    // Two threads (lane 0 of warps 12, 13) issue alternate promotion units, each
    // into its own partial buffer (unit g: buffer and thread g & 1, stage (g / U) %
    // kStages).  Every unit is a fresh accumulation of 4 / U MMAs, so the order in
    // which the two streams reach the tensor core changes no result.  A unit
    // waits for its stage's data first (that usually landed while the epilogue
    // was still promoting), then for its buffer: the epilogue's release of unit
    // g - 2 (bounded mbarrier waits).  One commit per unit on its stage's empty barrier frees the stage
    // (after all U units) and completes the partial.
    if ((warp == 12 || warp == 13) && lane == 0) {
      const int me = warp - 12;
      int g = 0;                                 // global unit counter
      int stage = 0;                             // stage of the current 128-K step, and its phase
      uint32_t phase = 0;
      bool ok = true;
      const long long c_start = kProf ? clock64() : 0;
      long long c_pe = 0, c_full = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int kb = 0; kb < KB && ok; ++kb) {
          for (int h = 0; h < U; ++h, ++g) {
            if ((g & 1) != me) continue;
            const long long tm0 = kProf ? clock64() : 0;
            if (!mbar_wait(&full[stage], phase, st, s_abort, kSiteFull)) { ok = false; break; }
            const long long tm1 = kProf ? clock64() : 0;
            if (!mbar_wait(&pempty[me], ((g >> 1) & 1) ^ 1, st, s_abort, kSitePEmpty)) { ok = false; break; }
            if (kProf) { c_full += tm1 - tm0; c_pe += clock64() - tm1; }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + SmemLayout::tok + stage * kTokBytes);
            const uint32_t b0 = smem_u32(smem + SmemLayout::wgt + stage * kWgtBytes);
            const uint32_t acc = tmem + me * kBN;
            if (U == 1) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma_f8f6f4(acc, make_smem_desc(a0 + kk * 32, 16, 1024, 2), make_smem_desc(b0 + kk * 32, 16, 1024, 2),
                              make_idesc(), kk != 0);
            } else {                             // the unit's 64-K half: two of the stage's four 32-K slices
              const uint32_t k0 = h * 64;
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                tc_mma_f8f6f4(acc, make_smem_desc(a0 + k0 + kk * 32, 16, 1024, 2),
                              make_smem_desc(b0 + k0 + kk * 32, 16, 1024, 2), make_idesc(), kk != 0);
            }
            tc_commit(&empty[stage]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // every MMA this thread issued has completed before TMEM is freed (its own
      // barrier: the other issuer may still be waiting out a deadline)
      tc_commit(&drain[me]);
      mbar_wait_drain(&drain[me], 0, st, kSiteDrainMma);
      if (kProf && me == 0) {
        args.prof[blockIdx.x * 8 + 0] = clock64() - c_start;
        args.prof[blockIdx.x * 8 + 1] = c_pe;
        args.prof[blockIdx.x * 8 + 2] = c_full;
        args.prof[blockIdx.x * 8 + 6] = g;
      }
    } else if (warp == 14) {
      // Unit g's commit, passed on to the epilogue through barrier kBarDone0 + (g & 1).
      // This warp is at most one unit ahead on each barrier (the partial of unit g + 2
      // needs the epilogue's release of unit g first).  It arrives once for every unit
      // of every task even after a failed wait, so no epilogue warp is ever left at a
      // barrier; the epilogue checks the abort flag after each one.
      bool ok = true;
      int g = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        for (int j = 0; j < KB * U; ++j, ++g) {
          const int sg = g / U;
          if (lane == 0 && ok) ok = mbar_wait(&empty[sg % kStages], (sg / kStages) & 1, st, s_abort, kSitePFull);
          __syncwarp();
          named_arrive(kBarDone0 + (g & 1), kBarThreads);
        }
      }
    }
    __syncwarp();
  } else {
    regs_inc();
    // ------------------------------------------------------------------ epilogue (8 warps)
    const int q = warp & 3;
    const int half = wg - 1;                    // 0 or 1
    const int m = q * 32 + lane;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    // TMEM columns this thread accumulates: L1 gate [64h, 64h+64) and up
    // [128+64h, 128+64h+64); L2 [128h, 128h+128)
    const int c0 = PHASE == 1 ? 64 * half : 128 * half;
    const int c1 = PHASE == 1 ? 128 + 64 * half : 128 * half + 64;
    int g = 0;
    uint32_t ephase = 0;
    const long long e_start = kProf ? clock64() : 0;
    long long e_wait = 0, e_promo = 0, e_tail = 0, e_setup = 0, e_math = 0, e_rdv = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const long long ts0 = kProf ? clock64() : 0;
      int e, n, b, valid;
      decode_tile(tile, args.nblocks, s_blk, s_cnt, E, e, n, b, valid);
      const bool live = m < valid;
      const size_t row = static_cast<size_t>(b) * kBT + m;
      const int s = live ? __ldg(args.src + row) : 0;
      const float w = (PHASE == 1 && live) ? __ldg(args.topk_w + s) : 0.f;
      const int wrows = PHASE == 1 ? 2 * args.I / 128 : args.H / 128;   // weight scale block rows
      // weight scale rows: L1 gate (row n) and up (row I/128 + n) for both halves;
      // L2 this half's 128 columns (row 2n + half, the last row past H)
      const int ra = PHASE == 1 ? n : (2 * n + half < wrows ? 2 * n + half : wrows - 1);
      const int rb = PHASE == 1 ? (args.I >> 7) + n : ra;
      const float* w0g = args.sw + (static_cast<size_t>(e) * wrows + ra) * KB;
      const float* w1g = args.sw + (static_cast<size_t>(e) * wrows + rb) * KB;
      const int NU = KB * U;                     // promotion units of the task
      const float* sxr = args.sx + row * NU;
      float acc0[64], acc1[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) { acc0[j] = 0.f; acc1[j] = 0.f; }
      bool ok = true;
      if (kProf) e_setup += clock64() - ts0;
      auto promote = [&](float sx, float w0, float w1) -> bool {
        const int pb = g & 1;
        const long long tw0 = kProf ? clock64() : 0;
        named_sync(kBarDone0 + pb, kBarThreads);   // warp 14 saw the unit's commit
        if (__any_sync(0xffffffffu, *s_abort != 0)) {   // warp-uniform: the barriers count whole warps
          ++g;                                          // this unit's barrier is passed
          return false;
        }
        const long long tw1 = kProf ? clock64() : 0;
        tc_fence_after();
        const float f0 = sx * w0;
        const float f1 = sx * w1;
        // one 32-column slice at a time keeps at most 128 sums + 32 loaded values
        // live; the buffer is released once its last slice has landed
        const uint32_t tb = tlane + pb * kBN;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc0[j] = fmaf(__uint_as_float(v[j]), f0, acc0[j]);
        tmem_ld_32x32b_x32(tb + c0 + 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc0[32 + j] = fmaf(__uint_as_float(v[j]), f0, acc0[32 + j]);
        tmem_ld_32x32b_x32(tb + c1, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc1[j] = fmaf(__uint_as_float(v[j]), f1, acc1[j]);
        tmem_ld_32x32b_x32(tb + c1 + 32, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[pb]);     // the buffer may take unit g + 2
#pragma unroll
        for (int j = 0; j < 32; ++j) acc1[32 + j] = fmaf(__uint_as_float(v[j]), f1, acc1[32 + j]);
        if (kProf) { e_wait += tw1 - tw0; e_promo += clock64() - tw1; }
        ++g;
        return true;
      };
      // Scale operands (row scale, gate / up or column-block weight scale) reach
      // registers a group of four units ahead of their promotions.  Every load
      // instruction of these warps waits behind the TMEM traffic, so when the
      // task's units come in fours (the rows then 16-byte aligned) one vector load
      // per operand serves the group; otherwise four scalar loads do.
      const bool vec = (NU & 3) == 0;
      auto load4 = [&](int q, float4& s4, float4& a4, float4& b4) {
        if (vec) {
          s4 = live ? __ldg(reinterpret_cast<const float4*>(sxr) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
          if (U == 1) {
            a4 = __ldg(reinterpret_cast<const float4*>(w0g) + q);
            b4 = __ldg(reinterpret_cast<const float4*>(w1g) + q);
          } else {                               // units 4q .. 4q+3 take weight k-blocks 2q, 2q, 2q+1, 2q+1
            const float2 a2 = __ldg(reinterpret_cast<const float2*>(w0g) + q);
            const float2 b2 = __ldg(reinterpret_cast<const float2*>(w1g) + q);
            a4 = make_float4(a2.x, a2.x, a2.y, a2.y);
            b4 = make_float4(b2.x, b2.x, b2.y, b2.y);
          }
        } else {
          float sv[4], av[4], bv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int u = 4 * q + i < NU ? 4 * q + i : NU - 1;
            sv[i] = live ? __ldg(sxr + u) : 0.f;
            av[i] = __ldg(w0g + u / U);
            bv[i] = __ldg(w1g + u / U);
          }
          s4 = make_float4(sv[0], sv[1], sv[2], sv[3]);
          a4 = make_float4(av[0], av[1], av[2], av[3]);
          b4 = make_float4(bv[0], bv[1], bv[2], bv[3]);
        }
      };
      float4 s4, a4, b4;
      float4 ns4 = make_float4(0.f, 0.f, 0.f, 0.f), na4 = ns4, nb4 = ns4;
      load4(0, s4, a4, b4);
      for (int u = 0; u < NU; ++u) {
        const int i = u & 3;
        if (i == 0 && u + 4 < NU) load4((u >> 2) + 1, ns4, na4, nb4);
        const float sx = i == 0 ? s4.x : (i == 1 ? s4.y : (i == 2 ? s4.z : s4.w));
        const float w0 = i == 0 ? a4.x : (i == 1 ? a4.y : (i == 2 ? a4.z : a4.w));
        const float w1 = i == 0 ? b4.x : (i == 1 ? b4.y : (i == 2 ? b4.z : b4.w));
        if (!promote(sx, w0, w1)) { ok = false; break; }
        if (i == 3) {                            // the next group, loaded four promotions ago
          s4 = ns4;
          a4 = na4;
          b4 = nb4;
        }
      }
      if (!ok) break;
      const long long tw2 = kProf ? clock64() : 0;
      if (PHASE == 1) {
        // a = silu(gate) * up * w over this thread's 64 intermediate columns
        if (args.clamp < INFINITY) {   // the optional activation clamp, a pass of its own
          const float c = args.clamp;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            acc0[j] = fminf(fmaxf(acc0[j], -c), c);
            acc1[j] = fminf(fmaxf(acc1[j], -c), c);
          }
        }
        float amax = 0.f;
        if (args.precise) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            acc0[j] = silu_precise(acc0[j]) * acc1[j] * w;
            amax = fmaxf(amax, fabsf(acc0[j]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            acc0[j] = silu_fast(acc0[j]) * acc1[j] * w;
            amax = fmaxf(amax, fabsf(acc0[j]));
          }
        }
        const long long tr0 = kProf ? clock64() : 0;
        if (args.gran == 128) {
          // the 128-column requant block spans both halves: exchange row amax
          // one rendezvous per task: the exchange buffer alternates between tasks, and a
          // thread writes it again two tasks later only after everyone passed the next rendezvous
          float* xa = s_amax + (ephase & 1) * 256;
          xa[half * 128 + m] = amax;
          mbar_arrive(epibar);
          if (!__all_sync(0xffffffffu, mbar_wait(epibar, ephase, st, s_abort, kSiteAmax))) break;
          ephase ^= 1;
          amax = fmaxf(amax, xa[(half ^ 1) * 128 + m]);
        }   // per 64: this thread's 64 columns are the block
        if (kProf) { e_math += tr0 - tw2; e_rdv += clock64() - tr0; }
        if (live) {
          // s = amax / 448 and each code RNE_e4m3(a / s), both quotients IEEE-rounded
          // (DeepGEMM PR #440: the scale is the raw amax / 448 and the value is divided by it)
          const float sf = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
          const float rsf = __frcp_rn(sf);
          const bool exact = args.exact_div != 0;
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t lo = quot_e4m3x2(acc0[4 * i], acc0[4 * i + 1], sf, rsf, exact);
            const uint32_t hi = quot_e4m3x2(acc0[4 * i + 2], acc0[4 * i + 3], sf, rsf, exact);
            packed[i] = lo | (hi << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(args.out_codes + row * args.I + n * 128 + 64 * half);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
          if (args.gran == 64) args.out_sf[row * (args.I / 64) + 2 * n + half] = sf;
          else if (half == 0) args.out_sf[row * (args.I / 128) + n] = sf;
        }
      } else {
        if (live && n * kBN + 128 * half < args.H) {
          const int t = s / args.K;
          const int k = s - t * args.K;
          const size_t off = (static_cast<size_t>(k) * args.T + t) * args.H + n * kBN + 128 * half;
          if (args.pbf16) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.partials) + off;
            st_bf16x32(dst, acc0);
            st_bf16x32(dst + 32, acc0 + 32);
            st_bf16x32(dst + 64, acc1);
            st_bf16x32(dst + 96, acc1 + 32);
          } else {
            float* dst = args.partials + off;
            // 32-byte stores: half the store instructions of float4
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              st_global_v8(dst + 8 * i, acc0 + 8 * i);
              st_global_v8(dst + 64 + 8 * i, acc1 + 8 * i);
            }
          }
        }
      }
      if (kProf) e_tail += clock64() - tw2;
    }
    // After an abort every epilogue warp still syncs the "unit complete" barrier of
    // each remaining unit (warp 14 arrives for every unit, so the syncs return at
    // once): warps that saw the flag at different units all reach the same total,
    // so none is left waiting for another.
    __syncwarp();
    {
      const int ntasks = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
      for (const int units = ntasks * KB * U; g < units; ++g) named_sync(kBarDone0 + (g & 1), kBarThreads);
    }
    if (kProf && warp == 4 && lane == 0) {
      args.prof[blockIdx.x * 8 + 3] = e_wait;
      args.prof[blockIdx.x * 8 + 4] = e_promo;
      args.prof[blockIdx.x * 8 + 5] = e_tail;
      args.prof[blockIdx.x * 8 + 7] = clock64() - e_start;
      args.prof[4096 + blockIdx.x] = e_setup;   // inside this phase's 8192-entry region
      args.prof[4096 + 1024 + blockIdx.x] = e_math;
      args.prof[4096 + 2048 + blockIdx.x] = e_rdv;
    }
  }

  // the producers and the MMA issuer have waited for the async work they issued
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int PHASE>
cudaError_t launch_impl(const GemmLaunchF8& g, cudaStream_t s) {
  const Layout& L = *g.L;
  const WsPtrs& W = *g.W;
  const bool prof = g.prof != nullptr;
  auto kernel = prof ? gemm_f8_kernel<PHASE, true> : gemm_f8_kernel<PHASE, false>;
  // The register split assumes the kernel starts with exactly kLaunchRegs per thread.
  if (cudaError_t e = configure_kernel(reinterpret_cast<const void*>(kernel), kLaunchRegs,
                                       SmemLayout::total(kMaxE) + 1024))
    return e;
  CUtensorMap tmW;
  TokenMaps tmT;
  Args a{};
  a.T = L.T; a.H = L.H; a.I = L.I; a.E = L.E; a.K = L.K;
  a.cnt = W.cnt; a.blk_off = W.blk_off; a.src = W.src; a.topk_w = g.topk_w;
  a.status = W.status; a.timeout_ns = g.timeout_ns;
  a.prof = g.prof ? g.prof + (PHASE == 2 ? 8 * 1024 : 0) : nullptr;
  a.sw = g.wsf;
  a.clamp = g.clamp;   // both phases: L1 applies it, L2 ignores it
  a.precise = g.precise;
  a.gran = L.act_gran;
  a.exact_div = g.exact_div ? 1 : 0;
  a.unreachable = (PHASE == 1 && g.unreachable) ? 1 : 0;
  const uint8_t* pool;
  int kdim;
  if (PHASE == 1) {
    a.kblocks = L.H / 128;
    a.nblocks = L.I / 128;
    a.units = 1;
    a.sx = reinterpret_cast<const float*>(W.pool_x_sf);
    a.out_codes = W.pool2;
    a.out_sf = reinterpret_cast<float*>(W.pool2_sf);
    const uint64_t dims[3] = {static_cast<uint64_t>(L.H), static_cast<uint64_t>(L.E) * 2 * L.I - L.I, 2};
    const uint64_t strides[2] = {static_cast<uint64_t>(L.H), static_cast<uint64_t>(L.I) * L.H};
    const uint32_t box[3] = {128, 128, 2};
    if (encode_tmap(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    pool = W.pool_x;
    kdim = L.H;
  } else {
    a.kblocks = L.I / 128;
    a.nblocks = (L.H + kBN - 1) / kBN;
    a.units = L.act_gran == 64 ? 2 : 1;
    a.sx = reinterpret_cast<const float*>(W.pool2_sf);
    a.partials = W.part;
    a.pbf16 = L.part_elem == 2;
    if (encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w, L.I, static_cast<uint64_t>(L.E) * L.H, L.I, 128,
                       kBN, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    pool = W.pool2;
    kdim = L.I;
  }
  CUtensorMap* maps[3] = {&tmT.b32, &tmT.b64, &tmT.b128};
  for (int i = 0; i < 3; ++i)
    if (encode_tmap_2d(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, pool, kdim, L.P, kdim, 128, 32u << i,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  kernel<<<g.grid, kThreads, SmemLayout::total(L.E) + 1024, s>>>(tmW, tmT, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_f8_l1(const GemmLaunchF8& g, cudaStream_t s) { return launch_impl<1>(g, s); }
cudaError_t launch_gemm_f8_l2(const GemmLaunchF8& g, cudaStream_t s) { return launch_impl<2>(g, s); }

}  // namespace mm

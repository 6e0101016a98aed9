// Pieces of the fused task stream shared by both MX GEMM kernels: the gather
// warps that fill the pool, and the early combine of the epilogue warps.
// ArgsT is the kernel's argument struct; the fields used are named below.
#pragma once

#include <cuda_bf16.h>

#include "combine.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "sched.cuh"

namespace mm {

// wait sites of the early combine (reported through the status word)
constexpr int kSiteCombineWait = 109;    // a token's experts have not all finished L2
constexpr int kSiteDeferredWait = 110;   // a deferred entry was never written

// Gather warps of the fused stream: this CTA gathers pool blocks b =
// blockIdx.x, + gridDim.x, ... in order; warp gw of nw copies rows gw, gw + nw,
// ... of a block (codes and UE8M0 scales, or bf16 rows quantised on the way)
// and publishes its row count (release, after a proxy fence: TMA reads the
// rows).  Fields: H, E, K, BT, CPB, x, x_sf, x_bf16, src, pool_x, pool_x_sf,
// ctr_gather.
template <typename ArgsT>
__device__ __forceinline__ void gather_rows(const ArgsT& args, const int* s_blk, const int* s_cnt, const Sched& sch,
                                            volatile int* s_abort, int gw, int nw, int lane, int nblk) {
  const int KBx = args.H / 128;
  const int BT = args.BT;
  for (int b = blockIdx.x; b < nblk && !*s_abort; b += gridDim.x) {
    const int e = sch.largest_leq(s_blk, args.E, b, 1);
    const int rem = s_cnt[e] - (b - s_blk[e]) * BT;
    const int valid = rem < BT ? rem : BT;
    int done = 0;
    for (int r = gw; r < valid; r += nw) {
      const size_t row = static_cast<size_t>(b) * BT + r;
      const int64_t tok = __ldg(args.src + row) / args.K;
      uint4* drow = reinterpret_cast<uint4*>(args.pool_x + row * args.H);
      if (args.x_bf16) {
        const __nv_bfloat16* brow = reinterpret_cast<const __nv_bfloat16*>(args.x) + tok * args.H;
        quant_row_mx_bf16(brow, args.H, lane, [&](int j, const uint4 (&c)[2], uint8_t sfb, bool) {
          drow[2 * j] = c[0];
          drow[2 * j + 1] = c[1];
          args.pool_x_sf[pool_sf_word(b, j >> 2, KBx, args.CPB, r) + (j & 3)] = sfb;
        });
        ++done;
        continue;
      }
      const uint4* srow = reinterpret_cast<const uint4*>(args.x + tok * args.H);
      for (int i = lane; i < args.H / 16; i += 32) drow[i] = __ldg(srow + i);
      const uint32_t* ssf = reinterpret_cast<const uint32_t*>(args.x_sf + tok * (args.H / 32));
      for (int kb = lane; kb < KBx; kb += 32)
        *reinterpret_cast<uint32_t*>(args.pool_x_sf + pool_sf_word(b, kb, KBx, args.CPB, r)) = __ldg(ssf + kb);
      ++done;
    }
    fence_proxy_async_global();
    __syncwarp();
    if (lane == 0 && done) red_release_gpu_add(args.ctr_gather + b, done);
  }
}

// Early combine (DeepGEMM PR #440, "Also in the diff": math warps reduce the
// tokens whose selected experts have all published).  An epilogue warp comes
// here once its CTA has no tile group left, and by then every group of the
// stream has been dealt, so each L2 tile a token waits for belongs to a CTA
// that finishes it without any help from this warp: no wait below can close a
// cycle.  Pass 1 takes tokens in order: a token whose valid slots' experts
// have all finished L2 (per-expert counts of epilogue warps, read with
// acquire) is combined at once by the warp, any other is appended to a
// deferred list.  Pass 2 takes the deferred tokens and waits, bounded, for
// their experts.  The arithmetic is the combine kernel's (combine.cuh).  Every
// branch below is warp-uniform.  Each of an expert's l2_tiles L2 tasks per
// pool block adds one per epilogue warp (epi_warps of them) to ctr_l2[e].
// Fields: T, K, E, H, partials, cmb, topk_idx, ctr_l2, deferred, out.
template <typename PartT, typename ArgsT>
__device__ __forceinline__ void early_combine(const ArgsT& args, int epi_warps, int l2_tiles, const int* s_blk, const Status& st,
                                              volatile int* s_abort, int lane) {
  const int T = args.T, K = args.K, E = args.E;
  const PartT* part = reinterpret_cast<const PartT*>(args.partials);
  int* take = args.cmb;             // pass 1: tokens taken
  int* ndef = args.cmb + 1;         // deferred so far
  int* classified = args.cmb + 2;   // pass-1 tokens combined or deferred
  int* take2 = args.cmb + 3;        // pass 2: deferred entries taken
  auto stop = [&]() { return __shfl_sync(0xffffffffu, *s_abort ? 1 : 0, 0) != 0; };
  auto next = [&](int* ctr) {
    int c = 0;
    if (lane == 0) c = atomicAdd(ctr, 1);
    return __shfl_sync(0xffffffffu, c, 0);
  };
  // lane k < K checks slot k; vmask gets the valid slots
  auto ready = [&](int t, uint32_t& vmask) -> bool {
    bool ok = true, v = false;
    if (lane < K) {
      const int e = __ldg(args.topk_idx + static_cast<int64_t>(t) * K + lane);
      v = e >= 0 && e < E;
      if (v) ok = ld_acquire_gpu(args.ctr_l2 + e) >= epi_warps * l2_tiles * (s_blk[e + 1] - s_blk[e]);
    }
    vmask = __ballot_sync(0xffffffffu, v);
    const bool all = __all_sync(0xffffffffu, ok);
    __syncwarp();   // the checking lanes' acquires before every lane's partial loads
    return all;
  };
  while (!stop()) {
    const int t = next(take);
    if (t >= T) break;
    uint32_t vm;
    if (ready(t, vm)) combine_token_warp<PartT, 4>(part, t, T, args.H, K, vm, args.out, lane);
    else if (lane == 0) st_release_gpu(args.deferred + atomicAdd(ndef, 1), t + 1);
    __syncwarp();
    if (lane == 0) red_release_gpu_add(classified, 1);
  }
  while (!stop()) {
    const int c = next(take2);
    if (c >= T) break;
    int t = -1;   // stays -1 when entry c will never be written (every token classified, fewer deferred)
    if (lane == 0) {
      const uint64_t t0 = globaltimer();
      while (true) {
        const int v = ld_acquire_gpu(args.deferred + c);
        if (v > 0) { t = v - 1; break; }
        if (ld_acquire_gpu(classified) >= T && ld_acquire_gpu(ndef) <= c) break;
        if (*s_abort) break;
        if (globaltimer() - t0 > st.timeout_ns) {
          report_error(st, 4 /*MM_MOE_ERR_TIMEOUT*/, kSiteDeferredWait);
          *s_abort = 1;
          break;
        }
      }
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t < 0) break;
    uint32_t vm;
    const uint64_t t0 = globaltimer();
    bool ok = true;
    while (!ready(t, vm)) {
      int late = 0;
      if (lane == 0) late = (*s_abort || globaltimer() - t0 > st.timeout_ns) ? 1 : 0;
      if (__shfl_sync(0xffffffffu, late, 0)) { ok = false; break; }
    }
    if (!ok) {   // the first error recorded wins, so an abort raised elsewhere keeps its own
      if (lane == 0) {
        report_error(st, 4 /*MM_MOE_ERR_TIMEOUT*/, kSiteCombineWait);
        *s_abort = 1;
      }
      break;
    }
    combine_token_warp<PartT, 4>(part, t, T, args.H, K, vm, args.out, lane);
  }
}


}  // namespace mm

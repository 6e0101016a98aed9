// Internal declarations shared by the host API and the kernel translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mm_moe.h"

namespace mm {

constexpr int kBT = 128;        // tokens per pool block of the token-M kernels (one scale chunk)
constexpr int kBK = 128;        // contraction elements per pipeline stage
constexpr int kSFChunk = 512;   // bytes of one 128-row x 128-K scale chunk (MX)
constexpr int kMaxE = 1024;
constexpr int kMaxK = 16;
constexpr int kSchedCounters = 4;        // tile-group counters after the arrival counters, one per GEMM mode
constexpr int kCombineCounters = 4;      // early combine: tokens taken, deferred, classified, deferred taken

// Byte offsets of every buffer inside the caller's workspace.
struct Layout {
  int T, H, I, E, K, variant, BT;
  int CPB;                   // 128-row scale chunks per pool block: ceil(BT / 128)
  int64_t P;                 // pool row capacity (multiple of BT)
  int64_t nblk_cap;          // P / BT
  int KB1, KB2;              // H/128, I/128
  int part_elem;             // bytes of one partial: 4 (fp32) or 2 (bf16)
  int act_gran;              // F8: intermediate scale block along I (128 or 64); MX: 32
  int S;                     // shared experts (the last S of E and of K; 0 = none)
  int64_t ring;              // intermediate slots (pool blocks) of a wrapping ring; 0 = one per pool block
  size_t ext_idx, ext_w;     // shared experts: the routing extended by S slots, int32 / fp32 [T, K]
  size_t status, cnt, blk_off, dscr, ctr, slot, src, pool_x, pool_x_sf, pool2, pool2_sf, part, dbg, dbg_bytes, prof, total;
};

// E and K count the shared experts: E = routed + S, K = routed slots + S.
Layout make_layout(int T, int H, int I, int E, int K, int variant, int debug_flags = 0, int partials_bf16 = 0,
                   int BT = kBT, int act_gran = 128, int S = 0, int ring = 0);
// The F8 intermediate's scale width by the shape rule of DeepGEMM PR #440 ("Ring
// sizing, recycling, and why that granularity"): 128 when H % 512 == 0 and
// 2I % 512 == 0, else 64.
inline int f8_gran_rule(int H, int I) { return (H % 512 == 0 && (2 * I) % 512 == 0) ? 128 : 64; }

// Byte offset, in a pool scale region laid out [block][kb][CPB chunks][512], of
// the 4-byte word of row r of block b (r < BT) and 128-wide contraction block
// kb: chunk r / 128 of the block, then the tcgen05.cp 32x128b order inside the
// chunk (16-byte line r % 32, word (r % 128) / 32, byte = 32-wide sub-block).
__host__ __device__ __forceinline__ size_t pool_sf_word(int64_t b, int kb, int KB, int CPB, int r) {
  return ((static_cast<size_t>(b) * KB + kb) * CPB + (r >> 7)) * kSFChunk + (r & 31) * 16 + ((r & 127) >> 5) * 4;
}

// Ints of the counter region, zeroed before every forward: [2][nblk_cap]
// per-block arrival counters, kSchedCounters, kCombineCounters, [E] L2
// completions per expert, [T] deferred tokens of the early combine (t + 1),
// [nblk_cap] L2 tiles that have read each block's intermediate (ring reuse).
inline size_t ctr_ints(const Layout& L) {
  return 3 * static_cast<size_t>(L.nblk_cap) + kSchedCounters + kCombineCounters + L.E + L.T;
}

// Device pointers resolved from a workspace.
struct WsPtrs {
  int* status;
  int* cnt;
  int* blk_off;
  int* dscr;
  int* ctr;                  // the counter region (ctr_ints): arrival, tile-group and early-combine counters
  int* slot;
  int* src;
  uint8_t* pool_x;
  uint8_t* pool_x_sf;
  uint8_t* pool2;
  uint8_t* pool2_sf;
  float* part;
  float* dbg;
  unsigned long long* prof;
  int32_t* ext_idx;          // shared experts: extended routing (null without)
  float* ext_w;
};
WsPtrs ws_ptrs(void* ws, const Layout& L);

struct DevInfo {
  int sms;
  int cc_major, cc_minor;
  size_t smem_optin;
};
const DevInfo& dev_info();

// Once per kernel and device (thread-safe): when want_regs > 0, fail with
// cudaErrorInvalidConfiguration unless the kernel was built with exactly that
// many registers a thread (the setmaxnreg splits depend on it); when
// smem_bytes > 0, raise the kernel's dynamic shared-memory limit to it.
cudaError_t configure_kernel(const void* fn, int want_regs, int smem_bytes);
// How many 2-CTA clusters of this kernel (blockDim threads, smem_bytes of dynamic
// shared memory) the current device holds at once; cached per kernel and device.
cudaError_t max_pair_clusters(const void* fn, int threads, int smem_bytes, int* clusters);

// ---- launchers (return cudaError_t of the launch)
cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int K, int E, int block_m, int32_t* cnt,
                            int32_t* blk_off, int32_t* slot, int32_t* src, int32_t* status, int32_t* scratch,
                            int64_t scratch_ints, cudaStream_t s);
constexpr int kDispatchMaxCtas = 256;   // the dispatch scratch holds per-CTA counts [CTAs][E]
// x_bf16: x is bf16 [T, H] and each row is quantised on its way into the pool
cudaError_t launch_gather(const Layout& L, const WsPtrs& W, const uint8_t* x, const void* x_sf, bool x_bf16,
                          cudaStream_t s);
// pdl: programmatic launch after the GEMM (the combine waits for it in-kernel)
cudaError_t launch_combine(const Layout& L, const WsPtrs& W, const int32_t* topk_idx, void* out, bool pdl,
                           cudaStream_t s);
cudaError_t launch_prepare_sf_mx(const uint8_t* w1_sf, const uint8_t* w2_sf, int H, int I, int E,
                                 uint8_t* w1_sfp, uint8_t* w2_sfp, cudaStream_t s);
// topk_idx [T, K] / topk_w -> [T, K + S]: routed slots copied (ids in [E, E+S)
// turned into -2, out of range for the routing kernels), then S slots naming
// experts E .. E+S-1 with weight 1.
cudaError_t launch_extend_routing(const int32_t* topk_idx, const float* topk_w, int T, int K, int E, int S,
                                  int32_t* ext_idx, float* ext_w, cudaStream_t s);
cudaError_t launch_read_intermediate(const Layout& L, const WsPtrs& W, int64_t rows, uint8_t* codes,
                                     void* sf, cudaStream_t s);

struct GemmLaunch {
  const Layout* L;
  const WsPtrs* W;
  const uint8_t* w1;         // e2m1 weights and their prepared scale chunks
  const uint8_t* w1sfp;
  const uint8_t* w2;
  const uint8_t* w2sfp;
  const uint8_t* x;          // activations and scales (in-kernel gather of the fused stream)
  const void* x_sf;
  bool x_bf16;               // x is bf16 [T, H]: the gather quantises (x_sf unused)
  const float* topk_w;
  float* dbg;               // L1 raw accumulators (debug_flags bit 0) or null
  unsigned long long* prof; // per-CTA role timings (debug_flags bit 1) or null
  uint64_t timeout_ns;
  int grid;
  float clamp;              // activation clamp of gate and up (+inf: none)
  int precise;              // SwiGLU with expf and the IEEE division instead of the fast-math form
  bool early_combine;       // fused stream: the epilogue warps combine tokens once their experts are done
  const int32_t* topk_idx;  // early combine: the routing and the bf16 output [T, H]
  void* out;
  bool pdl;                 // programmatic launch after the routing kernel
  bool per_block;           // token-M kernel: deal (weight tile, pool block) pairs as separate groups
  uint8_t* trace;           // token-M kernel: per-task trace records of this launch ([grid][trace_cap] x 64 B) or null
  int trace_cap;            // records per CTA
};
// One per-task trace record (64 bytes; mm_moe.h, Options.trace_buf).
struct TraceRec {
  uint32_t cta, task, type, expert, tile, block, valid, mode;
  uint64_t t_issue, t_mma_done, t_epi_done, reserved;
};
static_assert(sizeof(TraceRec) == 64, "trace record");
// mode 1: L1 tiles, mode 2: L2 tiles, mode 3: gather + lag-ordered L1/L2 stream
cudaError_t launch_gemm_mx(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s);
int mx_lag_auto(int E);
// The same modes with the weights as the MMA's M operand and each pool block's
// tokens as N (gemm_mx_sw.cu); g.L->BT must be a supported block size.
cudaError_t launch_gemm_mx_sw(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s);
bool mx_sw_block_supported(int bt);
// The swapped form on 2-CTA clusters (gemm_mx_pair.cu): M = 256 weight rows per
// tcgen05 cta_group::2 MMA, half of each block's tokens in each CTA.
cudaError_t launch_gemm_mx_pair(const GemmLaunch& g, int mode, int lag, int l1_extra, cudaStream_t s);
bool mx_pair_block_supported(int bt);

struct GemmLaunchF8 {
  const Layout* L;
  const WsPtrs* W;
  const uint8_t* w;          // e4m3 weights (w1 or w2)
  const float* wsf;          // their fp32 128x128 block scales
  const float* topk_w;
  uint64_t timeout_ns;
  int grid;
  unsigned long long* prof;  // per-CTA role cycles (debug_flags bit 1) or null
  float clamp;               // activation clamp of gate and up (+inf: none)
  int precise;               // SwiGLU with expf and the IEEE division instead of the fast-math form
  bool exact_div;            // L1 requant: divide for every code (debug_flags bit 4), not only near a boundary
  bool unreachable;          // L1: the last stage of each CTA's last task is never loaded (debug_flags bit 2)
};
cudaError_t launch_gemm_f8_l1(const GemmLaunchF8& g, cudaStream_t s);
cudaError_t launch_gemm_f8_l2(const GemmLaunchF8& g, cudaStream_t s);

// TMA descriptor creation through the driver entry point.
CUresult encode_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz);
CUresult encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle swz);

}  // namespace mm

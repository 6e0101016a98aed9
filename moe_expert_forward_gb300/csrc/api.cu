// Host side of the C ABI: argument checks, workspace layout, TMA descriptors
// and the launch sequence of one forward.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "internal.h"

namespace mm {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

Layout make_layout(int T, int H, int I, int E, int K, int variant, int debug_flags, int partials_bf16, int BT,
                   int act_gran, int S, int ring) {
  Layout L{};
  L.T = T; L.H = H; L.I = I; L.E = E; L.K = K; L.variant = variant; L.BT = BT; L.S = S;
  L.act_gran = variant == MM_MOE_VARIANT_MX ? 32 : act_gran;
  L.CPB = (BT + 127) / 128;
  const int64_t pairs = static_cast<int64_t>(T) * K;
  const int64_t live_experts = pairs < E ? pairs : E;
  L.P = static_cast<int64_t>(align_up(static_cast<size_t>(pairs + live_experts * (BT - 1)), BT));
  L.nblk_cap = L.P / BT;
  L.KB1 = H / 128;
  L.KB2 = I / 128;
  L.ring = (ring > 0 && ring < L.nblk_cap) ? ring : 0;   // a ring as large as the pool never wraps
  const int64_t islots = L.ring ? L.ring : L.nblk_cap;   // pool blocks the intermediate holds
  size_t o = 0;
  L.status = o; o += 256;
  L.cnt = o; o = align_up(o + sizeof(int) * E, 256);
  L.blk_off = o; o = align_up(o + sizeof(int) * (E + 1), 256);
  L.dscr = o; o = align_up(o + sizeof(int) * static_cast<size_t>(kDispatchMaxCtas) * E, 256);
  L.ctr = o; o = align_up(o + sizeof(int) * ctr_ints(L), 256);
  L.slot = o; o = align_up(o + sizeof(int) * pairs, 256);
  L.src = o; o = align_up(o + sizeof(int) * L.P, 1024);
  L.pool_x = o; o = align_up(o + static_cast<size_t>(L.P) * H, 1024);
  // MX scales: [block][kb][CPB][512-byte chunk]; F8 scales: fp32 [P][H / 128] and [P][I / act_gran]
  const size_t chunks = static_cast<size_t>(L.nblk_cap) * L.CPB * kSFChunk;
  L.pool_x_sf = o;
  o = align_up(o + (variant == MM_MOE_VARIANT_MX ? chunks * (H / 128)
                                                 : static_cast<size_t>(L.P) * (H / 128) * sizeof(float)), 1024);
  L.pool2 = o; o = align_up(o + static_cast<size_t>(islots) * BT * I, 1024);
  L.pool2_sf = o;
  o = align_up(o + (variant == MM_MOE_VARIANT_MX ? static_cast<size_t>(islots) * L.CPB * kSFChunk * (I / 128)
                                                 : static_cast<size_t>(L.P) * (I / L.act_gran) * sizeof(float)), 1024);
  L.part_elem = partials_bf16 ? 2 : 4;
  L.part = o; o = align_up(o + static_cast<size_t>(pairs) * H * L.part_elem, 1024);
  L.dbg = o;
  L.dbg_bytes = (debug_flags & 1) ? static_cast<size_t>(L.P) * 2 * I * sizeof(float) : 0;
  o = align_up(o + L.dbg_bytes, 1024);
  L.prof = o;
  o = align_up(o + ((debug_flags & 2) ? 2 * 8 * 1024 * sizeof(unsigned long long) : 0), 1024);
  L.ext_idx = o;
  o = align_up(o + (S ? sizeof(int32_t) * pairs : 0), 256);
  L.ext_w = o;
  o = align_up(o + (S ? sizeof(float) * pairs : 0), 1024);
  L.total = o;
  return L;
}

WsPtrs ws_ptrs(void* ws, const Layout& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  WsPtrs W;
  W.status = reinterpret_cast<int*>(b + L.status);
  W.cnt = reinterpret_cast<int*>(b + L.cnt);
  W.blk_off = reinterpret_cast<int*>(b + L.blk_off);
  W.dscr = reinterpret_cast<int*>(b + L.dscr);
  W.ctr = reinterpret_cast<int*>(b + L.ctr);
  W.slot = reinterpret_cast<int*>(b + L.slot);
  W.src = reinterpret_cast<int*>(b + L.src);
  W.pool_x = b + L.pool_x;
  W.pool_x_sf = b + L.pool_x_sf;
  W.pool2 = b + L.pool2;
  W.pool2_sf = b + L.pool2_sf;
  W.part = reinterpret_cast<float*>(b + L.part);
  W.dbg = L.dbg_bytes ? reinterpret_cast<float*>(b + L.dbg) : nullptr;
  W.prof = (L.ext_idx > L.prof) ? reinterpret_cast<unsigned long long*>(b + L.prof) : nullptr;
  W.ext_idx = L.S ? reinterpret_cast<int32_t*>(b + L.ext_idx) : nullptr;
  W.ext_w = L.S ? reinterpret_cast<float*>(b + L.ext_w) : nullptr;
  return W;
}

const DevInfo& dev_info() {
  static DevInfo infos[64];
  static bool have[64] = {false};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> g(mu);
  if (!have[dev]) {
    cudaDeviceProp p;
    cudaGetDeviceProperties(&p, dev);
    infos[dev].sms = p.multiProcessorCount;
    infos[dev].cc_major = p.major;
    infos[dev].cc_minor = p.minor;
    infos[dev].smem_optin = p.sharedMemPerBlockOptin;
    have[dev] = true;
  }
  return infos[dev];
}

cudaError_t configure_kernel(const void* fn, int want_regs, int smem_bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> g(mu);
  if (done.count({fn, dev})) return cudaSuccess;
  if (want_regs > 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != want_regs) return cudaErrorInvalidConfiguration;
  }
  if (smem_bytes > 0) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
  }
  done.insert({fn, dev});
  return cudaSuccess;
}

cudaError_t max_pair_clusters(const void* fn, int threads, int smem_bytes, int* clusters) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find({fn, dev});
  if (it != cache.end()) {
    *clusters = it->second;
    return cudaSuccess;
  }
  cudaLaunchConfig_t q = {};
  q.gridDim = dim3(2);
  q.blockDim = dim3(threads);
  q.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute ca;
  ca.id = cudaLaunchAttributeClusterDimension;
  ca.val.clusterDim.x = 2; ca.val.clusterDim.y = 1; ca.val.clusterDim.z = 1;
  q.attrs = &ca;
  q.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fn, &q);
  if (e != cudaSuccess) return e;
  cache[{fn, dev}] = n;
  *clusters = n;
  return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

CUresult encode_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = fn(m, dt, rank, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS && getenv("MM_MOE_DEBUG"))
    fprintf(stderr, "mm_moe: cuTensorMapEncodeTiled(dt=%d rank=%d) = %d\n", static_cast<int>(dt), rank,
            static_cast<int>(r));
  return r;
}

CUresult encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS && getenv("MM_MOE_DEBUG"))
    fprintf(stderr, "mm_moe: cuTensorMapEncodeTiled(dt=%d inner=%llu outer=%llu stride=%llu box=%u x %u) = %d\n",
            static_cast<int>(dt), (unsigned long long)inner, (unsigned long long)outer,
            (unsigned long long)row_stride_bytes, box_inner, box_outer, static_cast<int>(r));
  return r;
}

}  // namespace mm

using namespace mm;

namespace {

mm_moe_options resolve(const mm_moe_options* opt) {
  mm_moe_options o;
  if (opt) o = *opt; else mm_moe_default_options(&o);
  if (o.wait_timeout_ms == 0) o.wait_timeout_ms = 2000;
  return o;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int T, int H, int I, int E, int K, int S = 0) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || K <= 0 || S < 0) return MM_MOE_ERR_INVALID_ARG;
  if (H % 128 || I % 128) return MM_MOE_ERR_INVALID_ARG;
  if (K + S > kMaxK || K > E || E + S > kMaxE) return MM_MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * (K + S) > (int64_t(1) << 30)) return MM_MOE_ERR_INVALID_ARG;
  return MM_MOE_OK;
}

// Which MX kernel runs and its pool block size (tokens per block).
struct Plan {
  bool swap;   // weights as the MMA's M operand, each block's tokens as N
  bool pair;   // ... on 2-CTA clusters (cta_group::2)
  int BT;
};

// expected tokens per expert above which the swapped kernel uses 160-token blocks
constexpr int kSwapLargeBlockTokens = 64;

int make_plan(const mm_moe_options& o, int T, int K, int E, Plan* p) {
  if (o.f8_act_gran != 0 && o.f8_act_gran != -1 && o.f8_act_gran != 64 && o.f8_act_gran != 128)
    return MM_MOE_ERR_INVALID_ARG;
  if (o.ring_blocks < 0) return MM_MOE_ERR_INVALID_ARG;
  if (o.ring_blocks > 0) {
    // the ring exists in the token-M MX kernel's fused stream, which reads each slot after its L1 tiles
    if (o.variant != MM_MOE_VARIANT_MX || !o.fused || o.swap_ab > 0 || o.retain_intermediate || (o.debug_flags & 1))
      return MM_MOE_ERR_UNSUPPORTED;
    // one expert owns at most ceil(T / 128) blocks: the ring must hold them with lag 0
    if (o.ring_blocks < (static_cast<int64_t>(T) + kBT - 1) / kBT) return MM_MOE_ERR_INVALID_ARG;
  }
  if (o.variant == MM_MOE_VARIANT_F8) {
    if (o.swap_ab > 0 || (o.block_m != 0 && o.block_m != kBT)) return MM_MOE_ERR_UNSUPPORTED;
    *p = {false, false, kBT};
    return MM_MOE_OK;
  }
  if (o.swap_ab < -1 || o.swap_ab > 2) return MM_MOE_ERR_INVALID_ARG;
  const bool swap = o.swap_ab >= 1;
  const bool pair = o.swap_ab == 2;
  if (!swap) {
    if (o.block_m != 0 && o.block_m != kBT) return MM_MOE_ERR_UNSUPPORTED;
    *p = {false, false, kBT};
    return MM_MOE_OK;
  }
  const int64_t per_expert = static_cast<int64_t>(T) * (K + o.shared_experts) / (E + o.shared_experts);
  const int bt = o.block_m ? o.block_m : (per_expert > kSwapLargeBlockTokens ? 160 : 80);
  if (!(pair ? mx_pair_block_supported(bt) : mx_sw_block_supported(bt))) return MM_MOE_ERR_UNSUPPORTED;
  *p = {true, pair, bt};
  return MM_MOE_OK;
}

// 0: per 128 (the default); -1: the pages' shape rule; 64 / 128 pinned
int f8_gran(const mm_moe_options& o, int H, int I) {
  return o.f8_act_gran == -1 ? f8_gran_rule(H, I) : (o.f8_act_gran ? o.f8_act_gran : 128);
}

// E and K are the caller's routed counts; the layout counts the shared experts in both.
Layout layout_for(const mm_moe_options& o, int T, int H, int I, int E, int K, const Plan& p) {
  const int S = o.shared_experts;
  return make_layout(T, H, I, E + S, K + S, o.variant, o.debug_flags, o.partials_bf16, p.BT, f8_gran(o, H, I), S,
                     o.ring_blocks);
}

int device_supported() {
  const DevInfo& d = dev_info();
  return (d.cc_major == 10 && d.cc_minor == 3) ? MM_MOE_OK : MM_MOE_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

void mm_moe_default_options(mm_moe_options* opt) {
  if (!opt) return;
  memset(opt, 0, sizeof(*opt));
  opt->variant = MM_MOE_VARIANT_MX;
  opt->fused = 1;
  opt->lag_units = -1;
  opt->retain_intermediate = 0;
  opt->wait_timeout_ms = 2000;
  opt->num_sms = 0;
  opt->early_combine = 0;
  opt->swap_ab = 0;
  opt->block_m = 0;
}

int mm_moe_workspace_size(const mm_moe_options* opt, int T, int H, int I, int E, int K, size_t* bytes) {
  if (!bytes) return MM_MOE_ERR_INVALID_ARG;
  const mm_moe_options o = resolve(opt);
  if (int r = check_shape(T, H, I, E, K, o.shared_experts)) return r;
  if (o.variant != MM_MOE_VARIANT_MX && o.variant != MM_MOE_VARIANT_F8) return MM_MOE_ERR_INVALID_ARG;
  Plan p;
  if (int r = make_plan(o, T, K, E, &p)) return r;
  *bytes = layout_for(o, T, H, I, E, K, p).total;
  return MM_MOE_OK;
}

int mm_moe_weight_sf_size(const mm_moe_options* opt, int H, int I, int E, size_t* w1b, size_t* w2b) {
  const mm_moe_options o = resolve(opt);
  if (!w1b || !w2b) return MM_MOE_ERR_INVALID_ARG;
  if (int r = check_shape(0, H, I, E, 1)) return r;
  if (o.variant == MM_MOE_VARIANT_MX) {
    *w1b = static_cast<size_t>(E) * 2 * I * (H / 32);
    *w2b = static_cast<size_t>(E) * ((H + 255) / 256) * 256 * (I / 32);
  } else {
    *w1b = static_cast<size_t>(E) * (2 * I / 128) * (H / 128) * sizeof(float);
    *w2b = static_cast<size_t>(E) * (H / 128) * (I / 128) * sizeof(float);
  }
  return MM_MOE_OK;
}

int mm_moe_prepare_weights(const mm_moe_options* opt, const void* w1_sf, const void* w2_sf, int H, int I, int E,
                           void* w1_sfp, void* w2_sfp, void* stream) {
  const mm_moe_options o = resolve(opt);
  if (!w1_sf || !w2_sf || !w1_sfp || !w2_sfp) return MM_MOE_ERR_INVALID_ARG;
  if (int r = check_shape(0, H, I, E, 1)) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (o.variant == MM_MOE_VARIANT_MX) {
    if (!aligned(w1_sf, 4) || !aligned(w2_sf, 4) || !aligned(w1_sfp, 16) || !aligned(w2_sfp, 16))
      return MM_MOE_ERR_INVALID_ARG;
    e = launch_prepare_sf_mx(static_cast<const uint8_t*>(w1_sf), static_cast<const uint8_t*>(w2_sf), H, I, E,
                             static_cast<uint8_t*>(w1_sfp), static_cast<uint8_t*>(w2_sfp), s);
  } else {
    size_t b1, b2;
    mm_moe_weight_sf_size(&o, H, I, E, &b1, &b2);
    e = cudaMemcpyAsync(w1_sfp, w1_sf, b1, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(w2_sfp, w2_sf, b2, cudaMemcpyDeviceToDevice, s);
  }
  return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_dispatch_scratch_size(int T, int K, int E, size_t* bytes) {
  if (!bytes || check_shape(T, 128, 128, E, K)) return MM_MOE_ERR_INVALID_ARG;
  *bytes = sizeof(int32_t) * static_cast<size_t>(kDispatchMaxCtas) * E;
  return MM_MOE_OK;
}

int mm_moe_dispatch(const int32_t* topk_idx, int T, int K, int E, int block_m, int32_t* cnt, int32_t* blk_off,
                    int32_t* slot, int32_t* src, int64_t src_capacity, void* scratch, size_t scratch_bytes,
                    int32_t* status, void* stream) {
  if (check_shape(T, 128, 128, E, K)) return MM_MOE_ERR_INVALID_ARG;
  if (block_m < 16 || block_m > 256 || block_m % 16) return MM_MOE_ERR_INVALID_ARG;
  if (!cnt || !blk_off || !status || !scratch || (T > 0 && (!topk_idx || !slot || !src)))
    return MM_MOE_ERR_INVALID_ARG;
  if (scratch_bytes < sizeof(int32_t) * static_cast<size_t>(E) || !aligned(scratch, 4)) return MM_MOE_ERR_INVALID_ARG;
  const int64_t pairs = static_cast<int64_t>(T) * K;
  const int64_t live = pairs < E ? pairs : E;
  if (src_capacity < pairs + live * (block_m - 1)) return MM_MOE_ERR_INVALID_ARG;
  if (device_supported()) return MM_MOE_ERR_UNSUPPORTED;
  cudaError_t e = launch_dispatch(topk_idx, T, K, E, block_m, cnt, blk_off, slot, src, status,
                                  static_cast<int32_t*>(scratch), static_cast<int64_t>(scratch_bytes / 4),
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_forward(const void* x, const void* x_sf, const int32_t* topk_idx, const float* topk_w, const void* w1,
                   const void* w1_sfp, const void* w2, const void* w2_sfp, void* out, int T, int H, int I, int E,
                   int K, void* workspace, size_t workspace_bytes, const mm_moe_options* opt, void* stream) {
  const mm_moe_options o = resolve(opt);
  if (int r = check_shape(T, H, I, E, K, o.shared_experts)) return r;
  if (o.variant != MM_MOE_VARIANT_MX && o.variant != MM_MOE_VARIANT_F8) return MM_MOE_ERR_INVALID_ARG;
  if (T == 0) {
    // nothing to compute; leave a clean status word for mm_moe_sync_status
    if (workspace && workspace_bytes >= 16 && aligned(workspace, 256))
      return cudaMemsetAsync(workspace, 0, 16, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MM_MOE_OK
                                                                                              : MM_MOE_ERR_CUDA;
    return MM_MOE_OK;
  }
  if (!x || (!x_sf && !o.x_bf16) || !topk_idx || !topk_w || !w1 || !w1_sfp || !w2 || !w2_sfp || !out || !workspace)
    return MM_MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (!o.x_bf16 && !aligned(x_sf, 4)) || !aligned(w1, 32) || !aligned(w2, 32) || !aligned(out, 16) ||
      !aligned(workspace, 256) || !aligned(w1_sfp, 16) || !aligned(w2_sfp, 16))
    return MM_MOE_ERR_INVALID_ARG;
  if (device_supported()) return MM_MOE_ERR_UNSUPPORTED;
  // cta_pairs is reserved: 0 and 1 mean one CTA per tile group, anything else is not built
  if (o.cta_pairs != 0 && o.cta_pairs != 1) return MM_MOE_ERR_UNSUPPORTED;
  Plan plan;
  if (int r = make_plan(o, T, K, E, &plan)) return r;
  // the fused stream exists for the MX format; F8 and the L1 debug dump run the two-launch path
  const bool fused = o.fused && o.variant == MM_MOE_VARIANT_MX && !(o.debug_flags & 1);
  const int grid = (o.num_sms > 0 && o.num_sms < dev_info().sms) ? o.num_sms : dev_info().sms;
  // per-task trace: [launch][CTA][cap] records of the token-M MX kernel
  int64_t trace_cap = 0;
  if (o.trace_buf) {
    if (o.variant != MM_MOE_VARIANT_MX || plan.swap) return MM_MOE_ERR_UNSUPPORTED;
    if (!aligned(o.trace_buf, 16)) return MM_MOE_ERR_INVALID_ARG;
    trace_cap = static_cast<int64_t>(o.trace_bytes / (sizeof(TraceRec) * grid * (fused ? 1 : 2)));
    if (trace_cap < 1) return MM_MOE_ERR_INVALID_ARG;
    if (trace_cap > (int64_t(1) << 30)) trace_cap = int64_t(1) << 30;
  }
  const Layout L = layout_for(o, T, H, I, E, K, plan);
  if (workspace_bytes < L.total) return MM_MOE_ERR_WORKSPACE_TOO_SMALL;
  // early combine in the fused stream
  const bool early = fused && o.early_combine;
  const WsPtrs W = ws_ptrs(workspace, L);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // from here on the routing, the expert count and the slot count include the shared experts
  const int32_t* idx = L.S ? W.ext_idx : topk_idx;
  const float* wts = L.S ? W.ext_w : topk_w;

  cudaEvent_t* ev = static_cast<cudaEvent_t*>(o.timing_events);
  auto mark = [&](int i) -> cudaError_t { return ev && ev[i] ? cudaEventRecord(ev[i], s) : cudaSuccess; };
  // kernels follow one another with programmatic launches only where no event sits between them
  const bool pdl_gemm = fused && !(ev && (ev[1] || ev[2]));
  const bool pdl_combine = !(ev && (ev[3] || ev[4]));

  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = cudaMemsetAsync(W.status, 0, 16, s);
  // the arrival counters of the fused stream and the tile-group counters of every GEMM launch,
  // cleared before the routing kernels so that those and the GEMM are adjacent on the stream
  if (e == cudaSuccess) e = cudaMemsetAsync(W.ctr, 0, sizeof(int) * ctr_ints(L), s);
  if (e == cudaSuccess && W.prof) e = cudaMemsetAsync(W.prof, 0, 2 * 8 * 1024 * sizeof(unsigned long long), s);
  if (e == cudaSuccess && L.S) e = launch_extend_routing(topk_idx, topk_w, T, K, E, L.S, W.ext_idx, W.ext_w, s);
  if (e == cudaSuccess)
    e = launch_dispatch(idx, T, L.K, L.E, L.BT, W.cnt, W.blk_off, W.slot, W.src, W.status, W.dscr,
                        static_cast<int64_t>(kDispatchMaxCtas) * L.E, s);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess && !fused) e = launch_gather(L, W, static_cast<const uint8_t*>(x), x_sf, o.x_bf16 != 0, s);
  if (e == cudaSuccess) e = mark(2);
  const uint64_t timeout_ns = static_cast<uint64_t>(o.wait_timeout_ms) * 1000000ull;
  const float clamp = o.activation_clamp > 0.f ? o.activation_clamp : INFINITY;
  if (o.variant == MM_MOE_VARIANT_MX) {
    GemmLaunch g{&L, &W, static_cast<const uint8_t*>(w1), static_cast<const uint8_t*>(w1_sfp),
                 static_cast<const uint8_t*>(w2), static_cast<const uint8_t*>(w2_sfp),
                 static_cast<const uint8_t*>(x), x_sf, o.x_bf16 != 0, wts, W.dbg, W.prof, timeout_ns, grid,
                 clamp, o.precise_swiglu != 0, early, idx, out, pdl_gemm,
                 // a shared expert has T / 128 blocks: deal them one by one, not as one CTA's run
                 (o.debug_flags & 8) != 0 || L.S > 0};
    g.trace = static_cast<uint8_t*>(o.trace_buf);
    g.trace_cap = static_cast<int>(trace_cap);
    auto gemm = plan.pair ? launch_gemm_mx_pair : (plan.swap ? launch_gemm_mx_sw : launch_gemm_mx);
    if (fused) {
      // one lag-ordered stream: gather, L1 and L2 in a single persistent launch
      const int lag = o.lag_units >= 0 ? o.lag_units : mx_lag_auto(L.E);
      if (e == cudaSuccess) e = gemm(g, 3, lag, (o.debug_flags & 4) ? 1 : 0, s);
      if (e == cudaSuccess) e = mark(3);
    } else {
      if (e == cudaSuccess) e = gemm(g, 1, 0, 0, s);
      if (e == cudaSuccess) e = mark(3);
      if (o.debug_flags & 1) return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
      if (g.trace) g.trace += static_cast<size_t>(grid) * trace_cap * sizeof(TraceRec);   // the L2 launch's slice
      if (e == cudaSuccess) e = gemm(g, 2, 0, 0, s);
    }
  } else {
    GemmLaunchF8 g{&L, &W, static_cast<const uint8_t*>(w1), static_cast<const float*>(w1_sfp), wts, timeout_ns,
                   grid, W.prof, clamp, o.precise_swiglu != 0, (o.debug_flags & 16) != 0, (o.debug_flags & 4) != 0};
    if (e == cudaSuccess) e = launch_gemm_f8_l1(g, s);
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess) {
      g.w = static_cast<const uint8_t*>(w2);
      g.wsf = static_cast<const float*>(w2_sfp);
      e = launch_gemm_f8_l2(g, s);
    }
  }
  if (e == cudaSuccess) e = mark(4);
  // the fused stream's early combine has written `out` already
  if (e == cudaSuccess && !early) e = launch_combine(L, W, idx, out, pdl_combine, s);
  if (e == cudaSuccess) e = mark(5);
  if (e != cudaSuccess) {
    if (getenv("MM_MOE_DEBUG")) fprintf(stderr, "mm_moe_forward: %s\n", cudaGetErrorString(e));
    return MM_MOE_ERR_CUDA;
  }
  return MM_MOE_OK;
}

int mm_moe_read_routing(const void* workspace, const mm_moe_options* opt, int T, int H, int I, int E, int K,
                        int32_t* cnt, int32_t* blk_off, int32_t* slot, int32_t* src, int* block_m, void* stream) {
  const mm_moe_options o = resolve(opt);
  if (int r = check_shape(T, H, I, E, K, o.shared_experts)) return r;
  if (!workspace) return MM_MOE_ERR_INVALID_ARG;
  Plan plan;
  if (int r = make_plan(o, T, K, E, &plan)) return r;
  const Layout L = layout_for(o, T, H, I, E, K, plan);
  const WsPtrs W = ws_ptrs(const_cast<void*>(workspace), L);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (cnt) e = cudaMemcpyAsync(cnt, W.cnt, sizeof(int) * L.E, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && blk_off) e = cudaMemcpyAsync(blk_off, W.blk_off, sizeof(int) * (L.E + 1), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && slot && T > 0)
    e = cudaMemcpyAsync(slot, W.slot, sizeof(int) * static_cast<size_t>(T) * L.K, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && src && L.P > 0)
    e = cudaMemcpyAsync(src, W.src, sizeof(int) * static_cast<size_t>(L.P), cudaMemcpyDeviceToDevice, s);
  if (block_m) *block_m = L.BT;
  return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_read_intermediate(const void* workspace, const mm_moe_options* opt, int T, int H, int I, int E, int K,
                             int64_t rows, uint8_t* codes, void* sf, void* stream) {
  const mm_moe_options o = resolve(opt);
  if (int r = check_shape(T, H, I, E, K, o.shared_experts)) return r;
  if (!workspace || !codes || !sf || rows < 0) return MM_MOE_ERR_INVALID_ARG;
  Plan plan;
  if (int r = make_plan(o, T, K, E, &plan)) return r;
  const Layout L = layout_for(o, T, H, I, E, K, plan);
  if (L.ring) return MM_MOE_ERR_UNSUPPORTED;   // a ring keeps only its last R blocks
  if (rows > L.P) return MM_MOE_ERR_INVALID_ARG;
  if (rows == 0) return MM_MOE_OK;
  const WsPtrs W = ws_ptrs(const_cast<void*>(workspace), L);
  cudaError_t e = launch_read_intermediate(L, W, rows, codes, sf, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}

int mm_moe_workspace_region(const void* workspace, const mm_moe_options* opt, int T, int H, int I, int E, int K,
                            int region, void** ptr, size_t* bytes) {
  const mm_moe_options o = resolve(opt);
  if (int r = check_shape(T, H, I, E, K, o.shared_experts)) return r;
  if (!ptr || !bytes) return MM_MOE_ERR_INVALID_ARG;
  Plan plan;
  if (int r = make_plan(o, T, K, E, &plan)) return r;
  const Layout L = layout_for(o, T, H, I, E, K, plan);
  const size_t offs[13] = {L.status, L.cnt, L.blk_off, L.slot, L.src, L.pool_x, L.pool_x_sf, L.pool2, L.pool2_sf,
                           L.part, L.dbg, L.prof, L.ext_idx};
  if (region < 0 || region > 11) return MM_MOE_ERR_INVALID_ARG;
  size_t n;
  if (region == 10) n = L.dbg_bytes;
  else if (region == 11) n = L.total - L.prof;
  else if (region == 0) n = 16;
  else if (region == 1) n = sizeof(int) * L.E;
  else if (region == 2) n = sizeof(int) * (L.E + 1);
  else if (region == 3) n = sizeof(int) * static_cast<size_t>(T) * L.K;
  else if (region == 4) n = sizeof(int) * static_cast<size_t>(L.P);
  else if (region == 9) n = static_cast<size_t>(L.part_elem) * T * L.K * H;
  else n = offs[region + 1] - offs[region];
  *ptr = static_cast<uint8_t*>(const_cast<void*>(workspace)) + offs[region];
  *bytes = n;
  return MM_MOE_OK;
}

int mm_moe_sync_status(const void* workspace, void* stream, int* where) {
  if (!workspace) return MM_MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MM_MOE_ERR_CUDA;
  int h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MM_MOE_ERR_CUDA;
  if (where) *where = h[1];
  if (h[0] && getenv("MM_MOE_DEBUG"))
    fprintf(stderr, "mm_moe: device status %d at site %d (detail %08x %08x)\n", h[0], h[1], h[2], h[3]);
  return h[0];
}

const char* mm_moe_status_string(int code) {
  switch (code) {
    case MM_MOE_OK: return "ok";
    case MM_MOE_ERR_INVALID_ARG: return "invalid argument";
    case MM_MOE_ERR_UNSUPPORTED: return "unsupported device or option";
    case MM_MOE_ERR_CUDA: return "CUDA error";
    case MM_MOE_ERR_TIMEOUT: return "device wait timed out";
    case MM_MOE_ERR_BAD_ROUTING: return "topk_idx holds expert ids >= E or < -1";
    case MM_MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    default: return "unknown status";
  }
}

}  // extern "C"

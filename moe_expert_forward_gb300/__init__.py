"""Python binding of libmm_moe.so (the GB300 MoE-layer forward).

Argument marshalling only: every step of the forward runs in the library's CUDA
kernels.  The C entry points are exposed under their own names (taking integer
device pointers); the tensor helpers below only turn torch tensors into
pointers and raise on a non-zero status.  There is no fallback: importing the
binding fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmm_moe.so")

MM_MOE_OK = 0
MM_MOE_ERR_INVALID_ARG = 1
MM_MOE_ERR_UNSUPPORTED = 2
MM_MOE_ERR_CUDA = 3
MM_MOE_ERR_TIMEOUT = 4
MM_MOE_ERR_BAD_ROUTING = 5
MM_MOE_ERR_WORKSPACE_TOO_SMALL = 6
MM_MOE_VARIANT_MX = 0
MM_MOE_VARIANT_F8 = 1
MM_MOE_NUM_TIMING_EVENTS = 6
STAGES = ["dispatch", "gather", "l1", "l2", "combine"]

# every symbol include/mm_moe.h declares
EXPORTS = ["mm_moe_default_options", "mm_moe_workspace_size", "mm_moe_weight_sf_size", "mm_moe_prepare_weights",
           "mm_moe_forward", "mm_moe_dispatch_scratch_size", "mm_moe_dispatch", "mm_moe_read_routing", "mm_moe_read_intermediate",
           "mm_moe_sync_status", "mm_moe_status_string", "mm_moe_workspace_region",
           "mm_moe_dispatch_noalloc", "mm_moe_ep_count", "mm_moe_ep_plan", "mm_moe_ep_push_meta", "mm_moe_ep_pull",
           "mm_moe_ep_combine", "mm_moe_ep_push_out", "mm_moe_ep_combine_local", "mm_moe_ep_recv_capacity",
           "mm_moe_ep_barrier", "mm_moe_ep_barrier_ranks"]


class mm_moe_options(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("fused", ctypes.c_int), ("lag_units", ctypes.c_int),
                ("retain_intermediate", ctypes.c_int), ("wait_timeout_ms", ctypes.c_uint),
                ("num_sms", ctypes.c_int), ("debug_flags", ctypes.c_int), ("cta_pairs", ctypes.c_int),
                ("partials_bf16", ctypes.c_int), ("activation_clamp", ctypes.c_float),
                ("precise_swiglu", ctypes.c_int), ("x_bf16", ctypes.c_int), ("early_combine", ctypes.c_int),
                ("swap_ab", ctypes.c_int), ("block_m", ctypes.c_int),
                ("f8_act_gran", ctypes.c_int), ("shared_experts", ctypes.c_int), ("ring_blocks", ctypes.c_int),
                ("trace_buf", ctypes.c_void_p), ("trace_bytes", ctypes.c_size_t),
                ("timing_events", ctypes.c_void_p)]


class MMError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {mm_moe_status_string(code)} ({code})")
        self.code = code


_lib: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_OPT = ctypes.POINTER(mm_moe_options)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with moe_expert_forward_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "mm_moe_default_options": (None, [_OPT]),
            "mm_moe_workspace_size": (_I, [_OPT, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
            "mm_moe_weight_sf_size": (_I, [_OPT, _I, _I, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
            "mm_moe_prepare_weights": (_I, [_OPT, _P, _P, _I, _I, _I, _P, _P, _P]),
            "mm_moe_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _OPT, _P]),
            "mm_moe_dispatch_scratch_size": (_I, [_I, _I, _I, ctypes.POINTER(_SZ)]),
            "mm_moe_dispatch": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I64, _P, _SZ, _P, _P]),
            "mm_moe_read_routing": (_I, [_P, _OPT, _I, _I, _I, _I, _I, _P, _P, _P, _P, ctypes.POINTER(_I), _P]),
            "mm_moe_read_intermediate": (_I, [_P, _OPT, _I, _I, _I, _I, _I, _I64, _P, _P, _P]),
            "mm_moe_sync_status": (_I, [_P, _P, ctypes.POINTER(_I)]),
            "mm_moe_status_string": (ctypes.c_char_p, [_I]),
            "mm_moe_dispatch_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I64, _P, _P]),
            "mm_moe_workspace_region": (_I, [_P, _OPT, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_P),
                                             ctypes.POINTER(_SZ)]),
            "mm_moe_ep_count": (_I, [_P, _I, _I, _I, _P, _P]),
            "mm_moe_ep_plan": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, ctypes.POINTER(_I64), _P, _I64]),
            "mm_moe_ep_push_meta": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
            "mm_moe_ep_pull": (_I, [_P, _I64, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
            "mm_moe_ep_combine": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
            "mm_moe_ep_push_out": (_I, [_P, _I64, _I, _P, _P, _P]),
            "mm_moe_ep_combine_local": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
            "mm_moe_ep_recv_capacity": (_I, [_I, _I, _I, _I, ctypes.POINTER(_I64)]),
            "mm_moe_ep_barrier": (_I, [_P, _I, _I, ctypes.c_uint32, ctypes.c_uint, _P, _P]),
            "mm_moe_ep_barrier_ranks": (_I, [_P, _I, ctypes.c_uint32, ctypes.c_uint, ctypes.c_uint64, _P, _P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------------ C entry points, same names
def mm_moe_default_options(opt: Optional[mm_moe_options] = None) -> mm_moe_options:
    opt = opt or mm_moe_options()
    lib().mm_moe_default_options(ctypes.byref(opt))
    return opt


def mm_moe_workspace_size(opt, T, H, I, E, K) -> int:
    n = _SZ(0)
    _check(lib().mm_moe_workspace_size(_opt(opt), T, H, I, E, K, ctypes.byref(n)), "mm_moe_workspace_size")
    return n.value


def mm_moe_weight_sf_size(opt, H, I, E):
    a, b = _SZ(0), _SZ(0)
    _check(lib().mm_moe_weight_sf_size(_opt(opt), H, I, E, ctypes.byref(a), ctypes.byref(b)), "mm_moe_weight_sf_size")
    return a.value, b.value


def mm_moe_prepare_weights(opt, w1_sf, w2_sf, H, I, E, w1_sfp, w2_sfp, stream) -> int:
    return lib().mm_moe_prepare_weights(_opt(opt), w1_sf, w2_sf, H, I, E, w1_sfp, w2_sfp, stream)


def mm_moe_forward(x, x_sf, topk_idx, topk_w, w1, w1_sfp, w2, w2_sfp, out, T, H, I, E, K, workspace, ws_bytes,
                   opt, stream) -> int:
    return lib().mm_moe_forward(x, x_sf, topk_idx, topk_w, w1, w1_sfp, w2, w2_sfp, out, T, H, I, E, K, workspace,
                                ws_bytes, _opt(opt), stream)


def mm_moe_dispatch_scratch_size(T, K, E) -> int:
    n = _SZ(0)
    _check(lib().mm_moe_dispatch_scratch_size(T, K, E, ctypes.byref(n)), "mm_moe_dispatch_scratch_size")
    return n.value


def mm_moe_dispatch(topk_idx, T, K, E, block_m, cnt, blk_off, slot, src, src_capacity, scratch, scratch_bytes,
                    status, stream) -> int:
    return lib().mm_moe_dispatch(topk_idx, T, K, E, block_m, cnt, blk_off, slot, src, src_capacity, scratch,
                                 scratch_bytes, status, stream)


def mm_moe_dispatch_noalloc(topk_idx, T, K, E, block_m, cnt, blk_off, slot, src, src_capacity, status,
                            stream) -> int:
    """Routing without caller scratch: for callers that cannot allocate device memory."""
    return lib().mm_moe_dispatch_noalloc(topk_idx, T, K, E, block_m, cnt, blk_off, slot, src, src_capacity, status,
                                         stream)


def mm_moe_read_routing(workspace, opt, T, H, I, E, K, cnt, blk_off, slot, src, stream):
    bm = _I(0)
    r = lib().mm_moe_read_routing(workspace, _opt(opt), T, H, I, E, K, cnt, blk_off, slot, src, ctypes.byref(bm),
                                  stream)
    return r, bm.value


def mm_moe_read_intermediate(workspace, opt, T, H, I, E, K, rows, codes, sf, stream) -> int:
    return lib().mm_moe_read_intermediate(workspace, _opt(opt), T, H, I, E, K, rows, codes, sf, stream)


def mm_moe_sync_status(workspace, stream):
    where = _I(0)
    r = lib().mm_moe_sync_status(workspace, stream, ctypes.byref(where))
    return r, where.value


def mm_moe_status_string(code: int) -> str:
    try:
        return lib().mm_moe_status_string(code).decode()
    except ImportError:
        return f"status {code}"


def mm_moe_workspace_region(workspace, opt, T, H, I, E, K, region):
    p, n = _P(0), _SZ(0)
    _check(lib().mm_moe_workspace_region(workspace, _opt(opt), T, H, I, E, K, region, ctypes.byref(p),
                                         ctypes.byref(n)), "mm_moe_workspace_region")
    return p.value or 0, n.value


REGIONS = {"status": 0, "cnt": 1, "blk_off": 2, "slot": 3, "src": 4, "pool_x": 5, "pool_x_sf": 6, "pool2": 7,
           "pool2_sf": 8, "partials": 9, "debug": 10, "prof": 11}


def workspace_view(workspace, opt, T, H, I, E, K, region: str, dtype=None):
    """A torch view of one workspace region (diagnostics and tests)."""
    import torch
    p, n = mm_moe_workspace_region(_ptr(workspace), opt, T, H, I, E, K, REGIONS[region])
    off = p - workspace.data_ptr()
    v = workspace[off:off + n]
    return v.view(dtype) if dtype is not None else v


def _opt(opt):
    return ctypes.byref(opt) if opt is not None else None


def _check(code: int, what: str):
    if code != MM_MOE_OK:
        raise MMError(code, what)


# ------------------------------------------------------------------ torch-tensor marshalling
def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def options(variant: int = MM_MOE_VARIANT_MX, **kw) -> mm_moe_options:
    o = mm_moe_default_options()
    o.variant = variant
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def _need(t, nbytes: int, name: str, what: str) -> None:
    """The C ABI takes bare pointers; check here that a tensor is a contiguous
    CUDA buffer of at least `nbytes` bytes before its address goes down."""
    if t is None or not t.is_cuda or not t.is_contiguous() or t.numel() * t.element_size() < nbytes:
        got = "None" if t is None else (f"{tuple(t.shape)} {t.dtype} on {t.device}"
                                        f"{'' if t.is_contiguous() else ' (not contiguous)'}")
        raise MMError(MM_MOE_ERR_INVALID_ARG, f"{what}: {name} must be a contiguous CUDA tensor of at least "
                                              f"{nbytes} bytes, got {got}")


def _input_bytes(variant: int, T: int, H: int, I: int, E: int, K: int) -> dict:
    """Bytes of every caller buffer of one forward, in the layouts of mm_moe.h."""
    if variant == MM_MOE_VARIANT_MX:
        return {"x": T * H, "x_sf": T * (H // 32), "w1": E * 2 * I * H // 2, "w1_sf": E * 2 * I * (H // 32),
                "w2": E * H * I // 2, "w2_sf": E * H * (I // 32), "topk_idx": 4 * T * K, "topk_w": 4 * T * K,
                "out": 2 * T * H}
    return {"x": T * H, "x_sf": 4 * T * (H // 128), "w1": E * 2 * I * H, "w1_sf": 4 * E * (2 * I // 128) * (H // 128),
            "w2": E * H * I, "w2_sf": 4 * E * (H // 128) * (I // 128), "topk_idx": 4 * T * K, "topk_w": 4 * T * K,
            "out": 2 * T * H}


def prepare_weights(w1_sf, w2_sf, H, I, E, opt=None, stream=None):
    """Return (w1_sfp, w2_sfp) device tensors in the kernels' scale layout."""
    import torch
    opt = opt or options()
    need = _input_bytes(opt.variant, 0, H, I, E, 1)
    _need(w1_sf, need["w1_sf"], "w1_sf", "prepare_weights")
    _need(w2_sf, need["w2_sf"], "w2_sf", "prepare_weights")
    n1, n2 = mm_moe_weight_sf_size(opt, H, I, E)
    a = torch.empty(n1, dtype=torch.uint8, device=w1_sf.device)
    b = torch.empty(n2, dtype=torch.uint8, device=w1_sf.device)
    _check(mm_moe_prepare_weights(opt, _ptr(w1_sf), _ptr(w2_sf), H, I, E, _ptr(a), _ptr(b), _stream(stream)),
           "mm_moe_prepare_weights")
    return a, b


def alloc_workspace(T, H, I, E, K, opt=None, device="cuda"):
    import torch
    n = mm_moe_workspace_size(opt or options(), T, H, I, E, K)
    return torch.empty(max(n, 1024), dtype=torch.uint8, device=device)


def forward(x, x_sf, topk_idx, topk_w, w1, w1_sfp, w2, w2_sfp, out, H, I, E, workspace, opt=None, stream=None):
    T, K = topk_idx.shape
    opt = opt or options()
    need = _input_bytes(opt.variant, T, H, I, E, K)
    S = max(int(opt.shared_experts), 0)   # shared experts: the weight arrays hold E + S experts
    wneed = _input_bytes(opt.variant, T, H, I, E + S, K)
    need.update({k: wneed[k] for k in ("w1", "w2")})
    if opt.x_bf16:
        need["x"] = 2 * T * H          # bf16 rows; the gather quantises them, x_sf is not read
    for name, t in (("x", x), ("x_sf", x_sf), ("topk_idx", topk_idx), ("topk_w", topk_w), ("w1", w1), ("w2", w2),
                    ("out", out)):
        if name == "x_sf" and opt.x_bf16:
            continue
        if T > 0 or name in ("w1", "w2"):
            _need(t, need[name], name, "forward")
    n1, n2 = mm_moe_weight_sf_size(opt, H, I, E + S)
    _need(w1_sfp, n1, "w1_sfp", "forward")
    _need(w2_sfp, n2, "w2_sfp", "forward")
    _need(workspace, 0, "workspace", "forward")   # its size goes down with it: the library checks that
    _check(mm_moe_forward(_ptr(x), _ptr(x_sf), _ptr(topk_idx), _ptr(topk_w), _ptr(w1), _ptr(w1_sfp), _ptr(w2),
                          _ptr(w2_sfp), _ptr(out), T, H, I, E, K, _ptr(workspace), workspace.numel(),
                          opt, _stream(stream)), "mm_moe_forward")
    return out


def sync_status(workspace, stream=None):
    code, where = mm_moe_sync_status(_ptr(workspace), _stream(stream))
    return code, where


# ------------------------------------------------------------------ expert parallelism (C entry points)
def mm_moe_ep_count(topk_idx, T, K, E, counts, stream) -> int:
    return lib().mm_moe_ep_count(topk_idx, T, K, E, counts, stream)


def mm_moe_ep_plan(counts_all, topk_idx, T, K, E, N, rank, recv_expert=True, recv_capacity=None):
    """Host planning (numpy in, numpy out): counts_all int32 [N, E], topk_idx int32
    [T, K] of this rank.  Returns (send_row int32 [T*K], recv_rows, recv_expert
    int32 [recv_rows] or None).  recv_capacity (e.g. mm_moe_ep_recv_capacity of the
    token bound): the library refuses a receive count above it."""
    import numpy as np
    counts_all = np.ascontiguousarray(counts_all, dtype=np.int32)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    send_row = np.empty(max(T * K, 1), dtype=np.int32)
    rows = _I64(0)
    _check(lib().mm_moe_ep_plan(counts_all.ctypes.data, topk_idx.ctypes.data, T, K, E, N, rank,
                                send_row.ctypes.data, ctypes.byref(rows), None, 0), "mm_moe_ep_plan")
    rex = None
    if recv_expert or recv_capacity is not None:
        cap = rows.value if recv_capacity is None else int(recv_capacity)
        rex = np.empty(max(cap, rows.value, 1), dtype=np.int32)
        if recv_capacity is not None:
            rex = rex[:max(cap, 1)]
        _check(lib().mm_moe_ep_plan(counts_all.ctypes.data, topk_idx.ctypes.data, T, K, E, N, rank,
                                    send_row.ctypes.data, ctypes.byref(rows), rex.ctypes.data,
                                    rex.size if recv_capacity is None else int(recv_capacity)), "mm_moe_ep_plan")
        rex = rex[:rows.value]
    return send_row[:T * K], rows.value, rex


def mm_moe_ep_push_meta(topk_idx, topk_w, send_row, T, K, E, N, rank, peer_meta, stream) -> int:
    return lib().mm_moe_ep_push_meta(topk_idx, topk_w, send_row, T, K, E, N, rank, peer_meta, stream)


def mm_moe_ep_pull(meta, rows, K, H, variant, peer_x, peer_x_sf, x_recv, x_sf_recv, idx_recv, w_recv, stream) -> int:
    return lib().mm_moe_ep_pull(meta, rows, K, H, variant, peer_x, peer_x_sf, x_recv, x_sf_recv, idx_recv, w_recv,
                                stream)


def mm_moe_ep_combine(topk_idx, send_row, T, K, E, N, H, peer_out, out, stream) -> int:
    return lib().mm_moe_ep_combine(topk_idx, send_row, T, K, E, N, H, peer_out, out, stream)


def mm_moe_ep_push_out(meta, rows, H, out_recv, peer_partials, stream) -> int:
    return lib().mm_moe_ep_push_out(meta, rows, H, out_recv, peer_partials, stream)


def mm_moe_ep_combine_local(topk_idx, T, K, E, H, partials, out, stream) -> int:
    return lib().mm_moe_ep_combine_local(topk_idx, T, K, E, H, partials, out, stream)


def mm_moe_ep_recv_capacity(num_tokens_bound, K, E, N) -> int:
    n = _I64(0)
    _check(lib().mm_moe_ep_recv_capacity(num_tokens_bound, K, E, N, ctypes.byref(n)), "mm_moe_ep_recv_capacity")
    return n.value


def mm_moe_ep_barrier(peer_flags, N, rank, epoch, timeout_ms, status, stream) -> int:
    return lib().mm_moe_ep_barrier(peer_flags, N, rank, epoch, timeout_ms, status, stream)


def mm_moe_ep_barrier_ranks(peer_flags, N, epoch, timeout_ms, absent, status, stream) -> int:
    return lib().mm_moe_ep_barrier_ranks(peer_flags, N, epoch, timeout_ms, absent, status, stream)

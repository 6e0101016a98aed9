"""The C-ABI library builds, loads and exports every entry point include/mm_moe.h
declares; host-side argument checks and workspace sizing (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    from moe_expert_forward_gb300 import build
    build.build()
    import moe_expert_forward_gb300 as M
    return M


def _declared():
    txt = open(os.path.join(ROOT, "include", "mm_moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(mm_moe_[a-z_]+)\s*\(", txt)))


def test_header_declares_the_binding_exports(M):
    assert _declared() == sorted(M.EXPORTS)


def test_library_exports_every_declared_symbol(M):
    lib = ctypes.CDLL(M.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(M):
    for c in range(7):
        assert M.mm_moe_status_string(c)


def test_workspace_size_and_shape_checks(M):
    opt = M.options()
    n = M.mm_moe_workspace_size(opt, 64, 256, 128, 8, 2)
    assert n > 64 * 256
    n_big = M.mm_moe_workspace_size(opt, 2048, 4096, 2048, 256, 6)
    # pool capacity T*K + E*(128-1) rows of H bytes at least
    assert n_big >= (2048 * 6 + 256 * 127) * 4096
    for bad in [(64, 200, 128, 8, 2), (64, 256, 100, 8, 2), (64, 256, 128, 8, 0), (64, 256, 128, 2, 4),
                (-1, 256, 128, 8, 2), (64, 256, 128, 2000, 2), (64, 256, 128, 32, 17)]:
        with pytest.raises(M.MMError) as ei:
            M.mm_moe_workspace_size(opt, *bad)
        assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG


def test_forward_rejects_null_and_small_workspace_without_touching_the_gpu(M):
    opt = M.options()
    # null inputs are rejected before any device call
    r = M.mm_moe_forward(0, 0, 0, 0, 0, 0, 0, 0, 0, 64, 256, 128, 8, 2, 0, 0, opt, 0)
    assert r == M.MM_MOE_ERR_INVALID_ARG
    # T = 0 is a no-op that succeeds without pointers
    assert M.mm_moe_forward(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 256, 128, 8, 2, 0, 0, opt, 0) == M.MM_MOE_OK


def test_weight_sf_sizes(M):
    a, b = M.mm_moe_weight_sf_size(M.options(), 4096, 2048, 256)
    assert a == 256 * 4096 * 4096 // 32 and b == 256 * 4096 * 2048 // 32
    a, b = M.mm_moe_weight_sf_size(M.options(M.MM_MOE_VARIANT_F8), 4096, 2048, 256)
    assert a == 256 * 32 * 32 * 4 and b == 256 * 32 * 16 * 4


def test_binding_rejects_wrong_buffers_before_any_device_work(M):
    """The C ABI takes bare pointers; the Python binding checks device, contiguity
    and byte size of every buffer against the layouts of mm_moe.h first, so a
    host tensor or the other variant's scale array never reaches a kernel."""
    import torch
    H, I, E = 256, 128, 8
    # F8 scale arrays ([E, 2I/128, H/128] fp32) are far smaller than MX's UE8M0 ones ([E, 2I, H/32] bytes)
    f8_w1_sf = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32)
    f8_w2_sf = torch.empty(E, H // 128, I // 128, dtype=torch.float32)
    with pytest.raises(M.MMError) as ei:
        M.prepare_weights(f8_w1_sf, f8_w2_sf, H, I, E, M.options(M.MM_MOE_VARIANT_MX))
    assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG and "w1_sf" in str(ei.value)
    # a host tensor of the right size is refused as well
    mx_w1_sf = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8)
    with pytest.raises(M.MMError) as ei:
        M.prepare_weights(mx_w1_sf, mx_w1_sf, H, I, E, M.options(M.MM_MOE_VARIANT_MX))
    assert "CUDA" in str(ei.value)
    T, K = 4, 2
    idx = torch.zeros(T, K, dtype=torch.int32)
    with pytest.raises(M.MMError) as ei:
        M.forward(torch.empty(T, H, dtype=torch.uint8), None, idx, None, None, None, None, None, None, H, I, E,
                  torch.empty(16, dtype=torch.uint8))
    assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG


def test_options_struct_layout_matches_the_header(M, tmp_path):
    """Every field of the ctypes mm_moe_options sits at the offset the C header
    gives it, and the struct has the header's size (compiled with the host C
    compiler), so a field added in one place only is caught on the CPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    names = [f[0] for f in M.mm_moe_options._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mm_moe.h"', 'int main(void) {',
             '  printf("%zu\\n", sizeof(mm_moe_options));']
    lines += [f'  printf("%zu\\n", offsetof(mm_moe_options, {n}));' for n in names]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([cc, "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(M.mm_moe_options)
    for n, off in zip(names, got[1:]):
        assert getattr(M.mm_moe_options, n).offset == off, n


def test_f8_scale_width_option_host_checks(M):
    """f8_act_gran takes 0 (per 128), -1 (the pages' shape rule), 64 or 128; the
    per-64 intermediate holds twice the scales of the per-128 one (fp32 [P, I / 64])."""
    T, H, I, E, K = 300, 512, 384, 5, 2
    for g in (32, 96, 256, -2):
        with pytest.raises(M.MMError) as ei:
            M.mm_moe_workspace_size(M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=g), T, H, I, E, K)
        assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG
    n = {g: M.mm_moe_workspace_size(M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=g), T, H, I, E, K)
         for g in (0, -1, 64, 128)}
    assert n[0] == n[128] < n[64] == n[-1]        # H = 512, 2I = 768: the rule takes 64
    _, sf_bytes = M.mm_moe_workspace_region(0, M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=64), T, H, I, E, K, 8)
    _, sf128 = M.mm_moe_workspace_region(0, M.options(M.MM_MOE_VARIANT_F8, f8_act_gran=128), T, H, I, E, K, 8)
    assert sf_bytes >= 2 * (sf128 - 1023)


def test_shared_experts_host_checks(M):
    """Shared experts add S slots per token and S experts: K + S <= 16 and
    E + S <= 1024, and the workspace grows with them."""
    T, H, I, E, K = 64, 256, 128, 8, 2
    base = M.mm_moe_workspace_size(M.options(), T, H, I, E, K)
    one = M.mm_moe_workspace_size(M.options(shared_experts=1), T, H, I, E, K)
    assert one > base
    assert M.mm_moe_workspace_size(M.options(shared_experts=14), T, H, I, E, K) > one
    for bad in (dict(shared_experts=15), dict(shared_experts=-1)):
        with pytest.raises(M.MMError) as ei:
            M.mm_moe_workspace_size(M.options(**bad), T, H, I, E, K)
        assert ei.value.code == M.MM_MOE_ERR_INVALID_ARG
    with pytest.raises(M.MMError):
        M.mm_moe_workspace_size(M.options(shared_experts=2), T, H, I, 1023, K)
    # the routing regions count the shared slots and experts
    _, cnt_bytes = M.mm_moe_workspace_region(0, M.options(shared_experts=3), T, H, I, E, K, 1)
    _, slot_bytes = M.mm_moe_workspace_region(0, M.options(shared_experts=3), T, H, I, E, K, 3)
    assert cnt_bytes == 4 * (E + 3) and slot_bytes == 4 * T * (K + 3)


def test_ring_host_checks(M):
    """ring_blocks: 0 = the whole pool; R > 0 only for the token-M MX fused
    stream (else UNSUPPORTED) and only with R >= ceil(T / 128) (else INVALID_ARG);
    the intermediate then holds R blocks of codes and scales instead of one per
    pool block, and a ring as large as the pool changes nothing."""
    T, H, I, E, K = 2048, 4096, 2048, 256, 6
    mx = lambda **kw: M.options(M.MM_MOE_VARIANT_MX, **kw)
    full = M.mm_moe_workspace_size(mx(), T, H, I, E, K)
    ring = M.mm_moe_workspace_size(mx(ring_blocks=64), T, H, I, E, K)
    blocks = ((T * K + E * 127) + 127) // 128
    assert full - ring >= (blocks - 64) * 128 * I * 33 // 32 - 4096
    _, codes = M.mm_moe_workspace_region(0, mx(ring_blocks=64), T, H, I, E, K, 7)
    assert 64 * 128 * I <= codes < 64 * 128 * I + 1024
    assert M.mm_moe_workspace_size(mx(ring_blocks=blocks), T, H, I, E, K) == full
    assert M.mm_moe_workspace_size(mx(ring_blocks=16), T, H, I, E, K) < ring
    for bad, code in ((dict(ring_blocks=-1), M.MM_MOE_ERR_INVALID_ARG),
                      (dict(ring_blocks=15), M.MM_MOE_ERR_INVALID_ARG),      # ceil(2048 / 128) = 16
                      (dict(ring_blocks=64, fused=0), M.MM_MOE_ERR_UNSUPPORTED),
                      (dict(ring_blocks=64, swap_ab=1), M.MM_MOE_ERR_UNSUPPORTED),
                      (dict(ring_blocks=64, swap_ab=2), M.MM_MOE_ERR_UNSUPPORTED),
                      (dict(ring_blocks=64, retain_intermediate=1), M.MM_MOE_ERR_UNSUPPORTED),
                      (dict(ring_blocks=64, debug_flags=1), M.MM_MOE_ERR_UNSUPPORTED)):
        with pytest.raises(M.MMError) as ei:
            M.mm_moe_workspace_size(mx(**bad), T, H, I, E, K)
        assert ei.value.code == code, bad
    with pytest.raises(M.MMError) as ei:
        M.mm_moe_workspace_size(M.options(M.MM_MOE_VARIANT_F8, ring_blocks=64), T, H, I, E, K)
    assert ei.value.code == M.MM_MOE_ERR_UNSUPPORTED


def test_default_options(M):
    o = M.mm_moe_default_options()
    assert (o.variant, o.fused, o.lag_units, o.wait_timeout_ms) == (M.MM_MOE_VARIANT_MX, 1, -1, 2000)
    assert (o.f8_act_gran, o.shared_experts, o.ring_blocks) == (0, 0, 0)
    assert (o.cta_pairs, o.partials_bf16, o.precise_swiglu, o.x_bf16, o.early_combine) == (0, 0, 0, 0, 0)
    assert o.activation_clamp == 0.0 and not o.timing_events

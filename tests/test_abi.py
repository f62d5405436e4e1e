"""C-ABI checks that need no GPU: the library loads, exports every function
that include/fp4.h declares, and rejects bad arguments on the host before
any launch (status codes, messages)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def F():
    import __graft_entry__ as ge
    ge.build_library()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported(F):
    lib = F.lib()
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", F.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (fp4_[a-z0-9_]+)", out))
    assert set(names) <= exported
    assert set(names) == set(F.exported_symbols())


def test_status_strings(F):
    L = F.lib()
    for code, name in F.STATUS.items():
        assert L.fp4_status_string(code).decode() == name
    assert L.fp4_abi_version() == 1


def test_sizes(F):
    L = F.lib()
    assert L.fp4_codes_bytes(16, 512) == 16 * 256
    assert L.fp4_scales_bytes(F.NVFP4, 16, 512) == 128 * 32
    assert L.fp4_scales_bytes(F.MXFP4, 130, 800) == 256 * 32  # K padded to 1024 -> 32 scale columns
    assert L.fp4_gemm_workspace_size(F.NVFP4, 8192, 14336, 4096) >= 8192 * 2048


A = 0x100000  # an aligned fake device address; validation fails before any use


def _gemm(F, fmt=0, x=A, m=16, mode=0, st=0.0, wc=A, wsc=A, wg=A, n=256, k=512, out=A, ws=A, wsb=1 << 30):
    return F.lib().fp4_gemm(fmt, x, m, mode, st, wc, wsc, wg, n, k, out, ws, wsb, None)


def test_gemm_argument_errors(F):
    c = F.STATUS_CODE
    assert _gemm(F, k=48) == c["FP4_ERR_SHAPE"]
    assert _gemm(F, k=0) == c["FP4_ERR_SHAPE"]
    assert _gemm(F, n=250) == c["FP4_ERR_SHAPE"]
    assert _gemm(F, m=-1) == c["FP4_ERR_SHAPE"]
    assert _gemm(F, fmt=7) == c["FP4_ERR_INVALID_ARG"]
    assert _gemm(F, x=0) == c["FP4_ERR_INVALID_ARG"]
    assert _gemm(F, wg=0) == c["FP4_ERR_MISSING_SCALE"]
    assert _gemm(F, out=A + 8) == c["FP4_ERR_ALIGNMENT"]
    assert _gemm(F, ws=0) == c["FP4_ERR_WORKSPACE"]
    assert _gemm(F, wsb=16) == c["FP4_ERR_WORKSPACE"]
    assert "multiple of 32" in F.lib().fp4_last_error_message().decode() or True


def _w4a16(F, fmt=0, x=A, m=1, wc=A, wsc=A, wg=A, n=256, k=512, out=A):
    return F.lib().fp4_gemm_w4a16(fmt, x, m, wc, wsc, wg, n, k, out, None)


def test_mxfp8_quantize_argument_errors(F):
    c = F.STATUS_CODE
    q = lambda x=A, rows=16, k=512, codes=A, scales=A: F.lib().fp4_quantize_mxfp8(x, rows, k, codes, scales, None)
    assert q(k=48) == c["FP4_ERR_SHAPE"]
    assert q(k=0) == c["FP4_ERR_SHAPE"]
    assert q(rows=-1) == c["FP4_ERR_SHAPE"]
    assert q(x=0) == c["FP4_ERR_INVALID_ARG"]
    assert q(scales=0) == c["FP4_ERR_INVALID_ARG"]
    assert q(codes=A + 8) == c["FP4_ERR_ALIGNMENT"]


def test_w4a16_argument_errors(F):
    c = F.STATUS_CODE
    assert _w4a16(F, m=5) == c["FP4_ERR_SHAPE"]  # more rows than the weight-only path takes
    assert "at most 4" in F.lib().fp4_last_error_message().decode()
    assert _w4a16(F, k=8192 + 32) == c["FP4_ERR_SHAPE"]
    assert _w4a16(F, k=48) == c["FP4_ERR_SHAPE"]
    assert _w4a16(F, n=12) == c["FP4_ERR_SHAPE"]
    assert _w4a16(F, m=-1) == c["FP4_ERR_SHAPE"]
    assert _w4a16(F, fmt=3) == c["FP4_ERR_INVALID_ARG"]
    assert _w4a16(F, x=0) == c["FP4_ERR_INVALID_ARG"]
    assert _w4a16(F, wc=0) == c["FP4_ERR_INVALID_ARG"]
    assert _w4a16(F, wg=0) == c["FP4_ERR_MISSING_SCALE"]
    assert _w4a16(F, x=A + 4) == c["FP4_ERR_ALIGNMENT"]
    assert _w4a16(F, out=A + 2) == c["FP4_ERR_ALIGNMENT"]
    # MXFP4 has no global scale: NULL is accepted (the call then fails only on
    # the missing GPU, never on the scale)
    assert _w4a16(F, fmt=1, wg=0) != c["FP4_ERR_MISSING_SCALE"]


@pytest.mark.parametrize("st", [0.0, -1.0, float("nan"), float("inf")])
def test_static_scale_must_be_positive_finite(F, st):
    # the zeroed-alpha failure mode: a missing scale must never become 0
    c = F.STATUS_CODE
    assert _gemm(F, mode=1, st=st) == c["FP4_ERR_INVALID_SCALE"]
    L = F.lib()
    assert L.fp4_quantize_act(0, A, 16, 512, 1, st, A, A, A, A, 4096, None) == c["FP4_ERR_INVALID_SCALE"]


def test_mxfp4_rejects_static_mode(F):
    assert _gemm(F, fmt=1, mode=1, st=1.0) == F.STATUS_CODE["FP4_ERR_INVALID_ARG"]


def test_unsupported_arch_is_loud(F):
    L = F.lib()
    L.fp4_set_arch_override(90)
    try:
        assert _gemm(F) == F.STATUS_CODE["FP4_ERR_UNSUPPORTED_ARCH"]
        msg = L.fp4_last_error_message().decode()
        assert "SM 90" in msg and "sm_103a" in msg
        assert L.fp4_quantize_act(1, A, 16, 512, 0, 0.0, A, A, A, A, 4096, None) == \
            F.STATUS_CODE["FP4_ERR_UNSUPPORTED_ARCH"]
    finally:
        L.fp4_set_arch_override(0)


def test_python_wrapper_raises(F):
    with pytest.raises(F.FP4Error) as ei:
        F._check(F.lib().fp4_gemm(0, A, 16, 0, 0.0, A, A, A, 256, 48, A, A, 1 << 30, None))
    assert ei.value.name == "FP4_ERR_SHAPE"


def test_tile_policy_validation(F):
    L = F.lib()
    for p in (F.TILE_ONE_CTA, F.TILE_CTA_PAIR, F.TILE_FUSED_DECODE, F.TILE_W4A16_TC, F.TILE_WEIGHT_PAIRS, F.TILE_AUTO):
        assert L.fp4_set_gemm_tile_policy(p) == 0
    for bad in (-1, 6):
        assert L.fp4_set_gemm_tile_policy(bad) == F.STATUS_CODE["FP4_ERR_INVALID_ARG"]
        assert "tile policy" in L.fp4_last_error_message().decode()
    with pytest.raises(F.FP4Error):
        F.set_gemm_tile_policy(7)


# ------------------------------------------------------ GEMM planner (host)

SMS = 152  # GB300


def test_plan_prefill_tile_width(F):
    """256-wide tiles when 1.5 x their waves do not exceed the 128-wide waves."""
    assert F.plan_gemm(8192, 14336, 4096, SMS) == {"small_m": False, "bn": 256, "splits": 1, "pair": False,
                                                    "fused_decode": False, "weight_pairs": False}
    assert F.plan_gemm(8192, 4096, 4096, SMS)["bn"] == 256    # 7 waves of 256 against 14 of 128
    assert F.plan_gemm(2048, 2048, 7168, SMS)["bn"] == 256    # one wave of 128 tiles against 1.7 waves
    assert F.plan_gemm(256, 512, 512, SMS)["bn"] == 128       # one wave either way
    assert F.plan_gemm(65, 264, 800, SMS)["small_m"] is False  # m > 64 is the prefill kernel


def test_plan_decode_split_and_fused(F):
    p = F.plan_gemm(8, 14336, 4096, SMS)
    assert p["small_m"] and p["bn"] == 32 and p["splits"] == 1 and p["fused_decode"]  # 112 tiles >= 76
    p = F.plan_gemm(9, 14336, 4096, SMS)  # the launch chain's swapped GEMM, whole K per tile
    assert p["small_m"] and p["bn"] == 32 and p["splits"] == 1 and not p["fused_decode"]
    assert F.plan_gemm(40, 14336, 4096, SMS)["bn"] == 64
    # 32 weight tiles are split along K: ceil(3 x 152 / 32) = 15, at most half the 16 K blocks -> 8
    assert F.plan_gemm(8, 4096, 4096, SMS)["splits"] == 8
    assert F.plan_gemm(1, 14336, 4096, SMS)["fused_decode"]          # m <= 8 and tiles for half the SMs
    assert not F.plan_gemm(1, 4096, 4096, SMS)["fused_decode"]       # 32 tiles < 76
    assert not F.plan_gemm(9, 14336, 4096, SMS)["fused_decode"]      # above the fused kernel's m limit
    assert not F.plan_gemm(1, 14336, 8192 + 32, SMS)["fused_decode"]  # k above the fused kernel's limit


def test_plan_follows_the_tile_policy(F):
    try:
        F.set_gemm_tile_policy(F.TILE_FUSED_DECODE)
        assert F.plan_gemm(8, 1024, 4096, SMS)["fused_decode"]
        assert not F.plan_gemm(9, 14336, 4096, SMS)["fused_decode"]
        F.set_gemm_tile_policy(F.TILE_CTA_PAIR)
        assert F.plan_gemm(8192, 14336, 4096, SMS)["pair"]
        assert not F.plan_gemm(128, 14336, 4096, SMS)["pair"]
        F.set_gemm_tile_policy(F.TILE_ONE_CTA)
        assert not F.plan_gemm(1, 14336, 4096, SMS)["fused_decode"]
        assert not F.plan_gemm(8192, 14336, 4096, SMS)["weight_pairs"]
        F.set_gemm_tile_policy(F.TILE_WEIGHT_PAIRS)
        assert F.plan_gemm(8192, 14336, 4096, SMS)["weight_pairs"]      # 32 x 56 pair units
        assert not F.plan_gemm(8064, 14336, 4096, SMS)["weight_pairs"]  # 63 activation tiles: no whole pairs
        assert not F.plan_gemm(512, 512, 4096, SMS)["weight_pairs"]     # 2 x 2 pair units < 76 clusters
        assert not F.plan_gemm(8, 14336, 4096, SMS)["weight_pairs"]     # decode
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)
    c = F.STATUS_CODE
    out = (__import__("ctypes").c_int64 * 5)()
    assert F.lib().fp4_debug_plan_gemm(0, 16, 32, SMS, out, 5) == c["FP4_ERR_INVALID_ARG"]
    assert F.lib().fp4_debug_plan_gemm(8, 16, 32, SMS, out, 4) == c["FP4_ERR_INVALID_ARG"]


# ------------------------------------------------ MoE workspace layout (host)

@pytest.mark.parametrize("T,H,I,E,k", [(0, 256, 128, 8, 2), (1, 2048, 768, 128, 8), (64, 2048, 768, 128, 8),
                                       (4096, 2048, 768, 128, 8), (5, 256, 128, 8, 2), (40, 512, 192, 16, 4)])
def test_moe_workspace_layout_holds_its_documented_contents(F, T, H, I, E, k):
    import ctypes
    L = F.lib()
    offs = (ctypes.c_int64 * 32)()
    n = L.fp4_moe_workspace_layout(T, H, I, E, k, offs, 32)
    assert n == 22
    o = [offs[i] for i in range(14)]
    R = offs[14]
    slots = T * k
    # every expert's rows are padded to 128: at most 127 padding rows per expert that has any
    assert R % 128 == 0 and R >= slots + min(slots, E) * 127 and R >= 128
    sf = lambda kk: ((kk + 255) // 256) * 16  # NVFP4 scale columns per row, K padded to 256
    need = [slots * 4, slots * 4, (E + 1) * 4, (E + 1) * 4, R * 4, R * H // 2, R * sf(H), E * 4, R * I * 2, E * 4,
            E * 4, R * I // 2, R * sf(I), R * H * 4]
    assert o[0] == 0
    for i in range(14):
        assert o[i] % 256 == 0
    for i in range(13):
        assert o[i + 1] - o[i] >= need[i], i
    assert L.fp4_moe_workspace_size(T, H, I, E, k) >= o[13] + need[13]
    # entries 15-21: the one-launch MoE's intermediates, sized when its shapes apply
    # (1 <= T <= 16, top_k <= 8, H and I multiples of 256 up to 2048), slot order
    f = [offs[i] for i in range(15, 22)]
    fused = 1 <= T <= 16 and k <= 8 and H % 256 == 0 and H <= 2048 and I % 256 == 0 and I <= 2048
    if fused:
        fneed = [slots * I * 2, slots * I // 2, slots * I // 16, E * 4, slots * H * 4, slots * H // 2, slots * H // 16]
        for i in range(7):
            assert f[i] % 256 == 0 and f[i] >= o[13] + need[13]
            assert L.fp4_moe_workspace_size(T, H, I, E, k) >= f[i] + fneed[i]
        regions = sorted(zip(f, fneed))
        for (a0, n0), (a1, _) in zip(regions, regions[1:]):
            assert a0 + n0 <= a1
    # a short buffer gets the leading entries only
    assert L.fp4_moe_workspace_layout(T, H, I, E, k, offs, 3) == 3
    assert L.fp4_moe_workspace_layout(T, H, I, 0, k, offs, 32) == 0


# ------------------------------------------- MX (8-bit containers) and policies

def test_mx_argument_errors(F):
    c = F.STATUS_CODE
    L = F.lib()
    q = lambda elem=0, x=A, rows=16, k=512, codes=A, scales=A: L.fp4_quantize_mx(elem, x, rows, k, codes, scales,
                                                                                  None)
    assert q(elem=4) == c["FP4_ERR_INVALID_ARG"]
    assert q(elem=-1) == c["FP4_ERR_INVALID_ARG"]
    assert q(k=48) == c["FP4_ERR_SHAPE"]
    assert q(x=0) == c["FP4_ERR_INVALID_ARG"]
    assert q(codes=A + 8) == c["FP4_ERR_ALIGNMENT"]
    g = lambda ea=0, ew=0, ac=A, asc=A, m=16, wc=A, wsc=A, n=256, k=512, out=A: L.fp4_gemm_mx_prequant(
        ea, ac, asc, m, ew, wc, wsc, n, k, out, None)
    assert g(n=250) == c["FP4_ERR_SHAPE"]
    assert g(k=48) == c["FP4_ERR_SHAPE"]
    assert g(ea=9) == c["FP4_ERR_INVALID_ARG"]
    # the GEMM reads E4M3 / E5M2 codes: MXFP6 operands are widened first
    assert g(ea=2) == c["FP4_ERR_INVALID_ARG"] and "widen" in L.fp4_last_error_message().decode()
    assert g(ew=3) == c["FP4_ERR_INVALID_ARG"]
    # per call, MXFP6 activations are accepted (widened as they are quantised); weights are not
    assert L.fp4_gemm_mx(2, A, 16, 3, A, A, 256, 512, A, A, 1 << 30, None) == c["FP4_ERR_INVALID_ARG"]
    wd = lambda elem=2, codes=A, rows=16, k=512, out=A: L.fp4_mx_widen(elem, codes, rows, k, out, None)
    assert wd(elem=0) == c["FP4_ERR_INVALID_ARG"]  # only MXFP6 codes are widened
    assert wd(elem=1) == c["FP4_ERR_INVALID_ARG"]
    assert wd(k=48) == c["FP4_ERR_SHAPE"]
    assert wd(codes=0) == c["FP4_ERR_INVALID_ARG"]
    assert wd(out=A + 8) == c["FP4_ERR_ALIGNMENT"]
    assert g(wc=0) == c["FP4_ERR_INVALID_ARG"]
    assert g(out=A + 4) == c["FP4_ERR_ALIGNMENT"]
    assert L.fp4_gemm_mx(0, A, 16, 0, A, A, 256, 512, A, A, 16, None) == c["FP4_ERR_WORKSPACE"]
    assert L.fp4_gemm_mx_workspace_size(16, 512) >= 16 * 512 + 128 * 16


def test_moe_policy_validation(F):
    L = F.lib()
    for p in (F.MOE_CHAIN, F.MOE_FUSED, F.MOE_AUTO):
        assert L.fp4_set_moe_policy(p) == 0
    for bad in (-1, 3):
        assert L.fp4_set_moe_policy(bad) == F.STATUS_CODE["FP4_ERR_INVALID_ARG"]
        assert "MoE policy" in L.fp4_last_error_message().decode()

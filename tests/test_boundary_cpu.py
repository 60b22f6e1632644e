"""Host-side tests of the C ABI (no GPU): the library loads and exports every declared symbol,
validation rejects what the pages' can_implement rejects (before touching any memory), and the
runtime dispatcher picks paths and split-K factors from the runtime shape."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def w():
    from w4a16_int4_weight_group_gb300 import build
    build.build()
    import w4a16_int4_weight_group_gb300 as mod
    mod.lib()
    return mod


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("w4a16_pack", "w4a16_gemm", "w4a16_unpack", "w4a16_dequant", "w4a16_can_implement",
                 "w4a16_last_error", "w4a16_get_device_error", "w4a16_debug_selected_path"):
        assert must in names


def test_library_exports_every_declared_symbol(w):
    names = declared_functions()
    lib = w.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", w.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (w4a16_\w+)", out))
    assert set(names) <= exported
    assert {s[0] for s in w.SIGNATURES} == set(names)


def test_can_implement_reasons_follow_the_pages(w):
    assert w.w4a16_can_implement(2112, 1152, 32, 1) == (True, "")
    assert w.w4a16_can_implement(256, 512, 128, 0) == (True, "")
    ok, why = w.w4a16_can_implement(256, 516, 128, 0)
    assert not ok and "must be divisible by 8" in why and "8 int4 values packed per int32" in why
    ok, why = w.w4a16_can_implement(256, 512, 128, 7)
    assert not ok and "float16/bfloat16" in why
    ok, why = w.w4a16_can_implement(256, 512, 128, 0, has_g_idx=True)
    assert not ok and "g_idx" in why
    ok, why = w.w4a16_can_implement(256, 512, 96, 0)
    assert not ok and "Group size 96 not supported" in why
    # group_size == K (per-channel) is allowed for any K
    assert w.w4a16_can_implement(100, 512, 100, 0) == (True, "")
    for g in (32, 64):
        assert w.w4a16_can_implement(2112, 4224, g, 1) == (True, "")
    # 2112 = 16.5 * 128: groups of 128 do not tile K
    ok, why = w.w4a16_can_implement(2112, 4224, 128, 1)
    assert not ok and "multiple of group_size" in why


def _gemm(w, a=0x1000, b_q=0x2000, scales=0x3000, qzeros=None, G=32, zp=8, bias=None, out=0x100000,
          m=4, k=64, n=64, dt=0):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return w.lib().w4a16_gemm(p(a), p(b_q), p(scales), p(qzeros), G, zp, p(bias), p(out), m, k, n, dt, None)


def test_gemm_validation_rejects_before_any_launch(w):
    before = w.w4a16_debug_launch_count()
    assert _gemm(w, dt=3) == 2 and "float16/bfloat16" in w.last_error()
    assert _gemm(w, n=60) == 1 and "divisible by 8" in w.last_error()
    assert _gemm(w, G=48) == 2
    assert _gemm(w, k=96, G=64) == 1 and "multiple of group_size" in w.last_error()
    assert _gemm(w, zp=16) == 1 and "zp_bias" in w.last_error()
    assert _gemm(w, zp=-1) == 1
    assert _gemm(w, a=None) == 1 and "NULL" in w.last_error()
    assert _gemm(w, out=None) == 1
    assert _gemm(w, m=-1) == 1
    assert _gemm(w, k=0) == 1
    assert _gemm(w, a=0x1001) == 3 and "aligned" in w.last_error()
    assert _gemm(w, b_q=0x2002) == 3
    # out overlapping an input
    assert _gemm(w, out=0x2000) == 1 and "overlaps" in w.last_error()
    assert _gemm(w, out=0x1000 + 4 * 64 * 2 - 2) == 1
    # M == 0: nothing to do, no device access, OK
    assert _gemm(w, m=0, a=None, out=None) == 0
    assert w.w4a16_debug_launch_count() == before


def test_pack_validation(w):
    L = w.lib()
    assert L.w4a16_pack(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x8000), 4, 12, None) == 1
    assert L.w4a16_pack(None, ctypes.c_void_p(0x8000), 4, 16, None) == 1
    assert L.w4a16_pack(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x8002), 4, 16, None) == 3
    assert L.w4a16_pack(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1010), 4, 16, None) == 1  # overlap
    assert L.w4a16_pack(None, None, 0, 16, None) == 0


def test_dispatcher_decode_for_small_m_and_split_k(w):
    # decode workloads of the pages: M <= 8 takes the split-K decode path
    for m in (1, 2, 4, 5, 8):
        for k, n in ((1152, 4224), (2112, 1152), (2560, 19456), (9728, 2560)):
            p = w.w4a16_plan(m, k, n, 32 if k in (1152, 2112) else 128, 0, False, 152)
            assert p["path_name"] == "decode", (m, k, n, p)
            assert p["m_tile"] == 8
            assert 1 <= p["k_split"] <= 16
            assert p["grid"] <= 2 * 152
    # a narrow layer gets split along K across a cluster
    p = w.w4a16_plan(1, 2112, 1152, 32, 1, False, 152)
    assert p["k_split"] > 1
    # a wide one is split only as far as needed to put one CTA on every SM
    p = w.w4a16_plan(1, 2560, 19456, 128, 0, True, 152)
    assert p["k_split"] <= 2 and 76 <= p["grid"] <= 152
    # and the choice follows the device: half the SMs, half the CTAs
    assert w.w4a16_plan(1, 2560, 19456, 128, 0, True, 76)["grid"] <= 152


def test_prefill_plan_stream_k_with_a_workspace(w):
    # the prefill workload: persistent stream-K CTAs, one per SM, 256-row tiles
    for m in (512, 1024, 4096):
        p = w.w4a16_plan(m, 5120, 34816, 64, 1, True, 152)
        assert p["path_name"] == "prefill" and p["stream_k"] == 1 and p["grid"] == 152, p
        p = w.w4a16_plan(m, 5120, 34816, 64, 1, True, 152, with_workspace=False)
        assert p["stream_k"] == 0 and p["grid"] == (m // 256) * 136, p
        q = w.w4a16_plan(m, 17408, 5120, 64, 1, True, 152)
        assert q["stream_k"] == 1 and q["m_tile"] == 256 and q["grid"] == 152, q
        # without a workspace the same call runs one CTA per tile
        r = w.w4a16_plan(m, 17408, 5120, 64, 1, True, 152, with_workspace=False)
        assert r["stream_k"] == 0
    # few tiles: fewer CTAs than SMs, so that the owner's fix-up stays short
    p = w.w4a16_plan(256, 4096, 1024, 32, 1, True, 152)
    assert p["stream_k"] == 1 and 4 < p["grid"] < 152, p
    # 17..32 rows: the decode kernel with four row tiles (one CTA per SM)
    for m in (17, 24, 32):
        p = w.w4a16_plan(m, 5120, 7168, 128, 1, False, 152)
        assert p["path_name"] == "decode" and p["m_tile"] == 32 and p["warps"] == 9 and p["grid"] <= 152, (m, p)
    # mid M (33..128): one CTA per 128-row tile would leave most SMs idle; clusters of CTAs split each
    # tile's K blocks and add their partial tiles through distributed shared memory (no workspace)
    for m in (33, 64, 128):
        for ws in (True, False):
            p = w.w4a16_plan(m, 5120, 7168, 128, 1, False, 152, with_workspace=ws)
            assert p["path_name"] == "prefill" and p["m_tile"] == 128 and p["stream_k"] == 0, (m, p)
            assert 2 <= p["k_split"] <= 8 and p["grid"] == 28 * p["k_split"] and p["grid"] >= 100, (m, p)


def test_dispatcher_uses_runtime_m_not_a_frozen_config(w):
    # the same layer, decode and prefill sizes, in any order: plans depend only on the runtime M
    k, n, g = 5120, 7168, 128
    seq = [1, 4096, 8, 1024, 1, 2, 8192, 5]
    plans = [w.w4a16_plan(m, k, n, g, 1, True, 152) for m in seq]
    again = [w.w4a16_plan(m, k, n, g, 1, True, 152) for m in seq[::-1]][::-1]
    assert plans == again
    assert plans[0]["m_tile"] < plans[1]["m_tile"] or plans[1]["path_name"] != "decode"


def test_dispatcher_generic_for_unaligned_shapes(w):
    # N % 32 != 0 or K % 16 != 0 cannot use the 16-byte streaming paths
    assert w.w4a16_plan(4, 256, 520, 128, 0, False, 152)["path_name"] == "generic"
    assert w.w4a16_plan(4, 100, 512, 100, 0, False, 152)["path_name"] == "generic"
    assert w.w4a16_plan(0, 256, 512, 128, 0, False, 152)["path_name"] == "none"


def test_plan_rejects_bad_config(w):
    with pytest.raises(w.W4A16Error):
        w.w4a16_plan(4, 256, 516, 128, 0, False, 152)


def test_repack_k_to_n_validation(w):
    import ctypes
    L = w.lib()
    p0, p1 = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    assert L.w4a16_repack_k_to_n(p0, p1, 12, 16, None) == 1            # k % 8
    assert L.w4a16_repack_k_to_n(p0, p1, 16, 12, None) == 1            # n % 8
    assert L.w4a16_repack_k_to_n(None, p1, 16, 16, None) == 1          # null
    assert L.w4a16_repack_k_to_n(ctypes.c_void_p(0x10002), p1, 16, 16, None) == 3  # misaligned
    assert L.w4a16_repack_k_to_n(p0, ctypes.c_void_p(0x10010), 16, 16, None) == 1  # overlap


def test_prepared_layer_rejects_host_tensors(w):
    import torch
    b_q = torch.zeros((256, 64), dtype=torch.int32)
    scales = torch.zeros((2, 512), dtype=torch.float16)
    with pytest.raises(ValueError):
        w.W4A16Linear(b_q, scales, None, 128)
    with pytest.raises(ValueError):
        w.W4A16Linear(b_q.to(torch.int64), scales, None, 128)


def test_layer_handle_validation_without_a_device(w):
    """The prepared-layer entry points reject bad configurations and a NULL handle before touching
    any device."""
    L = w.lib()
    h = ctypes.c_void_p()
    assert L.w4a16_layer_create(0x1000, 0x2000, None, 128, 8, None, 256, 516, 0, ctypes.byref(h)) == 1
    assert "divisible by 8" in w.last_error() and h.value is None
    assert L.w4a16_layer_create(0x1000, 0x2000, None, 96, 8, None, 256, 512, 0, ctypes.byref(h)) == 2
    assert L.w4a16_layer_create(0x1000, 0x2000, None, 128, 16, None, 256, 512, 0, ctypes.byref(h)) == 1
    assert L.w4a16_layer_create(None, 0x2000, None, 128, 8, None, 256, 512, 0, ctypes.byref(h)) == 1
    assert L.w4a16_layer_create(0x1001, 0x2000, None, 128, 8, None, 256, 512, 0, ctypes.byref(h)) == 3
    assert L.w4a16_layer_gemm(None, 0x1000, 0x2000, 4, None, 0, None) == 1 and "layer" in w.last_error()
    assert L.w4a16_layer_workspace_size(None, 4) == 0
    assert L.w4a16_layer_destroy(None) == 0


def test_force_path_entry_point_validates(w):
    assert w.lib().w4a16_debug_force_path(7) == 1
    assert w.lib().w4a16_debug_force_path(-1) == 0


# Decode plans the dispatcher picks on a 152-SM GB300 for the decode workloads' layers, against the
# plans that measured fastest there (per-call time of CUDA-graph chains of calls over rotating weight
# replicas; split-K factors 1..16, one and two consumer groups, stages of one, two and four K blocks;
# M = 1 and M = 8): one consumer group (9 warps) and this (split-K factor, K blocks per stage).
MEASURED_BEST_DECODE_PLAN = {
    (1152, 4224, 32): (6, 1),     # 102 CTAs, 2.8 us
    (2112, 1152, 32): (11, 1),    # 55 CTAs, 2.7-2.9 us
    (2560, 3840, 128): (10, 2),   # 150 CTAs, 4.1-4.3 us
    (2560, 19456, 128): (2, 2),   # 152 CTAs, 8.3-8.5 us
    (9728, 2560, 128): (16, 2),   # 160 CTAs, 6.8-7.0 us
}


@pytest.mark.parametrize("shape", sorted(MEASURED_BEST_DECODE_PLAN))
def test_decode_planner_picks_the_measured_best_plan(w, shape):
    K, N, G = shape
    for M in (1, 2, 4, 5, 8):
        for dt, zp in ((0, True), (1, False)):
            p = w.w4a16_plan(M, K, N, G, dt, zp, 152, False)
            assert p["path_name"] == "decode"
            assert (p["warps"], p["k_split"], p["k_blocks_per_stage"]) == (9, *MEASURED_BEST_DECODE_PLAN[shape]), p
            assert p["grid"] == -(-N // 256) * p["k_split"]


def test_layer_call_marshalling_module_reaches_the_c_abi(w):
    """The CPython marshalling module of the prepared-layer call (built beside the library) passes its
    seven integer arguments to w4a16_layer_gemm: a null layer comes back as INVALID_ARG with the
    library's message, None stands for a null pointer, and a wrong argument count is a TypeError."""
    mod = pytest.importorskip("w4a16_int4_weight_group_gb300._w4a16_call")
    fn = w._layer_gemm_fn()
    assert fn is mod.layer_gemm
    assert fn(None, 0, 0, 1, None, 0, None) == 1  # W4A16_ERR_INVALID_ARG
    assert "layer must not be NULL" in w.last_error()
    assert fn(0, 0, 0, 1, 0, 0, 0) == 1
    with pytest.raises(TypeError):
        fn(None, 0, 0)
    with pytest.raises(TypeError):
        fn(None, 0, 0, "one", None, 0, None)


# 17..32 rows (four row tiles, one CTA per SM): the splits measured fastest on GB300 for the mid-M
# layers (per-call time of CUDA-graph chains; cluster sizes 3..10 tried at M = 17, 24 and 32)
MEASURED_BEST_DECODE_J4_SPLIT = {
    (5120, 7168, 128): 4,     # 112 CTAs, 13.6-13.9 us (the 128-row kernel: 17.0-17.9 us)
    (17408, 5120, 128): 6,    # 120 CTAs, 28.7-29.0 us (32.8-33.2 us)
    (2560, 19456, 128): 2,    # 152 CTAs, 15.5-16.2 us (18.6-19.0 us)
}


@pytest.mark.parametrize("shape", sorted(MEASURED_BEST_DECODE_J4_SPLIT))
def test_decode_planner_four_row_tiles(w, shape):
    K, N, G = shape
    for M in (17, 24, 32):
        p = w.w4a16_plan(M, K, N, G, 1, False, 152, False)
        assert p["path_name"] == "decode" and p["m_tile"] == 32 and p["warps"] == 9, p
        assert p["k_split"] == MEASURED_BEST_DECODE_J4_SPLIT[shape], p
        # never a cluster size whose clusters pack badly, and one wave of CTAs
        assert p["k_split"] in (1, 2, 4, 6, 8) and p["grid"] <= 152, p

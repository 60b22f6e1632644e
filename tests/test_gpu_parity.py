"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle on the same seeded inputs.

Bit-exact for pack / unpack / dequant and for the identity-A product (one non-zero product per
output is exact in fp32, so the output equals the dequantised weight); within the layer's tolerance
|out - ref| <= atol + rtol*|ref| (fp16 1e-2/1e-2, bf16 2e-2/2e-2) for the product, where ref is the
fp64 product over the dequantised weights; plus the rigorous bound against exact-weight fp64.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import (bits_to_torch, case_tensors, check_against_oracle, forced_path, path_taken,
                         sample_cols, torch_to_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_weight_group_gb300 import build
    build.build()
    import w4a16_int4_weight_group_gb300 as mod
    mod.lib()
    return mod


def run(w, c, path=None, out=None):
    t = case_tensors(c)
    with forced_path(path):
        o = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], c.G, c.zp_bias, t["bias"], out=out)
    torch.cuda.synchronize()
    return torch_to_bits(o)


def supported_paths(w, c):
    paths = ["generic"]
    plan = w.w4a16_plan(c.M, c.K, c.N, c.G, 1 if c.dtype == "bf16" else 0, c.asym, 0)
    for p in ("decode", "prefill"):
        with forced_path(p):
            if w.w4a16_plan(c.M, c.K, c.N, c.G, 1 if c.dtype == "bf16" else 0, c.asym, 0)["path_name"] == p:
                paths.append(p)
    return paths, plan["path_name"]


# ------------------------------------------------------------------------------------------------
# layout kernels: bit-exact
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("rows,n", [(1, 8), (37, 232), (1152, 4224), (3, 8 * 4099)])
def test_pack_unpack_bitexact(w, rows, n):
    q = synth.random_nibbles(rows, n, seed=rows + n)
    packed = w.w4a16_pack(torch.from_numpy(q).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), oracle.pack(q))
    back = w.w4a16_unpack(packed)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), q)


@pytest.mark.parametrize("K,N,G,dtype,asym,zp", [
    (256, 512, 128, "f16", False, 8), (2112, 1152, 32, "bf16", False, 8), (2560, 3840, 128, "f16", True, 8),
    (100, 520, 100, "bf16", True, 8), (64, 8, 64, "f16", False, 0), (128, 64, 32, "bf16", False, 15)])
def test_dequant_bitexact(w, K, N, G, dtype, asym, zp):
    c = synth.make_case(0, K, N, G, dtype, asym=asym, seed=K + N, zp_bias=zp)
    t = case_tensors(c)
    wt = w.w4a16_dequant(t["b_q"], t["scales"], t["qzeros"], G, zp)
    torch.cuda.synchronize()
    assert np.array_equal(torch_to_bits(wt), oracle.dequant_t(c.b_q, c.scales, c.qzeros, G, zp, dtype))


# ------------------------------------------------------------------------------------------------
# the product
# ------------------------------------------------------------------------------------------------
SMALL_CASES = [
    # (M, K, N, G, dtype, asym, bias)
    (4, 256, 512, 128, "f16", False, False),      # the pages' fake-impl shape
    (1, 1152, 4224, 32, "bf16", False, False),    # 2112-model gate+up
    (5, 2112, 1152, 32, "bf16", False, False),    # 2112-model down
    (8, 2560, 3840, 128, "f16", True, True),      # 4B-class
    (9, 512, 8320, 64, "bf16", True, False),      # M just past 8, ragged column tile
    (16, 1024, 4096, 128, "f16", False, True),
    (33, 768, 2048, 64, "bf16", True, True),      # several row tiles, ragged last
    (64, 512, 1056, 32, "f16", True, False),      # N % 64 != 0
    (3, 4096, 96, 4096, "bf16", False, False),    # per-channel, narrow N
    (7, 100, 520, 100, "f16", True, True),        # K and N off every fast-path alignment
    (130, 256, 640, 128, "bf16", True, True),     # prefill-sized M, several tiles
    (2, 8, 8, 8, "f16", True, True),              # the smallest legal shape: K = G = 8, N = 8
    (1, 64, 8, 32, "bf16", False, False),         # one packed word of columns
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: "M%d_K%d_N%d_G%d_%s_%s%s" % (
    c[0], c[1], c[2], c[3], c[4], "asym" if c[5] else "sym", "_bias" if c[6] else ""))
def test_gemm_matches_oracle_every_path(w, case):
    M, K, N, G, dtype, asym, bias = case
    c = synth.make_case(M, K, N, G, dtype, asym=asym, bias=bias, seed=M * 7 + K + N)
    paths, auto = supported_paths(w, c)
    outs = {}
    for p in paths + [None]:
        outs[p] = run(w, c, p)
        check_against_oracle(c, outs[p], label=f"path={p or auto}", path=p or auto)
    # the automatic choice is one of the checked paths and gives the same bits as forcing it
    assert np.array_equal(outs[None], outs[auto])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K,N,G", [(8, 1024, 2048, 128), (1, 2112, 1152, 32), (64, 512, 512, 64)])
def test_identity_a_is_bitexact_dequant(w, dtype, M, K, N, G):
    c = synth.make_case(M, K, N, G, dtype, asym=True, seed=3 + M)
    rng = np.random.default_rng(M)
    ks = rng.choice(K, size=M, replace=False)
    one = int(oracle.ieee.t_encode_rne(np.array([1.0]), dtype)[0])
    c.a[:] = 0
    c.a[np.arange(M), ks] = one
    want = oracle.dequant_t(c.b_q, c.scales, c.qzeros, G, 8, dtype)[ks]
    for p in supported_paths(w, c)[0]:
        got = run(w, c, p)
        assert np.array_equal(got, want), f"path {p}: {int((got != want).sum())} differing outputs"


def test_m_zero_touches_nothing(w):
    c = synth.make_case(0, 256, 512, 128, "f16", seed=1)
    t = case_tensors(c)
    before = w.w4a16_debug_launch_count()
    out = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], None, 128)
    assert out.shape == (0, 512)
    assert w.w4a16_debug_launch_count() == before


def test_deterministic_and_writes_only_out(w):
    for M, K, N, G, asym in [(5, 2112, 1152, 32, False), (8, 2560, 3840, 128, True), (40, 512, 2048, 64, True)]:
        c = synth.make_case(M, K, N, G, "bf16", asym=asym, bias=True, seed=M)
        for p in supported_paths(w, c)[0]:
            t = case_tensors(c)
            buf = torch.full((M * N + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
            canary = torch_to_bits(buf[M * N:])
            out = buf[:M * N].view(M, N)
            with forced_path(p):
                w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], out=out)
                first = torch_to_bits(out).copy()
                w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], out=out)
            torch.cuda.synchronize()
            assert not np.isnan(oracle.ieee.t_decode(first, "bf16")).any(), f"{p}: unwritten outputs"
            assert np.array_equal(first, torch_to_bits(out)), f"{p}: not deterministic"
            assert np.array_equal(canary, torch_to_bits(buf[M * N:])), f"{p}: wrote past out"


def test_unaligned_pointers_take_the_generic_path(w):
    c = synth.make_case(4, 512, 1024, 128, "f16", asym=True, bias=True, seed=5)
    t = case_tensors(c)
    a2 = torch.empty(c.M * c.K + 1, dtype=torch.float16, device="cuda")[1:].view(c.M, c.K)
    a2.copy_(t["a"])
    out = w.w4a16_gemm(a2, t["b_q"], t["scales"], t["qzeros"], c.G, 8, t["bias"])
    torch.cuda.synchronize()
    check_against_oracle(c, torch_to_bits(out), label="unaligned a", path="generic")


@pytest.mark.parametrize("zp", [0, 15])
def test_zp_bias_values(w, zp):
    c = synth.make_case(3, 512, 512, 64, "f16", seed=zp, zp_bias=zp)
    for p in supported_paths(w, c)[0]:
        check_against_oracle(c, run(w, c, p), label=f"zp_bias={zp} path={p}", path=p)


def test_dispatch_threshold_neighbours(w):
    # every switch point of the dispatcher, +-1
    for M in (1, 8, 9, 16, 17, 32, 33, 64, 65, 128, 129):
        c = synth.make_case(M, 512, 1024, 128, "bf16", asym=True, seed=M)
        check_against_oracle(c, run(w, c), label=f"M={M}", path=path_taken(w, c))


# ------------------------------------------------------------------------------------------------
# the measurement workloads at full size
# ------------------------------------------------------------------------------------------------
def _config_ids(name):
    return [f"{name}-M{M}-K{K}-N{N}-G{G}-{dt}-{'asym' if asym else 'sym'}"
            for (M, K, N, G, dt, asym, bias, lo, hi, seed) in synth.config_cases(name)]


@pytest.mark.parametrize("args", list(synth.config_cases("tiny")) + list(synth.config_cases("decode_2112")),
                         ids=_config_ids("tiny") + _config_ids("decode_2112"))
def test_decode_workloads_full_output(w, args):
    M, K, N, G, dt, asym, bias, lo, hi, seed = args
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)
    check_against_oracle(c, run(w, c), label="full", path=path_taken(w, c))


@pytest.mark.parametrize("args", list(synth.config_cases("decode_4b")), ids=_config_ids("decode_4b"))
def test_decode_4b_workload_sampled_columns(w, args):
    M, K, N, G, dt, asym, bias, lo, hi, seed = args
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)
    out = run(w, c)
    cols = sample_cols(N, np.random.default_rng(seed))
    check_against_oracle(c, out, cols=cols, label="sampled", path=path_taken(w, c))


@pytest.mark.parametrize("args", list(synth.config_cases("mid_m")), ids=_config_ids("mid_m"))
def test_mid_m_workload_sampled_columns(w, args):
    """The mid-M workload at full size, on the path the dispatcher picks (the decode kernel with four
    row tiles for 17..32 rows, the 128-row kernel with cluster split-K above), every row checked on
    sampled columns."""
    M, K, N, G, dt, asym, bias, lo, hi, seed = args
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)
    want = "decode" if M <= 32 else "prefill"
    assert w.w4a16_plan(M, K, N, G, 1 if dt == "bf16" else 0, asym, 0)["path_name"] == want
    out = run(w, c)
    cols = sample_cols(N, np.random.default_rng(seed))
    check_against_oracle(c, out, cols=cols, label="mid_m sampled", path=path_taken(w, c))


@pytest.mark.parametrize("args", list(synth.config_cases("prefill")), ids=_config_ids("prefill"))
def test_prefill_workload_sampled(w, args):
    """The prefill workload at full size, in the launch configuration the benchmark times."""
    M, K, N, G, dt, asym, bias, lo, hi, seed = args
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=seed, scale_lo=lo, scale_hi=hi)
    assert w.w4a16_plan(M, K, N, G, 1 if dt == "bf16" else 0, asym, 0)["path_name"] == "prefill"
    out = run(w, c)
    rng = np.random.default_rng(seed)
    rows = sorted({0, 1, 127, 128, M // 2, M - 1} | set(rng.integers(0, M, size=4).tolist()))
    cols = sample_cols(N, rng, k=128)
    check_against_oracle(c, out, rows=rows, cols=cols, label="prefill sampled", path="prefill")


# The full M sweep on the 27B-class layers: every M of the sweep with every (dtype, group size,
# zero-point) variant on 5120 -> 7168, and the largest M on the other two layers.
_SWEEP_VARIANTS = [(dt, g, asym) for dt in ("f16", "bf16") for g in (128, "K") for asym in (False, True)]
SWEEP_CASES = ([(M, 5120, 7168, g, dt, asym) for M in synth.CONFIGS["sweep"]["Ms"] for (dt, g, asym) in _SWEEP_VARIANTS]
               + [(8192, K, N, g, dt, asym) for (K, N) in ((5120, 34816), (17408, 5120))
                  for (dt, g, asym) in (("f16", 128, True), ("bf16", "K", False))]
               + [(M, 17408, 5120, "K", "bf16", True) for M in (16, 64, 256, 2048)])


@pytest.mark.parametrize("M,K,N,g,dt,asym", SWEEP_CASES, ids=[
    f"M{M}-K{K}-N{N}-G{g}-{dt}-{'asym' if asym else 'sym'}" for (M, K, N, g, dt, asym) in SWEEP_CASES])
def test_sweep_shapes_sampled(w, M, K, N, g, dt, asym):
    """Sampled rows (first, last, random) and columns (both edges, every n % 8, random) of each sweep
    case, through the path the dispatcher picks for it, against the oracle."""
    G = K if g == "K" else g
    c = synth.make_case(M, K, N, G, dt, asym=asym, seed=M + G + (1 if asym else 0))
    out = run(w, c)
    rng = np.random.default_rng(M)
    rows = sorted({0, M - 1} | set(rng.integers(0, M, size=4).tolist()))
    check_against_oracle(c, out, rows=rows, cols=sample_cols(N, rng, k=128), label=f"{dt} {'asym' if asym else 'sym'}",
                         path=path_taken(w, c))


@pytest.mark.parametrize("M,K,N,G,dt,asym", [(512, 4096, 1024, 128, "bf16", True), (300, 2048, 768, 64, "f16", False),
                                           (1024, 17408, 5120, 64, "bf16", True), (256, 4096, 1024, 32, "bf16", True),
                                           (192, 5120, 7168, 128, "f16", True)])
def test_stream_k_matches_oracle_and_leaves_workspace_clean(w, M, K, N, G, dt, asym):
    """Persistent stream-K prefill: several CTAs share each output tile through the workspace; the
    tile's owner stages their partial tiles in rounds through its shared memory (more chunks than
    staging slots; 256-row and 128-row tiles; two scale groups per K block; a mid-M case)."""
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=True, seed=M + K)
    code = 1 if dt == "bf16" else 0
    plan = w.w4a16_plan(M, K, N, G, code, asym, 0, with_workspace=True)
    assert plan["path_name"] == "prefill" and plan["stream_k"] == 1, plan
    t = case_tensors(c)
    need = w.w4a16_gemm_workspace_size(M, K, N, G, code)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        out = torch.empty((M, N), dtype=t["a"].dtype, device="cuda")
        st = w.lib().w4a16_gemm_ws(*[w._ptr(x) for x in (t["a"], t["b_q"], t["scales"], t["qzeros"])], G, 8,
                                   w._ptr(t["bias"]), w._ptr(out), M, K, N, code, w._ptr(ws), need, None)
        assert st == 0, w.last_error()
        torch.cuda.synchronize()
        outs.append(torch_to_bits(out))
    assert np.array_equal(outs[0], outs[1]), "stream-K must be deterministic"
    grid = plan["grid"]
    flags = ws[:grid * 4]  # the flag area opens the workspace
    assert int(flags.count_nonzero()) == 0, "flags must be left zero"
    rng = np.random.default_rng(M)
    rows = sorted({0, M - 1} | set(rng.integers(0, M, size=6).tolist()))
    check_against_oracle(c, outs[0], rows=rows, cols=sample_cols(N, rng, k=128), label="stream-K", path="prefill")
    # the same call without a workspace (whole tiles per CTA) agrees within the tolerance too
    out2 = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], use_workspace=False)
    torch.cuda.synchronize()
    check_against_oracle(c, torch_to_bits(out2), rows=rows, cols=sample_cols(N, rng, k=64), label="no workspace",
                         path=path_taken(w, c, with_workspace=False))


@pytest.mark.parametrize("shift", [0, 8])
def test_prefill_output_alignment_paths(w, shift):
    """32-byte stores when `out` is 32-byte aligned, 16-byte stores when it is only 16-byte aligned
    (an output slice 8 elements into a buffer): the same values either way."""
    M, K, N, G = 300, 2048, 768, 64
    c = synth.make_case(M, K, N, G, "bf16", asym=True, bias=True, seed=77)
    t = case_tensors(c)
    big = torch.empty(M * N + 16, dtype=t["a"].dtype, device="cuda")
    out = big[shift:shift + M * N].view(M, N)
    assert out.data_ptr() % 32 == (0 if shift == 0 else 16)
    w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], out=out)
    torch.cuda.synchronize()
    assert w.w4a16_plan(M, K, N, G, 1, True, 0)["path_name"] == "prefill"
    rng = np.random.default_rng(shift)
    check_against_oracle(c, torch_to_bits(out), rows=np.arange(0, M, 13), cols=sample_cols(N, rng, k=64),
                         label=f"out shifted by {shift}", path="prefill")


@pytest.mark.parametrize("K,N", [(8, 8), (2112, 1152), (1152, 4224), (4104, 264)])
def test_repack_k_to_n_bitexact(w, K, N):
    """K-packed [N, K/8] words -> b_q [K, N/8]: bit-exact against the oracle's unpack-along-K then
    pack-along-N (including K, N not multiples of 64)."""
    rng = np.random.default_rng(K + N)
    kp = rng.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    got = w.w4a16_repack_k_to_n(torch.from_numpy(kp).cuda())
    torch.cuda.synchronize()
    want = oracle.pack(oracle.unpack_k(kp))
    assert np.array_equal(got.cpu().numpy(), want)



@pytest.mark.parametrize("M,K,N,G,dt,asym", [(1, 2112, 1152, 32, "bf16", False), (8, 2560, 3840, 128, "f16", True),
                                           (300, 2048, 768, 64, "f16", True), (40, 5120, 7168, 128, "bf16", False),
                                           (512, 4096, 1024, 128, "bf16", True), (7, 100, 520, 100, "f16", True)])
def test_prepared_layer_equals_the_function(w, M, K, N, G, dt, asym):
    """W4A16Linear (the library's prepared-layer handle: weights checked once, plan and weight
    descriptors kept per shape) gives exactly what w4a16_gemm gives on every path, and repeated
    calls with other activations and another M reuse the handle correctly."""
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=True, seed=5)
    t = case_tensors(c)
    layer = w.W4A16Linear(t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"])
    for m in (M, max(1, M // 2), M):
        a = t["a"][:m].contiguous() if m != M else t["a"]
        a2 = (a * 0.5).contiguous()
        for x in (a, a2):
            got = layer(x)
            want = w.w4a16_gemm(x, t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"])
            torch.cuda.synchronize()
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"m={m}"
    with pytest.raises(ValueError):
        layer(t["a"][:, :8].contiguous())  # wrong K
    # every argument check of the call, each rejected before anything is launched
    other = torch.float16 if t["a"].dtype == torch.bfloat16 else torch.bfloat16
    bad_inputs = [t["a"].reshape(-1),                                   # 1-D
                  t["a"].to(other)]                                     # dtype
    if M > 1:
        bad_inputs.append(t["a"].t().contiguous().t())                  # rows not contiguous
    for x in bad_inputs:
        with pytest.raises(ValueError):
            layer(x)
    good_out = torch.empty((M, N), dtype=t["a"].dtype, device="cuda")
    bad_outs = [torch.empty((M, N + 8), dtype=t["a"].dtype, device="cuda"),  # shape
                torch.empty((M, N), dtype=other, device="cuda")]               # dtype
    if M > 1:
        bad_outs.append(torch.empty((N, M), dtype=t["a"].dtype, device="cuda").t())  # not contiguous
    for o in bad_outs:
        with pytest.raises(ValueError):
            layer(t["a"], out=o)
    got = layer(t["a"], out=good_out)
    assert got is good_out


def test_layer_handle_through_the_c_abi(w):
    """w4a16_layer_create / _gemm / _workspace_size / _destroy called directly through the C ABI."""
    import ctypes
    M, K, N, G = 512, 4096, 1024, 128
    c = synth.make_case(M, K, N, G, "bf16", asym=True, bias=True, seed=9)
    t = case_tensors(c)
    L = w.lib()
    h = ctypes.c_void_p()
    assert L.w4a16_layer_create(t["b_q"].data_ptr(), t["scales"].data_ptr(), t["qzeros"].data_ptr(), G, 8,
                                t["bias"].data_ptr(), K, N, 1, ctypes.byref(h)) == 0, w.last_error()
    need = L.w4a16_layer_workspace_size(h, M)
    assert need == w.w4a16_gemm_workspace_size(M, K, N, G, 1) and need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert L.w4a16_layer_gemm(h, t["a"].data_ptr(), out.data_ptr(), M, ws.data_ptr(), need, None) == 0, w.last_error()
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    check_against_oracle(c, torch_to_bits(out), rows=np.arange(0, M, 41), cols=sample_cols(N, rng, k=64),
                         label="layer handle", path="prefill")
    # out overlapping the activations is rejected before any launch
    before = w.w4a16_debug_launch_count()
    assert L.w4a16_layer_gemm(h, t["a"].data_ptr(), t["a"].data_ptr(), M, None, 0, None) == 1
    assert w.w4a16_debug_launch_count() == before
    assert L.w4a16_layer_destroy(h) == 0


def test_plans_of_different_shapes_share_one_workspace(w):
    """Stream-K calls whose plans differ in grid and tile height, alternating on one workspace
    buffer: each call's flags must start at zero whatever the previous call left in the partials."""
    shapes = [(1024, 17408, 5120, 64, "bf16", True), (192, 5120, 7168, 128, "f16", False),
              (300, 2048, 768, 64, "bf16", False)]
    cases, plans = [], []
    for i, (M, K, N, G, dt, asym) in enumerate(shapes):
        c = synth.make_case(M, K, N, G, dt, asym=asym, bias=True, seed=40 + i)
        p = w.w4a16_plan(M, K, N, G, 1 if dt == "bf16" else 0, asym, 0, with_workspace=True)
        assert p["stream_k"] == 1
        cases.append((c, case_tensors(c)))
        plans.append((p["grid"], p["m_tile"]))
    assert len(set(plans)) == len(plans), plans  # all different layouts of the partials
    need = max(w.w4a16_gemm_workspace_size(c.M, c.K, c.N, c.G, 1 if c.dtype == "bf16" else 0) for c, _ in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(3)
    for rnd in range(2):
        for c, t in cases:
            out = torch.empty((c.M, c.N), dtype=t["a"].dtype, device="cuda")
            st = w.lib().w4a16_gemm_ws(*[w._ptr(x) for x in (t["a"], t["b_q"], t["scales"], t["qzeros"])], c.G, 8,
                                       w._ptr(t["bias"]), w._ptr(out), c.M, c.K, c.N,
                                       1 if c.dtype == "bf16" else 0, w._ptr(ws), need, None)
            assert st == 0, w.last_error()
            torch.cuda.synchronize()
            rows = np.unique(np.linspace(0, c.M - 1, 5).astype(int))
            check_against_oracle(c, torch_to_bits(out), rows=rows, cols=sample_cols(c.N, rng, k=32),
                                 label=f"round {rnd} M={c.M}", path="prefill")


@pytest.mark.parametrize("M,K,N,G,dt,asym", [(40, 5120, 7168, 128, "f16", True), (100, 2112, 1152, 32, "bf16", False),
                                           (128, 17408, 5120, 17408, "bf16", True), (17, 1152, 2112, 32, "bf16", False)])
def test_cluster_split_k_mid_m(w, M, K, N, G, dt, asym):
    """Mid M: the CTAs of a cluster split each 128-row tile's K blocks and add their partial tiles
    through distributed shared memory in rank order: oracle parity, determinism, no workspace. (At
    17..32 rows the dispatcher runs the decode kernel; the 128-row kernel is forced there.)"""
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=True, seed=M + 3)
    code = 1 if dt == "bf16" else 0
    w.w4a16_debug_force_path("prefill" if M <= 32 else None)
    try:
        plan = w.w4a16_plan(M, K, N, G, code, asym, 0, with_workspace=False)
        assert plan["path_name"] == "prefill" and plan["k_split"] > 1 and plan["stream_k"] == 0, plan
        t = case_tensors(c)
        outs = []
        for _ in range(2):
            out = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], use_workspace=False)
            torch.cuda.synchronize()
            outs.append(torch_to_bits(out))
    finally:
        w.w4a16_debug_force_path(None)
    assert np.array_equal(outs[0], outs[1]), "cluster split-K must be deterministic"
    assert w.w4a16_get_device_error() == 0
    rng = np.random.default_rng(M)
    rows = sorted({0, M - 1} | set(rng.integers(0, M, size=6).tolist()))
    check_against_oracle(c, outs[0], rows=rows, cols=sample_cols(N, rng, k=128), label="cluster split-K",
                         path="prefill")



DECODE_VARIANTS = [(ncg, C, sb) for ncg in (1, 2) for (C, sb) in ((1, 4), (2, 2), (3, 1), (5, 2), (9, 1), (16, 1), (2, 4))]


@pytest.mark.parametrize("M,K,N,G,dt,asym,bias", [(1, 1152, 4224, 32, "bf16", False, False),
                                                 (5, 2112, 1152, 32, "bf16", False, False),
                                                 (8, 2560, 3840, 128, "f16", True, True),
                                                 (3, 5120, 1024, 5120, "bf16", True, False),
                                                 (16, 1024, 2048, 64, "f16", False, True),
                                                 (12, 4104, 288, 4104, "f16", True, True),
                                                 (8, 1024, 768, 32, "f16", True, True),
                                                 (2, 640, 512, 64, "bf16", True, False),
                                                 (7, 4104, 288, 4104, "bf16", True, False),
                                                 (17, 1024, 2048, 64, "f16", True, True),
                                                 (24, 2112, 1152, 32, "bf16", False, False),
                                                 (32, 4104, 288, 4104, "bf16", True, False)])
def test_every_decode_configuration_matches_oracle(w, M, K, N, G, dt, asym, bias):
    """Each decode configuration (one or two consumer groups, split-K factors up to 16 with the
    split-K exchange through st.async pushes, stages of 1, 2 or 4 K blocks) against the oracle on the
    exact-weight reading, and the identity-A product bit-exact, on shapes with ragged K and N."""
    if N % 32:
        pytest.skip("decode needs N % 32 == 0")
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=M * 3 + K)
    t = case_tensors(c)
    one = int(oracle.ieee.t_encode_rne(np.array([1.0]), dt)[0])
    ks = np.random.default_rng(M).choice(K, size=M, replace=False)
    a_id = c.a.copy()
    a_id[:] = 0
    a_id[np.arange(M), ks] = one
    t_id = bits_to_torch(a_id, dt)
    want_id = oracle.dequant_t(c.b_q, c.scales, c.qzeros, G, 8, dt)[ks]
    seen = set()
    try:
        for ncg, C, sb in DECODE_VARIANTS:
            w.w4a16_debug_decode_override(ncg, C, sb)
            plan = w.w4a16_plan(M, K, N, G, 1 if dt == "bf16" else 0, asym, 0, with_workspace=False)
            assert plan["path_name"] == "decode"
            key = (plan["warps"], plan["k_split"], plan["k_blocks_per_stage"])
            if key in seen:
                continue
            seen.add(key)
            out = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], use_workspace=False)
            out_id = w.w4a16_gemm(t_id, t["b_q"], t["scales"], t["qzeros"], G, 8, None, use_workspace=False)
            torch.cuda.synchronize()
            check_against_oracle(c, torch_to_bits(out), label=f"decode plan {key}", path="decode")
            assert np.array_equal(torch_to_bits(out_id), want_id), f"identity A, decode plan {key}"
    finally:
        w.w4a16_debug_decode_override(0, 0, 0)
    assert w.w4a16_get_device_error() == 0


@pytest.mark.parametrize("K,N", [(64, 256), (130, 264), (2112, 1152), (2560, 3840), (4104, 288)])
def test_prepack_bitexact(w, K, N):
    """w4a16_prepack on the GPU writes exactly the oracle's prepacked layout, padding included."""
    rng = np.random.default_rng(K + N)
    b = rng.integers(0, 2 ** 32, size=(K, N // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    got = w.w4a16_prepack(torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    want = oracle.prepack(b).reshape(-1)
    assert got.numel() == want.size == w.lib().w4a16_prepack_bytes(K, N) // 4
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("M,K,N,G,dt,asym,bias", [(1, 1152, 4224, 32, "bf16", False, False),
                                                 (8, 2560, 3840, 128, "f16", True, True),
                                                 (5, 4104, 288, 4104, "bf16", True, False),
                                                 (40, 5120, 1024, 128, "f16", False, True),
                                                 (300, 2048, 768, 64, "bf16", True, True),
                                                 (1024, 4096, 1024, 32, "f16", True, False)])
def test_prepacked_layer_equals_the_canonical_one(w, M, K, N, G, dt, asym, bias):
    """A layer on the prepacked weights gives exactly the bits of the layer on b_q (decode, mid-M
    cluster split, prefill with stream-K; ragged K and N), and passes the oracle on its path's
    reading; on the decode path every configuration, and identity-A, as well."""
    c = synth.make_case(M, K, N, G, dt, asym=asym, bias=bias, seed=M + K + 1)
    t = case_tensors(c)
    canon = w.W4A16Linear(t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"])
    pp = w.W4A16Linear(t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"], prepacked=True)
    want, got = canon(t["a"]), pp(t["a"])
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    rng = np.random.default_rng(M)
    rows = sorted({0, M - 1} | set(rng.integers(0, M, size=4).tolist()))
    check_against_oracle(c, torch_to_bits(got), rows=rows, cols=sample_cols(N, rng, k=64), label="prepacked",
                         path=path_taken(w, c))
    if path_taken(w, c) == "decode":
        try:
            for ncg, C, sb in DECODE_VARIANTS:
                w.w4a16_debug_decode_override(ncg, C, sb)
                a, b = canon(t["a"]), pp(t["a"])
                torch.cuda.synchronize()
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (ncg, C, sb)
        finally:
            w.w4a16_debug_decode_override(0, 0, 0)


def test_prepacked_layer_refuses_the_generic_path(w):
    c = synth.make_case(4, 512, 1024, 128, "f16", seed=5)
    t = case_tensors(c)
    pp = w.W4A16Linear(t["b_q"], t["scales"], None, 128, 8, None, prepacked=True)
    a2 = torch.empty(c.M * c.K + 1, dtype=torch.float16, device="cuda")[1:].view(c.M, c.K)
    a2.copy_(t["a"])
    with pytest.raises(w.W4A16Error) as e:
        pp(a2)
    assert e.value.status == 2

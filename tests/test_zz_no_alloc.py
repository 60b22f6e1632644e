"""w4a16_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (code running while a CUDA graph is captured, allocator-less
runtimes and plugins that are handed only tensor pointers). For them the library keeps its stream-K
scratch in a static device array. This test calls the entry point through the C ABI and checks its
output against the workspace entry point's (w4a16_gemm_ws with a caller-owned workspace), within the
layer's tolerance, and against the CPU oracle on sampled outputs, on two calls in a row - the second
call finds the first call's leftovers in the shared array. The stream-K cases are asserted to plan
stream-K, so that they exercise the static array. It lives in a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import case_tensors, check_against_oracle, sample_cols, torch_to_bits

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


def _call(w, fn, t, c, code, extra=()):
    out = torch.empty((c.M, c.N), dtype=t["a"].dtype, device="cuda")
    args = [w._ptr(t["a"]), w._ptr(t["b_q"]), w._ptr(t["scales"]), w._ptr(t["qzeros"]), c.G, c.zp_bias,
            w._ptr(t["bias"]), w._ptr(out), c.M, c.K, c.N, code, *extra, None]
    st = fn(*args)
    assert st == 0, w.last_error()
    torch.cuda.synchronize()
    return torch_to_bits(out)


@pytest.mark.parametrize("M,K,N,G,dt,asym,stream_k", [(1024, 4096, 1024, 128, "bf16", True, True),
                                                    (512, 2048, 768, 64, "f16", False, True),  # other grid
                                                    (8, 2560, 3840, 128, "f16", True, False)])  # decode
def test_noalloc_matches_workspace_entry_point_twice(w, M, K, N, G, dt, asym, stream_k):
    code = 1 if dt == "bf16" else 0
    L = w.lib()
    # the first two shapes take a stream-K plan, so they really use the static array
    plan = w.w4a16_plan(M, K, N, G, code, asym, 0, with_workspace=True)
    assert bool(plan["stream_k"]) == stream_k, plan
    path = plan["path_name"]
    for call in range(2):  # two calls in a row: the array keeps the first call's contents
        c = synth.make_case(M, K, N, G, dt, asym=asym, bias=True, seed=100 * call + M)
        t = case_tensors(c)
        need = w.w4a16_gemm_workspace_size(M, K, N, G, code)
        assert (need > 0) == stream_k
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        ref = _call(w, L.w4a16_gemm_ws, t, c, code, extra=(w._ptr(ws), ctypes.c_size_t(ws.numel())))
        got = _call(w, L.w4a16_gemm_noalloc, t, c, code)
        atol, rtol = oracle.tolerance(dt)
        r = oracle.ieee.t_decode(ref, dt)
        g = oracle.ieee.t_decode(got, dt)
        assert np.all(np.isfinite(g))
        assert np.all(np.abs(g - r) <= atol + rtol * np.abs(r)), f"call {call}: outside tolerance"
        # and against the oracle on sampled rows and columns
        rng = np.random.default_rng(call + M)
        rows = sorted({0, M - 1} | set(rng.integers(0, M, size=4).tolist()))
        check_against_oracle(c, got, rows=rows, cols=sample_cols(N, rng, k=64), label=f"noalloc call {call}",
                             path=path)

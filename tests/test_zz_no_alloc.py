"""w4a16_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (code running while a CUDA graph is captured, allocator-less
runtimes and plugins that are handed only tensor pointers). For them the library keeps its stream-K
scratch in a static device array. This test calls the entry point through the C ABI and checks its
output against the workspace entry point's (w4a16_gemm_ws with a caller-owned workspace), within the
layer's tolerance, on two calls in a row - the second call finds the first call's leftovers in the
shared array. It lives in a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import case_tensors, torch_to_bits

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


@pytest.mark.parametrize("M,K,N,G,dt,asym", [(1024, 4096, 1024, 128, "bf16", True),   # stream-K prefill
                                           (512, 2048, 768, 64, "f16", False),      # stream-K, other grid
                                           (8, 2560, 3840, 128, "f16", True)])      # decode: no scratch
def test_noalloc_matches_workspace_entry_point_twice(w, M, K, N, G, dt, asym):
    code = 1 if dt == "bf16" else 0
    L = w.lib()
    for call in range(2):  # two calls in a row: the array keeps the first call's contents
        c = synth.make_case(M, K, N, G, dt, asym=asym, bias=True, seed=100 * call + M)
        t = case_tensors(c)
        need = w.w4a16_gemm_workspace_size(M, K, N, G, code)
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        ref = _call(w, L.w4a16_gemm_ws, t, c, code, extra=(w._ptr(ws), ctypes.c_size_t(ws.numel())))
        got = _call(w, L.w4a16_gemm_noalloc, t, c, code)
        atol, rtol = oracle.tolerance(dt)
        r = oracle.ieee.t_decode(ref, dt)
        g = oracle.ieee.t_decode(got, dt)
        assert np.all(np.isfinite(g))
        assert np.all(np.abs(g - r) <= atol + rtol * np.abs(r)), f"call {call}: outside tolerance"

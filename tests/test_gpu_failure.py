"""Failure detection without a GPU fault: every device-side wait of the TMA-fed kernels is bounded.

With the stall hook on, the worker warps first wait on a barrier that nothing arrives on; with the
bound shortened to 5 ms that wait runs out. The kernel then records an error word, drains its own
copies and MMAs, frees its tensor memory, honours its cluster barriers and exits; the host reads
the TIMEOUT status, and the next call with the hook off and the default bound is correct again.
Nothing hangs or traps.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import case_tensors, check_against_oracle, forced_path, torch_to_bits

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


@pytest.mark.parametrize("path,M,K,N", [("prefill", 256, 4096, 1024), ("prefill", 64, 4096, 1024), ("decode", 4, 4096, 1024),
                                        ("decode", 1, 2560, 19456), ("decode", 24, 4096, 1024)])
def test_bounded_wait_reports_timeout_and_recovers(w, path, M, K, N):
    c = synth.make_case(M, K, N, 128, "bf16", asym=True, seed=21)
    t = case_tensors(c)
    assert w.w4a16_get_device_error() == 0
    try:
        w.w4a16_debug_set_wait_limit_ns(5_000_000)
        w.w4a16_debug_inject_stall(True)
        with forced_path(path):
            w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], c.G, 8)
        torch.cuda.synchronize()
        assert w.w4a16_get_device_error() == 5        # W4A16_ERR_TIMEOUT
        assert "bounded device-side wait" in w.last_error()
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_limit_ns(0)
    assert w.w4a16_get_device_error() == 0             # read-and-clear
    with forced_path(path):
        out = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], c.G, 8)
    torch.cuda.synchronize()
    assert w.w4a16_get_device_error() == 0
    check_against_oracle(c, torch_to_bits(out), rows=np.arange(0, M, 17),
                         cols=np.arange(0, N, max(1, N // 512)), label="after recovery", path=path)


def test_stream_k_timeout_then_same_workspace_is_correct(w):
    """A stream-K call that gives up its waits may leave partial-tile flags set in its workspace; the
    binding zeroes the flag area of its workspaces when the TIMEOUT is read, and the next call on the
    same workspace is correct."""
    M, K, N, G = 512, 4096, 1024, 128
    c = synth.make_case(M, K, N, G, "bf16", asym=True, bias=True, seed=23)
    t = case_tensors(c)
    plan = w.w4a16_plan(M, K, N, G, 1, True, 0, with_workspace=True)
    assert plan["path_name"] == "prefill" and plan["stream_k"] == 1, plan
    assert w.w4a16_get_device_error() == 0
    try:
        w.w4a16_debug_set_wait_limit_ns(5_000_000)
        w.w4a16_debug_inject_stall(True)
        w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"])
        torch.cuda.synchronize()
        assert w.w4a16_get_device_error() == 5
    finally:
        w.w4a16_debug_inject_stall(False)
        w.w4a16_debug_set_wait_limit_ns(0)
    for buf in w._workspaces.values():
        assert int(buf[:4096].count_nonzero()) == 0
    out = w.w4a16_gemm(t["a"], t["b_q"], t["scales"], t["qzeros"], G, 8, t["bias"])
    torch.cuda.synchronize()
    assert w.w4a16_get_device_error() == 0
    check_against_oracle(c, torch_to_bits(out), rows=np.arange(0, M, 37), cols=np.arange(0, N, 3),
                         label="stream-K after timeout", path="prefill")

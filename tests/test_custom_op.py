"""The torch custom-op boundary (the lesson of the PR #51453 report).

CPU: under FakeTensorMode the fake implementation gives the output metadata of the pages' fake-impl
test (a(4,256) fp16, b_q(256,64), scales(2,512), qzeros None, group_size 128 -> out (4,512), dtype and
device of a), and make_fx records one call_function node for torch.ops.w4a16.gemm.default.
GPU: a torch.compile'd function over the op gives the oracle's results at decode and prefill sizes
in either order, and the library picks the decode kernel for the small M at run time.
"""
import json
import os

import numpy as np
import pytest
import torch
from torch._subclasses.fake_tensor import FakeTensorMode
from torch.fx.experimental.proxy_tensor import make_fx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fake_impl_shape.json")


@pytest.fixture(scope="module")
def ops():
    from w4a16_int4_weight_group_gb300 import ops as mod
    return mod


def test_fake_impl_metadata_and_graph_node(ops):
    g = json.load(open(GOLDEN))
    dt = torch.float16
    with FakeTensorMode():
        a = torch.empty(g["a"]["shape"], device="cuda", dtype=dt)
        b_q = torch.empty(g["b_q"]["shape"], device="cuda", dtype=torch.int32)
        scales = torch.empty(g["scales"]["shape"], device="cuda", dtype=dt)
        out = ops.w4a16_linear(a, b_q, scales, None, g["group_size"])
        assert list(out.shape) == g["out"]["shape"]
        assert out.dtype == a.dtype
        assert out.device == a.device
        graph = make_fx(lambda a, b_q, scales: ops.w4a16_linear(a, b_q, scales, None, g["group_size"]))(
            a, b_q, scales)
    assert any(n.op == "call_function" and n.target == torch.ops.w4a16.gemm.default for n in graph.graph.nodes)


@pytest.mark.gpu
def test_compiled_op_uses_runtime_m(ops):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import synth
    import w4a16_int4_weight_group_gb300 as w4
    from tests._util import bits_to_torch, check_against_oracle, torch_to_bits

    K, N, G = 2560, 3840, 128
    base = synth.make_case(1, K, N, G, "f16", asym=True, bias=True, seed=31)
    b_q = torch.from_numpy(base.b_q).cuda()
    scales = bits_to_torch(base.scales, "f16")
    qz = torch.from_numpy(base.qzeros).cuda()
    bias = bits_to_torch(base.bias, "f16")
    fn = torch.compile(lambda a: ops.w4a16_linear(a, b_q, scales, qz, G, 8, bias), backend="aot_eager",
                       dynamic=True)
    for M in (1024, 1, 8, 512):
        c = synth.make_case(M, K, N, G, "f16", asym=True, bias=True, seed=31)
        c.bias = base.bias  # the weights match the base case (drawn first); the bias is drawn after A
        out = fn(bits_to_torch(c.a, "f16"))
        torch.cuda.synchronize()
        rows = np.unique(np.linspace(0, M - 1, 6).astype(int))
        want = "decode" if M <= 32 else "prefill"
        assert w4.w4a16_plan(M, K, N, G, 0, True, 0)["path_name"] == want
        check_against_oracle(c, torch_to_bits(out), rows=rows, cols=np.arange(0, N, 7), label=f"compiled M={M}",
                             path=want)

"""torch.library custom op over the C ABI: ``torch.ops.w4a16.gemm``.

The PR #51453 report ("register Triton W4A16 GEMM as custom op", motivation and implementation
breakdown) traces a decode throughput regression to torch.compile tracing the Python tile
selection and freezing the prefill configuration into decode calls; the fix is an opaque custom op
with a fake implementation, so that the compiled graph holds one call node and tile selection sees
the real runtime shape. Here the tile, split-K and cluster choice already live inside the library
(chosen per call from the runtime M), and this module makes the call opaque to torch.compile:

* the real implementation forwards to ``w4a16_gemm`` of the binding (no computation in Python);
* the fake implementation only states the output metadata, as the pages' fake impl does:
  shape (a.size(0), b_q.size(1) * 8), dtype and device of ``a``; it checks nothing;
* ``mutates_args=()``: inputs are not written, the output is a new tensor.

Import this module to register the op.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import w4a16_gemm as _w4a16_gemm


@torch.library.custom_op("w4a16::gemm", mutates_args=())
def gemm(a: torch.Tensor, b_q: torch.Tensor, scales: torch.Tensor, qzeros: Optional[torch.Tensor],
         group_size: int, zp_bias: int = 8, bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out = cast(a @ dequant(b_q, scales, qzeros | zp_bias) + bias); runs libw4a16.so."""
    return _w4a16_gemm(a, b_q, scales, qzeros, group_size, zp_bias, bias)


@gemm.register_fake
def _gemm_fake(a, b_q, scales, qzeros, group_size, zp_bias=8, bias=None):
    return a.new_empty((a.size(0), b_q.size(1) * 8))


def w4a16_linear(a: torch.Tensor, b_q: torch.Tensor, scales: torch.Tensor, qzeros: Optional[torch.Tensor],
                 group_size: int, zp_bias: int = 8, bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Facade with the signature of the pages' ``triton_w4a16_gemm`` (plus bias), routed through the op."""
    return torch.ops.w4a16.gemm(a, b_q, scales, qzeros, group_size, zp_bias, bias)

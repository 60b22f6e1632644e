"""Seeded synthetic inputs for the W4A16 linear layer C = A . dequant(W) (+ bias).

This module only draws random data: it holds none of the layer's arithmetic
(no unpacking, no dequantisation, no product). Both the CPU oracle and the CUDA
library consume exactly the bytes produced here, so a parity test compares two
independent computations on identical inputs.

Shapes and value distributions follow the workloads described on the pages:

* the PR #51453 report ("register Triton W4A16 GEMM as custom op"), key source
  snippets: the fake-impl test uses a(4,256) fp16, b_q(256,64) int32,
  scales(2,512), qzeros=None, group_size=128 -> out(4,512);
* the PR #43731 report (Triton W4A16 as CUDA fallback), motivation: a model with
  intermediate_size=2112 that is not a multiple of 128;
* the PR #40977 report (ROCm RDNA hybrid W4A16), motivation: Qwen3-4B /
  Gemma-3-4B class decode layers; and the PR #51453 motivation: a Qwen 27B
  GPTQ-4bit decoder.

No model weights exist here, so every tensor is random:
A ~ N(0,1) rounded to the activation dtype; packed weight words are uniform
32-bit words (which is the same as eight independent uniform 4-bit values per
word); zero-point words likewise; scales ~ U[lo, hi] rounded to the dtype;
bias ~ N(0, bias_std) rounded to the dtype.

Every floating-point tensor is returned as its raw 16-bit patterns (uint16) so
that consumers decode it themselves.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

DTYPES = ("f16", "bf16")


def _round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 samples to the 16-bit dtype with a library conversion and return bit patterns."""
    if dtype == "f16":
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch  # CPU conversion only

        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(f"unknown dtype {dtype!r}")


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def random_words(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform random 32-bit words, returned as int32 (the packed-storage dtype)."""
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32).view(np.int32)


def random_nibbles(rows: int, cols: int, seed: int) -> np.ndarray:
    """uint8 [rows, cols] with each value uniform in 0..15 (input to the packer)."""
    return _rng(seed).integers(0, 16, size=(rows, cols), dtype=np.uint8)


@dataclass
class Case:
    """One linear-layer problem. Float tensors are uint16 bit patterns of `dtype`."""

    M: int
    K: int
    N: int
    G: int
    dtype: str
    a: np.ndarray                     # uint16 [M, K]
    b_q: np.ndarray                   # int32  [K, N/8]
    scales: np.ndarray                # uint16 [K/G, N]
    qzeros: Optional[np.ndarray]      # int32  [K/G, N/8] or None
    zp_bias: int
    bias: Optional[np.ndarray]        # uint16 [N] or None
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def asym(self) -> bool:
        return self.qzeros is not None


def make_case(M: int, K: int, N: int, G: int, dtype: str, *, asym: bool = False,
              bias: bool = False, seed: int = 0, scale_lo: float = 0.005,
              scale_hi: float = 0.02, bias_std: float = 0.1, zp_bias: int = 8,
              a_std: float = 1.0) -> Case:
    """Draw one seeded problem. M may be 0; K must be a multiple of G; N a multiple of 8."""
    if dtype not in DTYPES:
        raise ValueError(dtype)
    if N % 8 or K % G:
        raise ValueError("N must be a multiple of 8 and K a multiple of G")
    rng = _rng(seed)
    ng = K // G
    b_q = random_words(rng, (K, N // 8))
    scales = _round_to_bits(rng.uniform(scale_lo, scale_hi, size=(ng, N)), dtype)
    qzeros = random_words(rng, (ng, N // 8)) if asym else None
    a = _round_to_bits(rng.standard_normal(size=(M, K)) * a_std, dtype)
    bias_bits = _round_to_bits(rng.standard_normal(size=(N,)) * bias_std, dtype) if bias else None
    return Case(M=M, K=K, N=N, G=G, dtype=dtype, a=a, b_q=b_q, scales=scales, qzeros=qzeros,
                zp_bias=zp_bias, bias=bias_bits, seed=seed)


def activations(M: int, K: int, dtype: str, seed: int) -> np.ndarray:
    """A fresh activation matrix (uint16 bits) for an existing weight set."""
    return _round_to_bits(_rng(seed).standard_normal(size=(M, K)), dtype)


# The five measurement workloads, as data. Each entry lists (M values, (K, N) shapes, G values,
# dtypes, asym flags, bias flag, scale range).
CONFIGS = {
    # fake-impl shape of the custom-op test (PR #51453 report, key source snippets)
    "tiny": dict(Ms=[4], shapes=[(256, 512)], Gs=[128], dtypes=["f16"], asym=[False], bias=False,
                 scale=(0.005, 0.02)),
    # intermediate_size=2112 model (PR #43731 report, motivation): gate+up 1152->4224, down 2112->1152
    "decode_2112": dict(Ms=[1, 2, 4, 5, 8], shapes=[(1152, 4224), (2112, 1152)], Gs=[32],
                        dtypes=["bf16"], asym=[False], bias=False, scale=(0.005, 0.02)),
    # 4B-class decode layers (PR #40977 report, motivation)
    "decode_4b": dict(Ms=[1, 4, 8], shapes=[(2560, 3840), (2560, 19456), (9728, 2560)], Gs=[128],
                      dtypes=["f16"], asym=[True], bias=True, scale=(0.005, 0.02)),
    # prefill on a 27B-class decoder (PR #51453 report, motivation)
    "prefill": dict(Ms=[512, 1024, 4096], shapes=[(5120, 34816), (17408, 5120)], Gs=[64],
                    dtypes=["bf16"], asym=[True], bias=False, scale=(0.002, 0.01)),
    # mid M on two of the same 27B-class layers: one 128-row tile per column tile, K split over a
    # thread-block cluster (weight bytes still dominate the roofline up to M = 64)
    "mid_m": dict(Ms=[17, 24, 32, 64], shapes=[(5120, 7168), (17408, 5120)], Gs=[128],
                  dtypes=["bf16"], asym=[False], bias=False, scale=(0.005, 0.02)),
    # full M sweep on the same 27B-class layer
    "sweep": dict(Ms=[1, 2, 4, 5, 6, 8, 16, 24, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192],
                  shapes=[(5120, 7168), (5120, 34816), (17408, 5120)], Gs=[128, "K"],
                  dtypes=["f16", "bf16"], asym=[False, True], bias=False, scale=(0.005, 0.02)),
}


def config_cases(name: str):
    """Yield (M, K, N, G, dtype, asym, bias, scale_lo, scale_hi, seed) for every case of a workload.

    Seeds are 0 for the tiny workload and the running index of the case otherwise.
    """
    c = CONFIGS[name]
    idx = 0
    for dtype in c["dtypes"]:
        for asym in c["asym"]:
            for g in c["Gs"]:
                for (K, N) in c["shapes"]:
                    G = K if g == "K" else g
                    for M in c["Ms"]:
                        seed = 0 if name == "tiny" else idx
                        yield (M, K, N, G, dtype, asym, c["bias"], c["scale"][0], c["scale"][1], seed)
                        idx += 1

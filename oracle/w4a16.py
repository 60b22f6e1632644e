"""Plain CPU oracle of the W4A16 linear layer (fp64). Test infrastructure only.

What is computed, and where it is defined:

* Packed weights ``b_q[K, N/8]`` int32, eight 4-bit values per word along N
  (PR #51453 report, implementation breakdown item 1: ``N = b_q.shape[1] * 8``;
  key source snippets, fake-impl test: ``b_q (256, 64)`` for K=256, N=512).
  Nibble j of word c (bits 4j..4j+3) holds column 8c+j: the order inside a word
  is not printed on the pages, and this reading (sequential, little-endian) is
  the plainest one.
* Per-group scales ``scales[K/G, N]`` in the activation dtype (same snippets:
  ``scales (2, 512)`` for K=256, G=128).
* Zero points: ``qzeros[K/G, N/8]`` packed like b_q, or the fixed bias 8 of the
  symmetric uint4b8 type when qzeros is None (PR #51453 snippets: qzeros=None
  takes the zp_bias=8 branch).
* Dequantisation ``(q - zp) * scale``, with scales and zero points repeated
  ``group_size`` times along K, and the product taken with the activations in
  higher precision, bias added before the final cast (PR #40977 report, key
  source snippets, the test reference ``_rdna_hybrid_w4a16_reference``).

Two products are offered:

* ``weights="exact"``: the dequantised weights kept exact in fp64 (the
  PR #40977 test reference keeps them in fp32, where they are also exact);
* ``weights="dequant_t"``: the dequantised weights rounded once to the
  activation dtype, i.e. the values ``dequant_t`` returns. These are the values
  a 16-bit tensor-core product consumes.

Both products are then summed in fp64 (numpy matmul, a library primitive) and
returned in fp64 without the final cast.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .ieee import t_decode, t_encode_rne, t_unit_roundoff, t_min_subnormal

# Acceptance tolerance of the layer's output: |out - ref| <= atol + rtol * |ref|.
# The PR #40977 report's test compares against its reference "with 2e-2 tolerance";
# fp16 uses the tighter 1e-2 of this library's contract.
TOLERANCE = {"f16": (1e-2, 1e-2), "bf16": (2e-2, 2e-2)}

SUPPORTED_GROUP_SIZES = (32, 64, 128)


# ----------------------------------------------------------------------------------------------
# packing
# ----------------------------------------------------------------------------------------------
def pack(q: np.ndarray) -> np.ndarray:
    """uint8 [R, N] (values 0..15) -> int32 [R, N/8]; word c = sum_j q[:, 8c+j] << 4j."""
    q = np.asarray(q)
    if q.ndim != 2 or q.shape[1] % 8:
        raise ValueError("q must be [R, N] with N % 8 == 0")
    if np.any(q > 15):
        raise ValueError("q values must be 0..15")
    R, N = q.shape
    word = np.zeros((R, N // 8), dtype=np.uint64)
    for j in range(8):
        word |= q[:, j::8].astype(np.uint64) << np.uint64(4 * j)
    return word.astype(np.uint32).view(np.int32)


def unpack(packed: np.ndarray, n: Optional[int] = None, cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """int32 [R, N/8] -> uint8 [R, N] (or only the listed columns); logical shift on uint32."""
    w = np.asarray(packed).view(np.uint32)
    if cols is None:
        n = w.shape[1] * 8 if n is None else n
        cols = np.arange(n)
    cols = np.asarray(cols, dtype=np.int64)
    words = w[:, cols >> 3].astype(np.uint64)
    shifts = (4 * (cols & 7)).astype(np.uint64)
    return ((words >> shifts) & np.uint64(0xF)).astype(np.uint8)


def pack_k(q: np.ndarray) -> np.ndarray:
    """uint8 [K, N] -> int32 [N, K/8], packed along K (the PR #40977 report's "[N, K//8] int32"
    layout): word c of row n = sum_j q[8c + j, n] << 4j. The order inside a word is not printed;
    sequential little-endian along K is the reading taken (the same convention as ``pack``)."""
    q = np.asarray(q)
    if q.ndim != 2 or q.shape[0] % 8:
        raise ValueError("q must be [K, N] with K % 8 == 0")
    return pack(q.T)


def unpack_k(k_packed: np.ndarray) -> np.ndarray:
    """int32 [N, K/8] -> uint8 [K, N]; the inverse of ``pack_k``."""
    return unpack(k_packed).T.copy()


# ----------------------------------------------------------------------------------------------
# prepacked weight layout (this library's kernel-native layout; the pages' kernels read b_q as is)
# ----------------------------------------------------------------------------------------------
# The packed words b_q[K, N/8] regrouped into blocks of 64 rows x 32 words (a 64-row K block of a
# 256-column tile), blocks ordered tile-major then K block, each block contiguous (8 KB); K and N are
# padded with zero words to multiples of 64 and 256. Inside a block, row r occupies 32 consecutive
# words, and its 16-byte chunks (four words each) are permuted by XOR with r mod 8: word w of row r
# sits at position 4 * ((w // 4) ^ (r % 8)) + w % 4 of the row. (That is where a 2-D copy with a
# 128-byte swizzle places the same 64 x 128-byte box.)
PP_ROWS, PP_WORDS = 64, 32


def prepack(b_q: np.ndarray) -> np.ndarray:
    """int32 [K, N/8] -> int32 [ceil(N/256), ceil(K/64), 64, 32] in the prepacked layout."""
    b_q = np.asarray(b_q).view(np.int32)
    K, NW = b_q.shape
    tiles, kbs = -(-NW // PP_WORDS), -(-K // PP_ROWS)
    out = np.zeros((tiles, kbs, PP_ROWS, PP_WORDS), dtype=np.int32)
    for t in range(tiles):
        for kb in range(kbs):
            for r in range(PP_ROWS):
                k = kb * PP_ROWS + r
                if k >= K:
                    continue
                for w in range(PP_WORDS):
                    c = t * PP_WORDS + w
                    if c >= NW:
                        continue
                    pos = 4 * ((w // 4) ^ (r % 8)) + w % 4
                    out[t, kb, r, pos] = b_q[k, c]
    return out


def unprepack(b_pp: np.ndarray, k: int, n: int) -> np.ndarray:
    """The inverse of ``prepack`` for a [k, n] weight matrix: int32 [k, n/8]."""
    b_pp = np.asarray(b_pp).view(np.int32)
    nw = n // 8
    out = np.zeros((k, nw), dtype=np.int32)
    for kk in range(k):
        kb, r = divmod(kk, PP_ROWS)
        for c in range(nw):
            t, w = divmod(c, PP_WORDS)
            out[kk, c] = b_pp[t, kb, r, 4 * ((w // 4) ^ (r % 8)) + w % 4]
    return out


# ----------------------------------------------------------------------------------------------
# dequantisation
# ----------------------------------------------------------------------------------------------
def zero_points(qzeros: Optional[np.ndarray], zp_bias: int, n_groups: int, cols) -> np.ndarray:
    """int64 [K/G, len(cols)]: unpacked qzeros, or zp_bias everywhere when qzeros is None."""
    cols = np.asarray(cols, dtype=np.int64)
    if qzeros is None:
        return np.full((n_groups, cols.size), int(zp_bias), dtype=np.int64)
    return unpack(qzeros, cols=cols).astype(np.int64)


def dequant_exact(b_q, scales, qzeros, group_size: int, zp_bias: int, dtype: str,
                  cols=None) -> np.ndarray:
    """fp64 [K, N] (or [K, len(cols)]): W[k, n] = (q[k, n] - zp[k // G, n]) * s[k // G, n].

    Exact: an integer in [-15, 15] times a 16-bit float needs at most 4 + 11 significant bits.
    """
    K = b_q.shape[0]
    N = b_q.shape[1] * 8
    G = int(group_size)
    if K % G:
        raise ValueError("K must be a multiple of group_size")
    cols = np.arange(N) if cols is None else np.asarray(cols, dtype=np.int64)
    q = unpack(b_q, cols=cols).astype(np.int64)                       # [K, C]
    ng = K // G
    zp = zero_points(qzeros, zp_bias, ng, cols)                        # [ng, C]
    s = t_decode(np.asarray(scales)[:, cols], dtype)                   # [ng, C]
    g_of_k = np.arange(K) // G                                         # repeat_interleave along K
    return (q - zp[g_of_k]).astype(np.float64) * s[g_of_k]


def dequant_t(b_q, scales, qzeros, group_size: int, zp_bias: int, dtype: str, cols=None) -> np.ndarray:
    """uint16 [K, N]: the exact dequantised value rounded once to the activation dtype (RNE)."""
    return t_encode_rne(dequant_exact(b_q, scales, qzeros, group_size, zp_bias, dtype, cols), dtype)


# ----------------------------------------------------------------------------------------------
# the product
# ----------------------------------------------------------------------------------------------
def gemm_ref(a, b_q, scales, qzeros, group_size: int, zp_bias: int, bias, dtype: str, *,
             weights: str = "dequant_t", rows=None, cols=None) -> np.ndarray:
    """fp64 [M, N] = A . W (+ bias), no final cast. ``rows``/``cols`` select a sub-block."""
    a = np.asarray(a)
    if rows is not None:
        a = a[np.asarray(rows, dtype=np.int64)]
    A = t_decode(a, dtype)
    N = b_q.shape[1] * 8
    cols = np.arange(N) if cols is None else np.asarray(cols, dtype=np.int64)
    W = dequant_exact(b_q, scales, qzeros, group_size, zp_bias, dtype, cols)
    if weights == "dequant_t":
        W = t_decode(t_encode_rne(W, dtype), dtype)
    elif weights != "exact":
        raise ValueError(weights)
    out = A @ W
    if bias is not None:
        out = out + t_decode(np.asarray(bias)[cols], dtype)[None, :]
    return out


def weight_rounding_bound(a, b_q, scales, qzeros, group_size, zp_bias, dtype, *, rows=None,
                          cols=None) -> np.ndarray:
    """fp64 [M, N]: sum_k |A[m,k]| * |RNE_T(W[k,n]) - W[k,n]|.

    A rigorous bound on |gemm_ref(dequant_t) - gemm_ref(exact)| (up to fp64 rounding).
    """
    a = np.asarray(a)
    if rows is not None:
        a = a[np.asarray(rows, dtype=np.int64)]
    A = np.abs(t_decode(a, dtype))
    W = dequant_exact(b_q, scales, qzeros, group_size, zp_bias, dtype, cols)
    Wt = t_decode(t_encode_rne(W, dtype), dtype)
    return A @ np.abs(Wt - W)


def out_t(ref: np.ndarray, dtype: str) -> np.ndarray:
    """The reference cast to the output dtype (uint16 bits)."""
    return t_encode_rne(ref, dtype)


def tolerance(dtype: str):
    return TOLERANCE[dtype]


def within_tolerance(out_bits, ref, dtype: str, extra=0.0) -> np.ndarray:
    """Elementwise bool: |out - ref| <= atol + rtol*|ref| + extra (non-finite outputs fail)."""
    atol, rtol = TOLERANCE[dtype]
    out = t_decode(np.asarray(out_bits), dtype)
    ok = np.abs(out - ref) <= atol + rtol * np.abs(ref) + extra
    return ok & np.isfinite(out)


def fp64_eps_bound(K: int) -> float:
    """Relative headroom for fp64 summation order differences in tests of the oracle itself."""
    return 1e-12 * max(1, K)


__all__ = ["pack", "unpack", "pack_k", "unpack_k", "prepack", "unprepack", "zero_points", "dequant_exact", "dequant_t", "gemm_ref",
           "weight_rounding_bound", "out_t", "tolerance", "within_tolerance", "TOLERANCE",
           "SUPPORTED_GROUP_SIZES", "t_unit_roundoff", "t_min_subnormal"]

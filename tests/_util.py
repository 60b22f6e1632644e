"""Test helpers: move synthetic cases to the GPU, call the library, compare with the oracle."""
from __future__ import annotations

import contextlib

import numpy as np
import torch

import oracle
from oracle import ieee

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits_to_torch(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(TORCH_DT[dtype])
    return t.to(device)


def torch_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def case_tensors(c, device="cuda"):
    d = {
        "a": bits_to_torch(c.a, c.dtype, device),
        "b_q": torch.from_numpy(c.b_q).to(device),
        "scales": bits_to_torch(c.scales, c.dtype, device),
        "qzeros": None if c.qzeros is None else torch.from_numpy(c.qzeros).to(device),
        "bias": None if c.bias is None else bits_to_torch(c.bias, c.dtype, device),
    }
    return d


@contextlib.contextmanager
def forced_path(path):
    """Restrict the library's dispatcher to `path` ("generic", "decode", "prefill"; None: no
    restriction) for the duration of the block."""
    import w4a16_int4_weight_group_gb300 as w4
    w4.w4a16_debug_force_path(path)
    try:
        yield
    finally:
        w4.w4a16_debug_force_path(None)


def sample_cols(N: int, rng: np.random.Generator, k: int = 384) -> np.ndarray:
    """Columns to check on wide outputs: both edges (past the first and into the last 256-column
    tile, every n % 8 position), and k random ones."""
    base = set(range(0, min(N, 264))) | set(range(max(0, N - 264), N))
    base |= set(rng.integers(0, N, size=k).tolist())
    return np.array(sorted(base), dtype=np.int64)


# Which correct reading of the layer (see the oracle: exact weights, or weights rounded once to the
# dtype) each kernel computes. The decode kernel multiplies the exact integers q - zp on the tensor
# core and applies the scale in fp32, so it is held to the exact-weight product; the prefill and
# generic kernels feed RNE((q - zp) * s) to the multiply, so they are held to the product over those
# rounded weights.
READING_OF_PATH = {"decode": "exact", "prefill": "dequant_t", "generic": "dequant_t"}


def path_taken(w, c, forced=None, with_workspace=True):
    """The kernel path a call on case c takes (the forced one, or the dispatcher's choice)."""
    code = 1 if c.dtype == "bf16" else 0
    with forced_path(forced):
        return w.w4a16_plan(c.M, c.K, c.N, c.G, code, c.asym, 0, with_workspace=with_workspace)["path_name"]


def check_against_oracle(c, out_bits: np.ndarray, rows=None, cols=None, label="", path=None, reading=None):
    """Accept each output if |out - ref| <= atol + rtol*|ref|, where ref is the fp64 product over the
    weights the path multiplies: the exact weights for the decode kernel, the dtype-rounded dequantised
    weights for the prefill and generic kernels (`path` picks the reading; `reading` may name it
    directly; "either" accepts the nearer of the two). Always require the exact-weight product within
    tolerance plus the rigorous weight-rounding bound. Returns error statistics against the reading."""
    if reading is None:
        if path is None:
            raise ValueError("check_against_oracle needs the path the output came from (or a reading)")
        reading = READING_OF_PATH[path]
    kw = dict(rows=rows, cols=cols)
    sub = out_bits
    if rows is not None:
        sub = sub[np.asarray(rows)]
    if cols is not None:
        sub = sub[:, np.asarray(cols)]
    ref_t = oracle.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, c.G, c.zp_bias, c.bias, c.dtype,
                            weights="dequant_t", **kw)
    ref_e = oracle.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, c.G, c.zp_bias, c.bias, c.dtype,
                            weights="exact", **kw)
    out = ieee.t_decode(sub, c.dtype)
    atol, rtol = oracle.tolerance(c.dtype)
    err_t, err_e = np.abs(out - ref_t), np.abs(out - ref_e)
    use_t = err_t / (atol + rtol * np.abs(ref_t))
    use_e = err_e / (atol + rtol * np.abs(ref_e))
    if reading == "exact":
        ok, use, err = oracle.within_tolerance(sub, ref_e, c.dtype), use_e, err_e
    elif reading == "dequant_t":
        ok, use, err = oracle.within_tolerance(sub, ref_t, c.dtype), use_t, err_t
    elif reading == "either":
        ok = oracle.within_tolerance(sub, ref_t, c.dtype) | oracle.within_tolerance(sub, ref_e, c.dtype)
        use, err = np.minimum(use_t, use_e), np.minimum(err_t, err_e)
    else:
        raise ValueError(reading)
    if not ok.all():
        bad = np.argwhere(~ok)[:8]
        details = [(int(i), int(j), float(out[i, j]), float(ref_t[i, j]), float(ref_e[i, j])) for i, j in bad]
        raise AssertionError(f"{label}: {int((~ok).sum())} of {ok.size} outputs outside {atol}+{rtol}|ref| of the "
                             f"{reading} reading (max err {err.max():.3g}); first (i, j, out, ref_T, ref_E): "
                             f"{details}")
    bound = oracle.weight_rounding_bound(c.a, c.b_q, c.scales, c.qzeros, c.G, c.zp_bias, c.dtype, **kw)
    ok_e = err_e <= atol + rtol * np.maximum(np.abs(ref_t), np.abs(ref_e)) + bound * (1 + 1e-9)
    if not ok_e.all():
        raise AssertionError(f"{label}: exact-weight bound violated at {int((~ok_e).sum())} outputs")
    return {"max_err": float(err.max()) if err.size else 0.0,
            "max_rel_tol_use": float(use.max()) if use.size else 0.0, "reading": reading}

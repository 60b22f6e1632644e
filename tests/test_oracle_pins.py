"""Pins of the CPU oracle against things other than itself (no GPU).

Each check ties an oracle function to an independent fact: a value the pages
print (tests/golden), a hand derivation, a library conversion (numpy binary16,
torch bfloat16), exact rational arithmetic, a closed form or an invariant.
The mutation tests at the end plant plausible mistakes in the oracle and show
that these checks catch them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import exact, ieee
from oracle import w4a16 as ow
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _lib_decode(bits, dtype):
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def _lib_encode(x, dtype):
    """Library rounding of fp64 values to the dtype (bf16: values must be exact in fp32)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x, equal_nan=True)
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------------------------------------
# IEEE binary16 / bfloat16
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_exhaustive_matches_library(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = ieee.t_decode(bits, dtype)
    lib = _lib_decode(bits, dtype)
    both_nan = np.isnan(mine) & np.isnan(lib)
    assert np.all(both_nan | (mine == lib))
    # signed zeros are kept
    assert np.all(np.signbit(mine[~np.isnan(mine)]) == np.signbit(lib[~np.isnan(lib)]))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_exact_decoder_matches_library(dtype):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    lib = _lib_decode(bits, dtype)
    for b, v in zip(bits, lib):
        if np.isfinite(v):
            assert exact.decode(int(b), dtype) == Fraction(float(v))


def _all_finite_values(dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = ieee.t_decode(bits, dtype)
    v = np.unique(v[np.isfinite(v)])
    return v


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_encode_roundtrips_every_value(dtype):
    v = _all_finite_values(dtype)
    assert np.array_equal(ieee.t_decode(ieee.t_encode_rne(v, dtype), dtype), v)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_encode_ties_and_near_ties_match_library(dtype):
    v = _all_finite_values(dtype)
    pos = v[v >= 0]
    mids = (pos[:-1] + pos[1:]) / 2            # exact ties (exact in fp64 and fp32)
    span = pos[1:] - pos[:-1]
    near_lo = mids - span / 16                 # just below a tie (exact in fp32 too)
    near_hi = mids + span / 16
    x = np.concatenate([mids, -mids, near_lo, near_hi, -near_hi])
    assert np.array_equal(ieee.t_encode_rne(x, dtype), _lib_encode(x, dtype))


def test_encode_random_fp64_matches_numpy_binary16():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
        rng.uniform(-1e-7, 1e-7, 20000),          # subnormal range
        rng.uniform(65000, 70000, 2000),          # around overflow
        [0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.99, 65520.0, 2.0 ** -25, 2.0 ** -24 * 1.5],
    ])
    with np.errstate(over="ignore"):  # numpy's cast overflows to inf by design past 65520
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ieee.t_encode_rne(x, "f16"), want)


def test_encode_random_fp32_exact_matches_torch_bfloat16():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 3.0e38, -3.0e38, 1e-40, -1e-40], np.float32)])
    x = x.astype(np.float64)
    assert np.array_equal(ieee.t_encode_rne(x, "bf16"), _lib_encode(x, "bf16"))


def test_exact_round_matches_oracle_round():
    rng = np.random.default_rng(4)
    for dtype in ("f16", "bf16"):
        for _ in range(300):
            num = int(rng.integers(-10 ** 6, 10 ** 6))
            den = int(2 ** rng.integers(8, 24))
            fr = Fraction(num, den)
            assert exact.round_rne(fr, dtype) == int(ieee.t_encode_rne(np.array([num / den]), dtype)[0])


# ------------------------------------------------------------------------------------------------
# packing
# ------------------------------------------------------------------------------------------------
def test_pack_golden_words():
    g = _golden("pack_words.json")
    q = np.array([c["q"] for c in g["cases"]], dtype=np.uint8).reshape(1, -1)
    words = ow.pack(q)[0]
    assert [int(w) for w in words] == [c["int32"] for c in g["cases"]]
    assert [f"0x{int(w) & 0xFFFFFFFF:08X}" for w in words] == [c["word_hex"] for c in g["cases"]]
    assert np.array_equal(ow.unpack(words.reshape(1, -1)), q)


def test_pack_each_nibble_position_exhaustive():
    for j in range(8):
        for v in range(16):
            q = np.zeros((1, 8), np.uint8)
            q[0, j] = v
            w = int(ow.pack(q)[0, 0]) & 0xFFFFFFFF
            assert w == v << (4 * j)
            assert ow.unpack(np.array([[np.uint32(w).view(np.int32)]]))[0, j] == v


def test_pack_unpack_roundtrip_random():
    q = synth.random_nibbles(37, 8 * 29, seed=5)
    p = ow.pack(q)
    assert p.dtype == np.int32 and p.shape == (37, 29)
    assert np.array_equal(ow.unpack(p), q)
    # random words round-trip the other way
    w = synth.random_words(np.random.default_rng(6), (11, 13))
    assert np.array_equal(ow.pack(ow.unpack(w)), w)


def test_fake_impl_shapes_from_pages():
    g = _golden("fake_impl_shape.json")
    M, K = g["a"]["shape"]
    N = g["b_q"]["shape"][1] * 8
    G = g["group_size"]
    c = synth.make_case(M, K, N, G, g["a"]["dtype"], seed=0)
    assert list(c.b_q.shape) == g["b_q"]["shape"]
    assert list(c.scales.shape) == g["scales"]["shape"]
    ref = ow.gemm_ref(c.a, c.b_q, c.scales, None, G, g["zp_bias_default"], None, c.dtype)
    assert list(ref.shape) == g["out"]["shape"]
    assert list(ow.out_t(ref, c.dtype).shape) == g["out"]["shape"]


# ------------------------------------------------------------------------------------------------
# dequantisation
# ------------------------------------------------------------------------------------------------
def test_dequant_golden_values():
    for c in _golden("dequant_values.json")["cases"]:
        dt = c["dtype"]
        q = np.full((1, 8), c["q"], np.uint8)
        b_q = ow.pack(q)
        zq = ow.pack(np.full((1, 8), c["zp"], np.uint8))
        s = np.full((1, 8), int(c["scale_bits"], 16), np.uint16)
        assert ieee.t_decode(s[0, :1], dt)[0] == float(Fraction(c["scale_value"]))
        w = ow.dequant_exact(b_q, s, zq, 1, 8, dt)
        assert np.all(w == float(Fraction(c["exact"])))
        wt = ow.dequant_t(b_q, s, zq, 1, 8, dt)
        assert np.all(wt == int(c["out_bits"], 16)), (c, hex(int(wt[0, 0])))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_dequant_exhaustive_q_zp_against_fractions_and_library(dtype):
    rng = np.random.default_rng(7)
    scale_bits = np.concatenate([
        ieee.t_encode_rne(rng.uniform(0.002, 0.03, 40), dtype),
        ieee.t_encode_rne(np.array([1.0, 0.5, 1e-6, 3e-3, 700.0, -0.01]), dtype),
    ])
    qs = np.arange(16)
    for sb in scale_bits:
        s = exact.decode(int(sb), dtype)
        # one row per zero point, 16 q values per row (two words)
        q = np.tile(qs, (16, 1)).astype(np.uint8)
        zq = ow.pack(np.arange(16, dtype=np.uint8).repeat(16).reshape(16, 16))
        b_q = ow.pack(q)
        scales = np.full((16, 16), sb, np.uint16)
        w = ow.dequant_exact(b_q, scales, zq, 1, 8, dtype)      # G = 1: one group per row
        wt = ow.dequant_t(b_q, scales, zq, 1, 8, dtype)
        for zp in range(16):
            for qq in range(16):
                fr = (qq - zp) * s
                assert Fraction(float(w[zp, qq])) == fr
                want = exact.round_rne(fr, dtype)
                if fr == 0:   # a zero product keeps the IEEE sign of (+0) * s; both zeros are exact
                    assert int(wt[zp, qq]) in (0, 0x8000)
                else:
                    assert int(wt[zp, qq]) == want
        lib = _lib_encode(w.ravel(), dtype) if dtype == "f16" else None
        if lib is not None:
            assert np.array_equal(wt.ravel(), lib)
        else:
            # bf16: the exact products are fp32-exact only when they fit 24 bits; they do (<= 15 bits)
            assert np.array_equal(wt.ravel(), _lib_encode(w.ravel(), dtype))


def test_symmetric_uses_zp_bias_and_qzeros_overrides_it():
    c = synth.make_case(0, 64, 32, 32, "f16", asym=True, seed=8)
    w_sym = ow.dequant_exact(c.b_q, c.scales, None, 32, 8, "f16")
    q = ow.unpack(c.b_q).astype(np.int64)
    s = ieee.t_decode(c.scales, "f16")
    assert np.array_equal(w_sym, (q - 8) * np.repeat(s, 32, axis=0))
    w_asym = ow.dequant_exact(c.b_q, c.scales, c.qzeros, 32, 3, "f16")   # zp_bias ignored
    z = ow.unpack(c.qzeros).astype(np.int64)
    assert np.array_equal(w_asym, (q - np.repeat(z, 32, axis=0)) * np.repeat(s, 32, axis=0))


# ------------------------------------------------------------------------------------------------
# the product
# ------------------------------------------------------------------------------------------------
def _lists(c):
    return (c.a.tolist(), c.b_q.tolist(), c.scales.tolist(),
            None if c.qzeros is None else c.qzeros.tolist(),
            None if c.bias is None else c.bias.tolist())


@pytest.mark.parametrize("dtype,asym,bias,G,K", [
    ("f16", False, False, 32, 64), ("bf16", True, True, 32, 64), ("f16", True, True, 64, 64),
    ("bf16", False, True, 16, 48), ("f16", True, False, 8, 8)])
def test_gemm_brute_force_exact(dtype, asym, bias, G, K):
    c = synth.make_case(3, K, 16, G, dtype, asym=asym, bias=bias, seed=9)
    a, b_q, sc, qz, bi = _lists(c)
    ex = exact.gemm(a, b_q, sc, qz, G, c.zp_bias, bi, dtype)
    ref = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, G, c.zp_bias, c.bias, dtype, weights="exact")
    for m in range(3):
        for n in range(16):
            e = float(ex[m][n])
            assert abs(ref[m, n] - e) <= 1e-12 * (1 + abs(e))


def test_gemm_dequant_t_brute_force():
    dtype = "bf16"
    c = synth.make_case(2, 64, 16, 32, dtype, asym=True, bias=True, seed=10)
    a, b_q, sc, qz, bi = _lists(c)
    ref = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, 32, 8, c.bias, dtype, weights="dequant_t")
    for m in range(2):
        for n in range(16):
            acc = Fraction(0)
            for k in range(64):
                w = exact.weight(b_q, sc, qz, 32, 8, dtype, k, n)
                acc += exact.decode(a[m][k], dtype) * exact.decode(exact.round_rne(w, dtype), dtype)
            acc += exact.decode(bi[n], dtype)
            assert abs(ref[m, n] - float(acc)) <= 1e-12 * (1 + abs(float(acc)))


@pytest.mark.parametrize("asym", [False, True])
def test_q_equal_zp_gives_zero_or_bias(asym):
    M, K, N, G = 5, 256, 64, 64
    c = synth.make_case(M, K, N, G, "f16", asym=asym, bias=True, seed=11)
    if asym:
        b_q = np.repeat(c.qzeros, G, axis=0)      # every weight equals its zero point
    else:
        b_q = np.full((K, N // 8), np.uint32(0x88888888).view(np.int32), np.int32)
    for w in ("exact", "dequant_t"):
        ref = ow.gemm_ref(c.a, b_q, c.scales, c.qzeros, G, 8, None, "f16", weights=w)
        assert np.all(ref == 0)
        refb = ow.gemm_ref(c.a, b_q, c.scales, c.qzeros, G, 8, c.bias, "f16", weights=w)
        assert np.array_equal(refb, np.broadcast_to(ieee.t_decode(c.bias, "f16"), (M, N)))


def test_group_size_k_equals_per_channel_scaling():
    M, K, N = 4, 96, 40
    c = synth.make_case(M, K, N, K, "bf16", asym=True, seed=12)
    ref = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, K, 8, None, "bf16", weights="exact")
    # independent formulation: integer weights first, scale per output column afterwards
    A = _lib_decode(c.a, "bf16")
    q = np.array([[(int(w) >> (4 * j)) & 0xF for w in row.view(np.uint32) for j in range(8)]
                  for row in c.b_q], dtype=np.float64)
    z = np.array([(int(w) >> (4 * j)) & 0xF for w in c.qzeros[0].view(np.uint32) for j in range(8)],
                 dtype=np.float64)
    s = _lib_decode(c.scales[0], "bf16")
    per_channel = (A @ (q - z[None, :])) * s[None, :]
    assert np.allclose(ref, per_channel, rtol=1e-12, atol=1e-12)


def test_linearity_in_a():
    M, K, N, G = 6, 128, 24, 32
    c = synth.make_case(M, K, N, G, "f16", asym=True, bias=False, seed=13)
    a1 = c.a.copy()
    a2 = synth.activations(M, K, "f16", seed=14)
    mask = (np.arange(K) % 2 == 0)
    a1[:, ~mask] = 0          # disjoint supports make a1 + a2 exact
    a2[:, mask] = 0
    a_sum = a1 | a2
    two_a1 = ieee.t_encode_rne(2 * ieee.t_decode(a1, "f16"), "f16")   # exact doubling
    f = lambda a: ow.gemm_ref(a, c.b_q, c.scales, c.qzeros, G, 8, None, "f16", weights="exact")
    assert np.allclose(f(a_sum), f(a1) + f(a2), rtol=1e-12, atol=1e-12)
    assert np.allclose(f(two_a1), 2 * f(a1), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_a_returns_weight_rows(dtype):
    K, N, G = 64, 48, 32
    c = synth.make_case(0, K, N, G, dtype, asym=True, seed=15)
    one = int(ieee.t_encode_rne(np.array([1.0]), dtype)[0])
    a = np.zeros((K, K), np.uint16)
    a[np.arange(K), np.arange(K)] = one
    ref = ow.gemm_ref(a, c.b_q, c.scales, c.qzeros, G, 8, None, dtype, weights="dequant_t")
    wt = ow.dequant_t(c.b_q, c.scales, c.qzeros, G, 8, dtype)
    assert np.array_equal(ow.out_t(ref, dtype), wt)


def test_constant_q_closed_form():
    M, K, N, G, cval = 3, 128, 16, 32, 11
    c = synth.make_case(M, K, N, G, "f16", asym=True, seed=16)
    word = np.uint32(int("".join([f"{cval:X}"] * 8), 16)).view(np.int32)
    b_q = np.full((K, N // 8), word, np.int32)
    ref = ow.gemm_ref(c.a, b_q, c.scales, c.qzeros, G, 8, None, "f16", weights="exact")
    A = _lib_decode(c.a, "f16")
    zp = np.array([[(int(w) >> (4 * j)) & 0xF for w in row.view(np.uint32) for j in range(8)]
                   for row in c.qzeros], dtype=np.float64)
    s = _lib_decode(c.scales, "f16")
    closed = np.zeros((M, N))
    for g in range(K // G):
        closed += A[:, g * G:(g + 1) * G].sum(axis=1)[:, None] * ((cval - zp[g]) * s[g])[None, :]
    assert np.allclose(ref, closed, rtol=1e-12, atol=1e-12)


def test_sub_block_selection_matches_full_product():
    c = synth.make_case(9, 128, 64, 64, "bf16", asym=True, bias=True, seed=17)
    full = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, 64, 8, c.bias, "bf16")
    rows, cols = [0, 4, 8], [0, 7, 8, 33, 63]
    part = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, 64, 8, c.bias, "bf16", rows=rows, cols=cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])


def test_weight_rounding_bound_covers_the_difference():
    for dtype in ("f16", "bf16"):
        c = synth.make_case(8, 1024, 64, 128, dtype, asym=True, seed=18)
        e = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, 128, 8, None, dtype, weights="exact")
        t = ow.gemm_ref(c.a, c.b_q, c.scales, c.qzeros, 128, 8, None, dtype, weights="dequant_t")
        b = ow.weight_rounding_bound(c.a, c.b_q, c.scales, c.qzeros, 128, 8, dtype)
        assert np.all(np.abs(e - t) <= b * (1 + 1e-9) + 1e-12)
        assert np.any(b > 0)


def test_tolerance_predicate():
    for dtype, (atol, rtol) in ow.TOLERANCE.items():
        ref = np.array([0.0, 10.0, -3.0, 0.0])
        inside = np.array([atol * 0.9, 10.0 + (atol + 10 * rtol) * 0.9, -3.0 - (atol + 3 * rtol) * 0.5, np.inf])
        ok = ow.within_tolerance(ieee.t_encode_rne(inside, dtype), ref, dtype)
        assert ok.tolist() == [True, True, True, False]
        outside = np.array([atol * 1.6 + 0.01, 10.0 + (atol + 10 * rtol) * 1.5, np.nan, -1.0])
        assert not ow.within_tolerance(ieee.t_encode_rne(outside, dtype), ref, dtype).any()
    assert ow.TOLERANCE == {"f16": (1e-2, 1e-2), "bf16": (2e-2, 2e-2)}


# ------------------------------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the checks above
# ------------------------------------------------------------------------------------------------
def _runs_clean(fn):
    try:
        fn()
    except AssertionError:
        return False
    return True


def test_mutant_reversed_nibble_order_is_caught(monkeypatch):
    real = ow.unpack

    def bad_unpack(packed, n=None, cols=None):
        w = np.asarray(packed).view(np.uint32)
        cols = np.arange(w.shape[1] * 8 if n is None else n) if cols is None else np.asarray(cols)
        words = w[:, cols >> 3].astype(np.uint64)
        return ((words >> (4 * (7 - (cols & 7))).astype(np.uint64)) & np.uint64(0xF)).astype(np.uint8)

    monkeypatch.setattr(ow, "unpack", bad_unpack)
    assert not _runs_clean(test_pack_golden_words)
    monkeypatch.setattr(ow, "unpack", real)
    assert _runs_clean(test_pack_golden_words)


def test_mutant_wrong_group_index_is_caught(monkeypatch):
    real = ow.dequant_exact

    def bad_dequant(b_q, scales, qzeros, group_size, zp_bias, dtype, cols=None):
        K = b_q.shape[0]
        N = b_q.shape[1] * 8
        cols = np.arange(N) if cols is None else np.asarray(cols)
        q = ow.unpack(b_q, cols=cols).astype(np.int64)
        ng = K // group_size
        zp = ow.zero_points(qzeros, zp_bias, ng, cols)
        s = ieee.t_decode(np.asarray(scales)[:, cols], dtype)
        g_of_k = np.arange(K) % ng                      # planted: k mod (K/G) instead of k // G
        return (q - zp[g_of_k]).astype(np.float64) * s[g_of_k]

    monkeypatch.setattr(ow, "dequant_exact", bad_dequant)
    assert not _runs_clean(lambda: test_gemm_brute_force_exact("bf16", True, True, 32, 64))
    assert not _runs_clean(lambda: test_q_equal_zp_gives_zero_or_bias(True))
    monkeypatch.setattr(ow, "dequant_exact", real)


def test_mutant_dropped_bias_and_zero_point_are_caught(monkeypatch):
    real = ow.zero_points
    monkeypatch.setattr(ow, "zero_points", lambda qz, zb, ng, cols: real(qz, 7, ng, cols) if qz is None
                        else real(qz, zb, ng, cols))
    assert not _runs_clean(lambda: test_q_equal_zp_gives_zero_or_bias(False))
    monkeypatch.setattr(ow, "zero_points", real)

    real_gemm = ow.gemm_ref

    def no_bias(a, b_q, scales, qzeros, G, zp, bias, dtype, **kw):
        return real_gemm(a, b_q, scales, qzeros, G, zp, None, dtype, **kw)

    monkeypatch.setattr(ow, "gemm_ref", no_bias)
    assert not _runs_clean(lambda: test_gemm_brute_force_exact("bf16", True, True, 32, 64))


def test_mutant_rounding_mode_is_caught(monkeypatch):
    real = ieee.t_encode_rne

    def round_half_up(x, dtype):
        x = np.asarray(x, dtype=np.float64)
        bits = real(x, dtype)
        # planted: ties rounded away from zero instead of to even
        v = ieee.t_decode(bits, dtype)
        nxt = ieee.t_decode(bits.astype(np.int64) + 1, dtype)
        tie = np.isfinite(nxt) & (np.abs(x) - np.abs(v) == (np.abs(nxt) - np.abs(v)) / 2) & (np.abs(x) > np.abs(v))
        return np.where(tie, bits + 1, bits).astype(np.uint16)

    monkeypatch.setattr(ieee, "t_encode_rne", round_half_up)
    assert not _runs_clean(lambda: test_encode_ties_and_near_ties_match_library("f16"))


# ----------------------------------------------------------------------------------------------
# packing along K (the [N, K/8] layout of the PR #40977 report)
# ----------------------------------------------------------------------------------------------
def test_pack_k_hand_words():
    # q[k, n] = (k + 2n) % 16 on an 8 x 8 block. Row n of the K-packed tensor holds k = 0..7 of
    # column n, nibble j = k: n = 0 -> 0,1,...,7 = 0x76543210; n = 1 -> 2..9 = 0x98765432;
    # n = 7 -> 14,15,0,1,...,5 = 0x543210FE (worked by hand).
    q = np.array([[(k + 2 * n) % 16 for n in range(8)] for k in range(8)], dtype=np.uint8)
    kp = oracle.pack_k(q).view(np.uint32)
    assert kp.shape == (8, 1)
    assert int(kp[0, 0]) == 0x76543210
    assert int(kp[1, 0]) == 0x98765432
    assert int(kp[7, 0]) == 0x543210FE


def test_pack_k_round_trip_and_relation_to_n_packing():
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(24, 40), dtype=np.uint8)
    kp = oracle.pack_k(q)
    assert kp.shape == (40, 3)
    assert np.array_equal(oracle.unpack_k(kp), q)
    # the same weights in the two layouts: unpacking either gives the same matrix
    assert np.array_equal(oracle.unpack(oracle.pack(q)), oracle.unpack_k(kp))
    # the layouts really differ: the first K-packed word holds column 0, rows 0..7
    assert int(kp.view(np.uint32)[0, 0]) == sum(int(q[k, 0]) << (4 * k) for k in range(8))


def test_prepack_hand_derived_positions():
    """The prepacked layout: each hand-derived position (tests/golden/prepack_words.json) holds the
    word it should, the padding is zero, and the layout has exactly the words it should."""
    g = _golden("prepack_words.json")
    K, N = g["K"], g["N"]
    kk, cc = np.meshgrid(np.arange(K), np.arange(N // 8), indexing="ij")
    b_q = (1000 * kk + cc + 1).astype(np.int32)
    pp = oracle.prepack(b_q)
    assert list(pp.shape) == g["shape"]
    flat = pp.reshape(-1)
    for e in g["entries"]:
        assert flat[e["flat"]] == 1000 * e["k"] + e["c"] + 1, e["why"]
    for z in g["zeros"]:
        assert flat[z["flat"]] == 0, z["why"]
    assert int((flat == 0).sum()) == g["zero_words_total"]


def test_prepack_round_trip_and_block_contents():
    """unprepack(prepack(b)) == b on shapes with ragged K and N tails, and every 64-row block of a
    tile holds exactly the words of those rows and columns (as a set), whatever their order."""
    rng = np.random.default_rng(7)
    for K, N in ((64, 256), (130, 264), (200, 1000), (1, 8)):
        b = rng.integers(1, 2 ** 31, size=(K, N // 8), dtype=np.int64).astype(np.int32)
        pp = oracle.prepack(b)
        assert np.array_equal(oracle.unprepack(pp, K, N), b)
        for t in range(pp.shape[0]):
            for kb in range(pp.shape[1]):
                block = pp[t, kb]
                want = b[kb * 64:(kb + 1) * 64, t * 32:(t + 1) * 32]
                for r in range(want.shape[0]):
                    assert sorted(block[r][block[r] != 0].tolist()) == sorted(want[r].tolist())

"""Pins for the CPU oracle, against things other than the oracle itself.

* library routines: numpy's float16 and torch's bfloat16 / float8_e4m3fn conversions decode every
  fp16, bf16 and E4M3 code and round doubles, so the oracle's single parametric minifloat
  decoder and rounder are checked on three formats; E2M1 runs through the same code;
* landmarks stated on the pages (tests/golden/format_landmarks.txt);
* brute force in exact rational arithmetic (fractions.Fraction) from the raw bytes, with an
  independent table-search rounding, on tiny shapes of every format;
* closed forms and invariants: integer matmul, one-hot activations, implicit zero point,
  row independence, linearity, sign flips, the exactness of the NVFP4 scale fold;
* mutation checks: a brute force with a planted mistake (nibble order, zero point, scale block,
  transposed operand) must disagree with the oracle, so the comparison above is not vacuous.
"""
from __future__ import annotations

import bisect
import os
from fractions import Fraction

import dataclasses

import numpy as np
import pytest
import torch

from block_scaled_bit_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def landmarks():
    out = {}
    with open(os.path.join(GOLDEN, "format_landmarks.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


# ------------------------------------------------------------------ library-side code tables
def lib_f16_values():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)


def lib_bf16_values():
    t = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def lib_e4m3_values():
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def same(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return bool(np.all((a == b) | (np.isnan(a) & np.isnan(b))))


# ------------------------------------------------------------------ decoders vs libraries
def test_f16_decode_matches_numpy_all_codes(orc):
    assert same(orc.minifloat_values(np.arange(65536), orc.F16), lib_f16_values())


def test_bf16_decode_matches_torch_all_codes(orc):
    assert same(orc.minifloat_values(np.arange(65536), orc.BF16), lib_bf16_values())


def test_e4m3_decode_matches_torch_all_codes(orc):
    assert same(orc.e4m3_table(), lib_e4m3_values())


def test_e4m3_landmarks(orc):
    L = landmarks()
    t = orc.e4m3_table()
    finite = t[np.isfinite(t)]
    assert finite.max() == L["e4m3_max"] and t[0x7E] == 448.0
    assert finite[finite > 0].min() == L["e4m3_min_positive"] and t[0x01] == 2.0 ** -9
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF]) and np.isnan(t).sum() == 2
    assert not np.isinf(t).any()


def significand_bits(v: float) -> int:
    if v == 0:
        return 0
    m, _ = np.frexp(abs(v))
    bits = 0
    while m != 0:
        m = m * 2
        bits += 1
        m -= np.floor(m)
    return bits


def test_e2m1_table_structure_and_landmarks(orc):
    L = landmarks()
    t = orc.e2m1_table()
    pos = t[:8]
    assert np.all(np.diff(pos) > 0), "codes 0..7 are increasing magnitudes"
    assert pos[0] == 0.0
    assert same(t[8:], -pos), "bit 3 is the sign"
    assert pos.max() == L["e2m1_max"]
    assert pos[1:].min() == L["e2m1_min_positive"]
    assert max(significand_bits(v) for v in pos) == L["e2m1_significand_bits"]
    # every E2M1 value is an E4M3 value (both are binary minifloats with more range in E4M3)
    e4 = set(orc.e4m3_table()[np.isfinite(orc.e4m3_table())].tolist())
    assert set(t.tolist()) <= e4
    # the standard's printed magnitudes (OCP MX formats, E2M1 table)
    assert pos.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e4m3_is_lossless_in_f16_and_bf16(orc):
    """E4M3 -> FP16/BF16 is lossless (FP8 tensor-core paragraph of the decode-GEMV page)."""
    t = orc.e4m3_table()
    f = t[np.isfinite(t)]
    assert np.array_equal(f.astype(np.float16).astype(np.float64), f)
    bf = torch.from_numpy(f.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf, f)
    assert max(significand_bits(v) for v in f) == landmarks()["e4m3_significand_bits"]


def test_nvfp4_scale_fold_is_exact_in_16_bits(orc):
    """E2M1 x E4M3 needs at most 6 significand bits and lies in [2^-10, 2688], so it is exact in
    fp16 and bf16 (NVFP4 tensor-core paragraph of the decode-GEMV page); all 16 x 126 pairs."""
    L = landmarks()
    e2 = orc.e2m1_table()
    e4 = orc.e4m3_table()[1:0x7F]          # positive finite, nonzero
    prod = np.outer(e2, e4).ravel()
    assert np.array_equal(prod.astype(np.float16).astype(np.float64), prod)
    bf = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf, prod)
    nz = np.abs(prod[prod != 0])
    assert nz.max() == L["fold_max"] and nz.min() == L["fold_min_positive"]
    assert max(significand_bits(v) for v in nz) == L["fold_significand_bits"]


# ------------------------------------------------------------------ rounding vs libraries
def rounding_probe_values(rng, top_exp=17, bottom_exp=-30):
    x = [0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
         3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
         np.inf, -np.inf, np.nan]
    x += list(rng.standard_normal(20000))
    x += list(np.ldexp(rng.uniform(0.5, 1, 20000), rng.integers(bottom_exp, top_exp, 20000)))
    # exact ties between neighbouring fp16 values, both parities
    h = rng.integers(1, 0x7BFF, 5000).astype(np.uint16).view(np.float16).astype(np.float64)
    h2 = (rng.integers(1, 0x7BFF, 5000) + 0).astype(np.uint16)
    nxt = (h2 + 1).view(np.float16).astype(np.float64)
    x += list((h2.view(np.float16).astype(np.float64) + nxt) / 2) + list(h)
    x = np.array(x, dtype=np.float64)
    return np.concatenate([x, -x])


def test_round_f16_matches_numpy(orc):
    x = rounding_probe_values(np.random.default_rng(1))
    ours = orc.round_minifloat(x, orc.F16).astype(np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(ours[nan].view(np.float16)))


def test_round_bf16_matches_torch_on_float32_inputs(orc):
    rng = np.random.default_rng(2)
    with np.errstate(over="ignore"):
        x = rounding_probe_values(rng, top_exp=130, bottom_exp=-140).astype(np.float32)
    # fp32 numbers whose low 16 bits sit exactly on the bf16 tie point, both parities
    b = rng.integers(0, 2 ** 31 - 2 ** 24, 20000, dtype=np.int64).astype(np.uint32)
    ties = ((b & 0xFFFF0000) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([3.3895314e38, 3.4e38, 1e-40, -1e-45])])
    x = x[np.isfinite(x)]
    ours = orc.round_minifloat(x.astype(np.float64), orc.BF16).astype(np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def table_rne(frac: Fraction, values: np.ndarray, max_code: int) -> int:
    """Round an exact rational to a 16-bit IEEE format by searching its positive code table;
    ties go to the even code.  An implementation independent of the oracle's arithmetic."""
    neg = frac < 0
    a = -frac if neg else frac
    pos = [Fraction(float(v)) for v in values[: max_code + 1]]
    i = bisect.bisect_right(pos, a) - 1
    top_ulp = pos[max_code] - pos[max_code - 1]
    if a >= pos[max_code] + top_ulp / 2:
        code = max_code + 1                      # inf
    elif i == max_code or pos[i] == a:
        code = i
    else:
        lo, hi = pos[i], pos[i + 1]
        if a - lo < hi - a:
            code = i
        elif a - lo > hi - a:
            code = i + 1
        else:
            code = i if i % 2 == 0 else i + 1
    return code | (0x8000 if neg and code != 0 else 0)


_F16_VALUES = None
_BF16_VALUES = None


def act_table(act):
    global _F16_VALUES, _BF16_VALUES
    if act == "f16":
        if _F16_VALUES is None:
            _F16_VALUES = lib_f16_values()
        return _F16_VALUES, 0x7BFF
    if _BF16_VALUES is None:
        _BF16_VALUES = lib_bf16_values()
    return _BF16_VALUES, 0x7F7F


def test_round_bf16_matches_exact_rational_rounding(orc):
    rng = np.random.default_rng(3)
    vals, maxc = act_table("bf16")
    x = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.integers(-5, 5, 300),
                        # doubles just around bf16 ties (not representable in fp32)
                        (1 + 2.0 ** -8) * (1 + rng.choice([-1, 1], 200) * 2.0 ** -40)])
    ours = orc.round_minifloat(x, orc.BF16)
    for xi, oi in zip(x, ours):
        assert table_rne(Fraction(float(xi)), vals, maxc) == int(oi)


# ------------------------------------------------------------------ brute force from raw bytes
E2M1_MAGNITUDES = [0, Fraction(1, 2), 1, Fraction(3, 2), 2, 3, 4, 6]   # OCP MX E2M1 table


def frac_e2m1(code):
    v = Fraction(E2M1_MAGNITUDES[code & 7])
    return -v if code & 8 else v


_E4M3_FRACS = None


def frac_e4m3(code):
    global _E4M3_FRACS
    if _E4M3_FRACS is None:
        _E4M3_FRACS = [Fraction(float(v)) if np.isfinite(v) else None for v in lib_e4m3_values()]
    return _E4M3_FRACS[int(code)]


def frac_f16(bits):
    return Fraction(float(np.uint16(bits).view(np.float16)))


def frac_act(bits, act):
    if act == "f16":
        return frac_f16(bits)
    return Fraction(float(torch.tensor([int(bits)], dtype=torch.int32).to(torch.int16)
                          .view(torch.bfloat16).item()))


def brute_deq(case, n, k, mutate=None):
    """Exact rational deq(n, k) straight from the stored bytes.  `mutate` plants one mistake."""
    bs, nb = case.block_size, case.K // case.block_size
    b = k // bs
    if mutate == "scale_block":
        b = min(nb - 1, (k + 1) // bs)
    if case.fmt in ("int4", "nvfp4"):
        byte = int(case.W[n, k // 2])
        shift = 4 * (k % 2) if mutate != "nibble_order" else 4 * (1 - k % 2)
        q = (byte >> shift) & 0xF
    else:
        q = int(case.W[n, k])
    if case.fmt == "int4":
        zp = 8
        if case.has_zp and mutate != "ignore_zp":
            zp = (int(case.zp[n, b // 2]) >> (4 * (b % 2))) & 0xF
        return (q - zp) * frac_f16(case.scales[n, b])
    if case.fmt == "int8":
        zp = int(case.zp[n, b]) if (case.has_zp and mutate != "ignore_zp") else 128
        return (q - zp) * frac_f16(case.scales[n, b])
    if case.fmt == "fp8":
        return frac_e4m3(q) * Fraction(float(case.scales[n, b]))
    return frac_e2m1(q) * frac_e4m3(case.scales[n, b]) * Fraction(float(case.gscale[0]))


def brute_gemv(case, mutate=None):
    vals, maxc = act_table(case.act)
    M, N, K = case.M, case.N, case.K
    a = [[frac_act(case.A[m, k], case.act) for k in range(K)] for m in range(M)]
    deq = [[brute_deq(case, n, k, mutate) for k in range(K)] for n in range(N)]
    exact = [[sum((a[m][k] * deq[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
             for m in range(M)]
    if mutate == "transpose":   # a transposed operand: rows of A against W read column-wise
        exact = [[sum((a[m][k] * deq[k % N][n % K] for k in range(K)), Fraction(0))
                  for n in range(N)] for m in range(M)]
    bias = getattr(case, "bias", None)
    if bias is not None and mutate != "bias_dropped":
        # bias[n] added to every row m before the one rounding
        col = (lambda n: (n + 1) % N) if mutate == "bias_column" else (lambda n: n)
        exact = [[exact[m][n] + frac_act(bias[col(n)], case.act) for n in range(N)]
                 for m in range(M)]
    bits = np.array([[table_rne(e, vals, maxc) for e in row] for row in exact], dtype=np.uint16)
    return bits, exact


TINY = [
    ("int4", "f16", 32, True), ("int4", "bf16", 16, True), ("int4", "f16", 64, False),
    ("int4", "bf16", 128, False), ("int8", "f16", 32, True), ("int8", "bf16", 16, False),
    ("int8", "f16", 128, True), ("fp8", "f16", 128, False), ("fp8", "bf16", 128, False),
    ("nvfp4", "f16", 16, False), ("nvfp4", "bf16", 16, False),
]


def tiny_case(fmt, act, bs, zp, M=3, N=5, K=None, seed=7):
    K = K or max(2 * bs, 64)
    return synth.make_case(fmt, act, bs, zp, N, K, M, seed + bs)


@pytest.mark.parametrize("fmt,act,bs,zp", TINY)
def test_oracle_matches_exact_rational_brute_force(orc, fmt, act, bs, zp):
    case = tiny_case(fmt, act, bs, zp)
    ybits, exact, absdot = orc.gemv(case)
    bits, ex = brute_gemv(case)
    assert np.array_equal(ybits, bits)
    ex64 = np.array([[float(e) for e in row] for row in ex])
    assert np.allclose(exact, ex64, rtol=1e-12, atol=1e-300)
    # dequant agrees exactly with the brute force too
    deq = orc.dequant(case)
    for n in range(case.N):
        for k in range(case.K):
            assert Fraction(float(deq[n, k])) == brute_deq(case, n, k)
    assert np.all(absdot >= np.abs(exact))


@pytest.mark.parametrize("mutation,fmt,bs,zp", [
    ("nibble_order", "int4", 32, True), ("nibble_order", "nvfp4", 16, False),
    ("ignore_zp", "int4", 32, True), ("ignore_zp", "int8", 32, True),
    ("scale_block", "int8", 16, True), ("scale_block", "fp8", 128, False),
    ("transpose", "int8", 32, False),
])
def test_brute_force_detects_planted_mistakes(orc, mutation, fmt, bs, zp):
    """A mistake planted in the (CPU) brute force must make it disagree with the oracle: the
    brute-force comparison can tell a right oracle from a wrong one."""
    case = tiny_case(fmt, "f16", bs, zp, K=max(2 * bs, 64))
    ybits, _, _ = orc.gemv(case)
    bad, _ = brute_gemv(case, mutate=mutation)
    assert not np.array_equal(ybits, bad)


# ------------------------------------------------------------------ closed forms / invariants
def test_integer_matmul_special_case(orc):
    """scale 1, zero point 0, small integer activations: y is an integer matmul, rounded."""
    rng = np.random.default_rng(11)
    N, K, M = 7, 96, 4
    case = synth.make_case("int8", "f16", 32, True, N, K, M, 5)
    case.scales[:] = np.float16(1.0).view(np.uint16)
    case.zp[:] = 0
    ai = rng.integers(-3, 4, size=(M, K))
    case.A = ai.astype(np.float16).view(np.uint16)
    y_int = ai @ case.W.astype(np.int64).T
    ybits, exact, _ = orc.gemv(case)
    assert np.array_equal(exact, y_int.astype(np.float64))
    assert np.array_equal(ybits, y_int.astype(np.float64).astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("fmt,act,bs,zp", TINY)
def test_one_hot_activation_selects_a_weight(orc, fmt, act, bs, zp):
    case = tiny_case(fmt, act, bs, zp, M=4, N=6)
    ks = [0, 1, case.K // 2 + 3, case.K - 1]
    one = np.float16(1.0).view(np.uint16) if act == "f16" else np.uint16(0x3F80)
    case.A = np.zeros((4, case.K), dtype=np.uint16)
    for m, k in enumerate(ks):
        case.A[m, k] = one
    deq = orc.dequant(case)
    ybits, exact, _ = orc.gemv(case)
    for m, k in enumerate(ks):
        assert np.array_equal(exact[m], deq[:, k])
        # compare values: a sum that starts at +0 turns a -0 weight into +0
        got = orc.act_values(ybits[m], act)
        assert np.array_equal(got, orc.act_values(orc.round_act(deq[:, k], act), act))


@pytest.mark.parametrize("fmt,zpval", [("int4", 8), ("int8", 128)])
def test_implicit_zero_point_equals_explicit(orc, fmt, zpval):
    case = synth.make_case(fmt, "f16", 32, True, 9, 128, 3, 21)
    case.zp[:] = 0x88 if fmt == "int4" else zpval
    explicit = orc.gemv(case)
    case.has_zp = False
    implicit = orc.gemv(case)
    assert all(np.array_equal(a, b) for a, b in zip(explicit, implicit))


@pytest.mark.parametrize("fmt,act,bs,zp", TINY)
def test_rows_do_not_depend_on_M(orc, fmt, act, bs, zp):
    case16 = tiny_case(fmt, act, bs, zp, M=16, N=4)
    y16, e16, _ = orc.gemv(case16)
    for M in (1, 3, 8):
        yM, eM, _ = orc.gemv(case16.with_M(M))
        assert np.array_equal(yM, y16[:M]) and np.array_equal(eM, e16[:M])


def test_linearity_in_A(orc):
    case = synth.make_case("fp8", "f16", 128, False, 8, 256, 3, 31)
    _, e1, _ = orc.gemv(case)
    a = case.A.view(np.float16).astype(np.float64)
    case.A = (2 * a).astype(np.float16).view(np.uint16)   # exact doubling
    _, e2, _ = orc.gemv(case)
    assert np.array_equal(e2, 2 * e1)


def test_sign_flips_negate(orc):
    c4 = synth.make_case("nvfp4", "f16", 16, False, 6, 128, 2, 41)
    _, e, _ = orc.gemv(c4)
    c4.W = c4.W ^ np.uint8(0x88)        # sign bit of both E2M1 codes in each byte
    _, e_neg, _ = orc.gemv(c4)
    assert np.array_equal(e_neg, -e)
    c8 = synth.make_case("fp8", "bf16", 128, False, 6, 256, 2, 42)
    _, e, _ = orc.gemv(c8)
    c8.W = c8.W ^ np.uint8(0x80)
    _, e_neg, _ = orc.gemv(c8)
    assert np.array_equal(e_neg, -e)


def test_subset_rows_match_full(orc):
    case = synth.make_case("int4", "bf16", 32, True, 40, 256, 5, 51)
    y, e, d = orc.gemv(case)
    rows = [39, 0, 17, 17, 5]
    ys, es, ds = orc.gemv(case, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(es, e[:, rows])
    assert np.array_equal(ds, d[:, rows])


# ------------------------------------------------------------------ the optional bias
BIAS_TINY = [("int4", "f16", 32, True), ("int8", "bf16", 16, False), ("fp8", "f16", 128, False),
             ("nvfp4", "bf16", 16, False)]


@pytest.mark.parametrize("fmt,act,bs,zp", BIAS_TINY)
def test_oracle_with_bias_matches_exact_rational_brute_force(orc, fmt, act, bs, zp):
    """y = A . deq(W)^T + bias (bias[n] broadcast over the rows, one rounding): the oracle equals
    the exact rational result rounded by the independent table search."""
    case = tiny_case(fmt, act, bs, zp).with_bias(sigma=4.0)
    ybits, exact, absdot = orc.gemv(case)
    bits, ex = brute_gemv(case)
    assert np.array_equal(ybits, bits)
    ex64 = np.array([[float(e) for e in row] for row in ex])
    assert np.allclose(exact, ex64, rtol=1e-12, atol=1e-300)
    _, _, absdot0 = orc.gemv(dataclasses.replace(case, bias=None))
    assert np.array_equal(absdot, absdot0 + np.abs(orc.act_values(case.bias, act))[None, :])


@pytest.mark.parametrize("mutation", ["bias_dropped", "bias_column"])
def test_brute_force_detects_planted_bias_mistakes(orc, mutation):
    case = tiny_case("int8", "f16", 32, True).with_bias(sigma=4.0)
    ybits, _, _ = orc.gemv(case)
    bad, _ = brute_gemv(case, mutate=mutation)
    assert not np.array_equal(ybits, bad)


@pytest.mark.parametrize("fmt,act,bs,zp", BIAS_TINY)
def test_zero_activations_give_the_bias(orc, fmt, act, bs, zp):
    """With A = 0 every product is zero, so y is the bias itself (it is already representable)."""
    case = synth.make_case(fmt, act, bs, zp, 37, 256, 3, 5).with_bias()
    case = dataclasses.replace(case, A=np.zeros_like(case.A))
    ybits, exact, _ = orc.gemv(case)
    b = orc.act_values(case.bias, act)
    assert np.array_equal(orc.act_values(ybits, act), np.broadcast_to(b, ybits.shape))
    assert np.array_equal(exact, np.broadcast_to(b, exact.shape))


def test_bias_adds_to_the_exact_sum(orc):
    """The bias enters after the k-sum: exact(with bias) - exact(without) = bias, when the sums are
    small integers (s = 1, zp = 0 int8 weights, integer activations) so that nothing rounds."""
    case = synth.make_case("int8", "f16", 32, True, 21, 128, 4, 9,
                           scale_range=(1.0, 1.0), zp_range=(0, 0))
    A = synth.to_f16_bits(np.random.default_rng(3).integers(-3, 4, size=case.A.shape))
    case = dataclasses.replace(case, A=A).with_bias(sigma=8.0)
    _, e_b, _ = orc.gemv(case)
    _, e_0, _ = orc.gemv(dataclasses.replace(case, bias=None))
    assert np.array_equal(e_b - e_0, np.broadcast_to(orc.act_values(case.bias, "f16"), e_b.shape))


# ------------------------------------------------------------------ the dense small-N GEMV
def brute_dense(A, B, act, mutate=None):
    """Exact rational y = A . B ([M, K] x [K, N], row-major bit patterns), rounded by the table
    search.  `mutate` plants one mistake."""
    vals, maxc = act_table(act)
    M, K = A.shape
    N = B.shape[1]
    a = [[frac_act(A[m, k], act) for k in range(K)] for m in range(M)]
    if mutate == "transposed_B":   # B read as if it were stored [N, K]
        flat = B.reshape(-1)
        b = [[frac_act(flat[n * K + k], act) for n in range(N)] for k in range(K)]
    else:
        b = [[frac_act(B[k, n], act) for n in range(N)] for k in range(K)]
    row = (lambda m: (m + 1) % M) if mutate == "row_of_A" else (lambda m: m)
    exact = [[sum((a[row(m)][k] * b[k][n] for k in range(K)), Fraction(0)) for n in range(N)]
             for m in range(M)]
    bits = np.array([[table_rne(e, vals, maxc) for e in r] for r in exact], dtype=np.uint16)
    return bits, exact


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 64), (3, 5, 40), (2, 16, 33)])
def test_dense_oracle_matches_exact_rational_brute_force(orc, act, M, N, K):
    A, B = synth.dense_operands(act, M, N, K, seed=M * 100 + N + K)
    ybits, exact, absdot = orc.dense_gemv(A, B, act)
    bits, ex = brute_dense(A, B, act)
    assert np.array_equal(ybits, bits)
    assert np.allclose(exact, np.array([[float(e) for e in r] for r in ex]), rtol=1e-12, atol=1e-300)
    assert np.all(absdot >= np.abs(exact))


@pytest.mark.parametrize("mutation", ["transposed_B", "row_of_A"])
def test_dense_brute_force_detects_planted_mistakes(orc, mutation):
    A, B = synth.dense_operands("f16", 3, 6, 48, seed=5)
    ybits, _, _ = orc.dense_gemv(A, B, "f16")
    bad, _ = brute_dense(A, B, "f16", mutate=mutation)
    assert not np.array_equal(ybits, bad)


@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_dense_one_hot_activations_select_a_row_of_B(orc, act):
    """A = e_k picks row k of B: y[m, :] = B[k_m, :] exactly."""
    K, N = 96, 24
    _, B = synth.dense_operands(act, 1, N, K, seed=9)
    ks = [0, 17, 95]
    one = synth.to_f16_bits(np.ones(1))[0] if act == "f16" else synth.to_bf16_bits(np.ones(1))[0]
    A = np.zeros((len(ks), K), dtype=np.uint16)
    for m, k in enumerate(ks):
        A[m, k] = one
    ybits, _, _ = orc.dense_gemv(A, B, act)
    assert np.array_equal(orc.act_values(ybits, act), orc.act_values(B[ks, :], act))


def test_dense_small_integers_are_an_integer_matmul(orc):
    rng = np.random.default_rng(11)
    a = rng.integers(-4, 5, size=(4, 64))
    b = rng.integers(-4, 5, size=(64, 9))
    ybits, exact, _ = orc.dense_gemv(synth.to_f16_bits(a), synth.to_f16_bits(b), "f16")
    assert np.array_equal(exact, (a @ b).astype(np.float64))
    assert np.array_equal(orc.act_values(ybits, "f16"), (a @ b).astype(np.float64))


# ------------------------------------------------------------------ the parity bar itself
def test_ulp_matches_the_formats_spacing(orc):
    """ulp(|v|) is the distance from v to the next larger value of the dtype, subnormals
    included: numpy's float16 spacing, and for bf16 the difference of neighbouring codes."""
    codes = np.arange(1, 0x7BFF, 37, dtype=np.uint16)  # positive finite fp16, subnormals first
    v16 = codes.view(np.float16).astype(np.float64)
    assert np.array_equal(orc.ulp(v16, "f16"), np.spacing(codes.view(np.float16)).astype(np.float64))
    bcodes = np.arange(1, 0x7F7F, 41, dtype=np.uint16)  # positive finite bf16
    vb = orc.act_values(bcodes, "bf16")
    nxt = orc.act_values(bcodes + 1, "bf16")
    assert np.array_equal(orc.ulp(vb, "bf16"), nxt - vb)


def test_tolerance_check_accepts_the_oracle_and_flags_a_planted_error(orc):
    case = synth.make_case("int8", "f16", 32, True, 40, 256, 3, 12)
    ref_bits, _, absdot = orc.gemv(case)
    bad, worst, _ = orc.tolerance_violations(case, ref_bits)
    assert bad == 0 and worst == 0.0
    # one output off by twice its bound
    y = orc.act_values(ref_bits, "f16")
    bound = orc.ulp(y, "f16") + 1e-3 * absdot
    planted = y.copy()
    planted[1, 7] += 2 * bound[1, 7]
    bad, worst, _ = orc.tolerance_violations(case, synth.to_f16_bits(planted))
    assert bad == 1 and worst > 1.0
    # within the bound: accepted
    near = y.copy()
    near[2, 3] += 0.5 * bound[2, 3]
    bits = synth.to_f16_bits(near)
    ok, _, _ = orc.tolerance_violations(case, bits)
    assert ok == 0


def test_tolerance_check_requires_infinities_to_match(orc):
    """Where the oracle's result overflows, the GPU value must be the same infinity."""
    case = synth.make_case("int8", "f16", 32, False, 8, 256, 1, 3, scale_range=(60000.0, 60000.0))
    case = dataclasses.replace(case, A=synth.to_f16_bits(np.full((1, 256), 60000.0)))
    ref_bits, _, _ = orc.gemv(case)
    vals = orc.act_values(ref_bits, "f16")
    assert np.all(np.isinf(vals))
    assert orc.tolerance_violations(case, ref_bits)[0] == 0
    finite = synth.to_f16_bits(np.full(vals.shape, 65504.0) * np.sign(vals))
    assert orc.tolerance_violations(case, finite)[0] == vals.size

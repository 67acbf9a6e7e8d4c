"""Pins for the CPU oracle: checks against facts the oracle does not compute.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle disagrees with a hand-computed golden value, an exact rational
result, a closed form, an invariant, or a float64 brute force.  The same
pins run against the real oracle (they must all pass) and against mutated
copies of it (each mutant must fail at least one), see
test_oracle_mutants.py.

Method: FlagTree pull request "[TLERaw] Add NVSHMEM allreduce RMSNorm
tutorial", Summary (contract) and Implementation section 3 (epilogue).
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import bf16_exact as bx

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GOLDEN = os.path.join(GOLDEN_DIR, "hand_rows.txt")
GOLDEN_F32 = os.path.join(GOLDEN_DIR, "hand_rows_f32.txt")


# ------------------------------------------------------------------- goldens
def load_golden(path: str = GOLDEN) -> dict:
    cases, cur = {}, None
    with open(path) as fh:
        for raw in fh:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = cases.setdefault(line[1:-1], {})
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            cur[k] = v
    return cases


def _row(s: str) -> np.ndarray:
    return np.array([bx.bits(t) for t in s.split()], np.uint16)


def _compare(name, key, got, want):
    got = np.asarray(got).ravel()
    nan_w = bx.nan_mask(want)
    assert np.array_equal(bx.nan_mask(got), nan_w), f"{name}.{key}: NaN positions {got} vs {want}"
    ok = np.where(nan_w, True, got == want)
    assert ok.all(), f"{name}.{key}: got {[hex(v) for v in got]} want {[hex(v) for v in want]}"


def _row_f32(s: str) -> np.ndarray:
    vals = []
    for t in s.split():
        q = Fraction(t)
        f = np.float32(float(q))
        assert Fraction(float(f)) == q, f"{t} is not exact in fp32"
        vals.append(f)
    return np.array(vals, np.float32)


def pin_golden_cases(O, path=GOLDEN):
    for name, c in load_golden(path).items():
        xs = []
        r = 0
        f32 = c.get("partial_dtype") == "f32"
        while f"x{r}" in c:
            xs.append((_row_f32 if f32 else _row)(c[f"x{r}"])[None, :])
            r += 1
        res = _row(c["residual"])[None, :]
        w = _row(c["weight"])
        eps = float(c["eps"])
        red, ro, nrm = O.forward(xs, res, w, eps)
        for key, got in (("reduced", red), ("residual_out", ro), ("norm_out", nrm)):
            if key in c:
                _compare(name, key, got, _row(c[key]))


# ------------------------------------------------------- format conversions
def pin_bf16_widening_all_patterns(O):
    for b in range(0, 1 << 16, 7):            # every 7th pattern, all classes
        v = O.bf16_to_f32(b)
        d = bx.decode(b)
        if isinstance(d, float):
            if np.isnan(d):
                assert np.isnan(v), hex(b)
            else:
                assert v == d, hex(b)
        else:
            assert Fraction(v) == d, hex(b)
    for b in (0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F,
              0x7F80, 0xFF80, 0x3F80, 0xBF80):
        d = bx.decode(b)
        v = O.bf16_to_f32(b)
        assert (Fraction(v) == d) if not isinstance(d, float) else (v == d), hex(b)
    assert np.signbit(O.bf16_to_f32(0x8000))


def _f32_from_bits(u: int) -> float:
    return float(np.array([u], np.uint32).view(np.float32)[0])


def pin_bf16_rounding_vs_exact(O):
    rng = np.random.default_rng(1234)
    pats = list(rng.integers(0, 1 << 32, 4000, dtype=np.uint64))
    # ties, just-below/above ties, subnormals, overflow edge, specials
    for hi in (0x3F80, 0x3F81, 0xBF80, 0x0000, 0x0001, 0x7F7F, 0x8080, 0x4B80):
        for lo in (0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
            pats.append((hi << 16) | lo)
    pats += [0x7F800000, 0xFF800000, 0x7F800001, 0xFF800001, 0x7FC00000,
             0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x00000001, 0x80000001]
    for u in pats:
        u = int(u)
        f = _f32_from_bits(u)
        got = O.f32_bits_to_bf16(u)
        if np.isnan(f):
            assert bx.is_nan(got), (hex(u), hex(got))
            assert (got & 0x8000) == (u >> 16 & 0x8000), "NaN sign kept"
            continue
        want = bx.round_rne(f if (f == 0 or np.isinf(f)) else Fraction(f))
        assert got == want, (hex(u), hex(got), hex(want))


def pin_overflow_and_subnormal(O):
    mx = np.array([[0x7F7F]], np.uint16)
    red, _, _ = O.forward([mx, mx], np.zeros((1, 1), np.uint16),
                          np.array([bx.bits(1)], np.uint16), 1e-6)
    assert red[0, 0] == bx.POS_INF, hex(red[0, 0])
    tiny = np.array([[0x0001, 0x8001]], np.uint16)          # +-2^-133
    red, _, _ = O.forward([tiny, tiny], np.zeros((1, 2), np.uint16),
                          np.array([bx.bits(1)] * 2, np.uint16), 1e-6)
    assert list(red[0]) == [0x0002, 0x8002], [hex(v) for v in red[0]]


# ------------------------------------------------------------- rank sum (a1)
def pin_rank_sum_integers(O):
    """Integer-valued partials: the exact integer sum, rounded once."""
    rng = np.random.default_rng(7)
    for W in (1, 2, 3, 5, 8, 16, 32):
        vals = rng.integers(-128, 129, size=(W, 257))
        xs = [np.array([bx.bits(int(v)) for v in row], np.uint16) for row in vals]
        got = O.rank_sum(xs)
        want = [bx.round_rne(Fraction(int(s))) if s != 0 else 0
                for s in vals.sum(axis=0)]
        assert list(got) == want, f"W={W}"


def _fp32_exact(q: Fraction) -> bool:
    f = np.float32(float(q))
    return Fraction(float(f)) == q


def pin_rank_sum_brute_force(O):
    """bf16 partials of mixed magnitude: compare with the exact rational sum.

    Where every prefix sum is exact in fp32 the oracle must give the exact
    sum rounded once; elsewhere fp32 rounding can move it by at most 1 ulp."""
    rng = np.random.default_rng(11)
    n_exact = 0
    for W in (2, 3, 4):
        mags = rng.normal(size=(W, 600)) * np.exp2(rng.integers(-12, 12, (W, 600)))
        xs = [((m.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)) for m in mags]
        got = O.rank_sum(xs)
        for i in range(got.size):
            terms = [bx.decode(int(x[i])) for x in xs]
            prefix, exact = terms[0], True
            for t in terms[1:]:
                prefix = prefix + t
                exact &= _fp32_exact(prefix)
            want = bx.round_rne(prefix) if prefix != 0 else int(got[i]) & 0x8000
            if exact:
                n_exact += 1
                assert int(got[i]) == want or (prefix == 0 and (int(got[i]) & 0x7FFF) == 0), \
                    (W, i, hex(int(got[i])), hex(want))
            else:
                assert bx.ulp_diff(int(got[i]), want) <= 1, (W, i)
    assert n_exact > 1000


# ----------------------------------------------------------- residual (a2)
def pin_residual_add_brute_force(O):
    rng = np.random.default_rng(5)
    a = (rng.normal(size=3000) * np.exp2(rng.integers(-20, 20, 3000))).astype(np.float32)
    b = (rng.normal(size=3000) * np.exp2(rng.integers(-20, 20, 3000))).astype(np.float32)
    ab = (a.view(np.uint32) >> 16).astype(np.uint16)
    bb = (b.view(np.uint32) >> 16).astype(np.uint16)
    got = O.residual_add(ab, bb)
    for i in range(got.size):
        s = bx.decode(int(ab[i])) + bx.decode(int(bb[i]))
        if s == 0:
            assert (int(got[i]) & 0x7FFF) == 0
            continue
        want = bx.round_rne(s)
        if _fp32_exact(s):
            assert int(got[i]) == want, (i, hex(int(got[i])), hex(want))
        else:
            assert bx.ulp_diff(int(got[i]), want) <= 1


def pin_residual_adds_rounded_reduced(O):
    """The residual is added to the bf16-rounded reduced value: x = (1, 2^-8)
    gives reduced 1.0 (tie to even); + residual 2^-8 -> 1 + 2^-8 -> 1.0 again.
    Adding to the unrounded fp32 sum would give 1 + 2^-7 = 1.0078125."""
    one, q = bx.bits(1), bx.bits(Fraction(1, 256))
    xs = [np.array([[one]], np.uint16), np.array([[q]], np.uint16)]
    red, ro, _ = O.forward(xs, np.array([[q]], np.uint16),
                           np.array([one], np.uint16), 1e-6)
    assert red[0, 0] == one and ro[0, 0] == one, (hex(red[0, 0]), hex(ro[0, 0]))


# --------------------------------------------------------- RMSNorm (a3, a4)
def pin_rmsnorm_float64_brute_force(O):
    """Recompute the normalisation in float64 from the oracle's residual_out,
    round once: the oracle's fp32 result must be within 1 bf16 ulp."""
    rng = np.random.default_rng(3)
    for T, H, W in ((1, 1, 1), (3, 7, 2), (8, 64, 16), (5, 33, 4), (2, 64, 3)):
        xs = [(rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16)
              .astype(np.uint16) for _ in range(W)]
        res = (rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        w = (rng.uniform(0.5, 1.5, H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        eps = 1e-5
        _, ro, nrm = O.forward(xs, res, w, eps)
        r64 = bx.to_f64(ro)
        rstd = 1.0 / np.sqrt((r64 * r64).mean(axis=1, keepdims=True) + float(np.float32(eps)))
        want = bx.from_f64_rne(r64 * rstd * bx.to_f64(w)[None, :])
        d = bx.ulp_diff(nrm, want)
        assert d.max() <= 1, (T, H, W, int(d.max()))


def pin_rstd_closed_form(O):
    """rstd of a row = 1/sqrt(mean(ro^2) + eps) to fp32 accuracy."""
    rng = np.random.default_rng(9)
    for H in (4, 37, 256):
        ro = (rng.normal(size=H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        w = np.full(H, bx.bits(1), np.uint16)
        _, rstd = O.rmsnorm_row(ro, w, 1e-6)
        r64 = bx.to_f64(ro)
        exact = 1.0 / np.sqrt((r64 * r64).mean() + float(np.float32(1e-6)))
        assert abs(rstd / exact - 1) < 4e-6 + 1e-7 * H, (H, rstd, exact)


def pin_scale_invariance(O):
    """With eps = 0, scaling the input by 2 or 4 scales residual_out exactly
    and leaves norm_out bit-identical (power-of-two scaling is exact through
    square, sum, division by H, sqrt and reciprocal)."""
    rng = np.random.default_rng(21)
    for H in (64, 2048):
        x = rng.normal(size=(3, H)).astype(np.float32)
        w = (rng.normal(1.0, 0.3, H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        base = None
        for s in (1.0, 2.0, 4.0):
            xb = ((x * np.float32(s)).view(np.uint32) >> 16).astype(np.uint16)
            red, ro, nrm = O.forward([xb], np.zeros((3, H), np.uint16), w, 0.0)
            if base is None:
                base = (ro, nrm)
            else:
                assert np.array_equal(bx.to_f64(ro), bx.to_f64(base[0]) * s)
                assert np.array_equal(nrm, base[1]), f"H={H} s={s}"


def pin_unit_mean_square(O):
    """weight = 1 and mean(ro^2) >> eps: mean(norm_out^2) = 1 up to rounding."""
    rng = np.random.default_rng(4)
    H = 4096
    xs = [(rng.normal(size=(4, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(4)]
    res = (rng.normal(size=(4, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w = np.full(H, bx.bits(1), np.uint16)
    _, _, nrm = O.forward(xs, res, w, 1e-6)
    ms = (bx.to_f64(nrm) ** 2).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) < 2.0 ** -7), ms


def pin_row_tiling_independent(O):
    """Rows are independent: one call over T rows equals per-block calls."""
    rng = np.random.default_rng(8)
    T, H, W = 9, 40, 3
    xs = [(rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(W)]
    res = (rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w = (rng.normal(1, .1, H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    full = O.forward(xs, res, w, 1e-6)
    for lo, hi in ((0, 1), (1, 5), (5, 9)):
        part = O.forward([x[lo:hi] for x in xs], res[lo:hi], w, 1e-6)
        for a, b in zip(full, part):
            assert np.array_equal(a[lo:hi], b)
    # and each row on its own against the step functions
    for t in range(T):
        red = O.rank_sum([x[t] for x in xs])
        ro = O.residual_add(red, res[t])
        nrm, _ = O.rmsnorm_row(ro, w, 1e-6)
        assert np.array_equal(red, full[0][t]) and np.array_equal(ro, full[1][t])
        assert np.array_equal(nrm, full[2][t])


# ------------------------------------------------------- fp32 partials (a1)
def pin_golden_cases_f32_partials(O):
    pin_golden_cases(O, GOLDEN_F32)


def pin_rank_sum_f32_integers(O):
    """Integer-valued fp32 partials (|x| <= 2^18, W <= 32: every prefix sum
    exact in fp32): the exact integer sum rounded once to bf16."""
    rng = np.random.default_rng(17)
    for W in (1, 2, 5, 16, 32):
        vals = rng.integers(-(1 << 18), (1 << 18) + 1, size=(W, 301))
        xs = [v.astype(np.float32) for v in vals]
        got = O.rank_sum(xs)
        want = [bx.round_rne(Fraction(int(t))) if t != 0 else 0 for t in vals.sum(axis=0)]
        assert list(got) == want, f"W={W}"


def pin_rank_sum_f32_brute_force(O):
    """fp32 partials of mixed magnitude against the exact rational sum: equal
    where every prefix is exact in fp32, within 1 ulp elsewhere."""
    rng = np.random.default_rng(19)
    n_exact = 0
    for W in (2, 3, 4):
        # 12 significant bits, so that many (not all) prefix sums are exact
        m = np.round(rng.normal(size=(W, 500)) * 2048) / 2048
        xs = [(mi * np.exp2(rng.integers(-10, 10, 500))).astype(np.float32) for mi in m]
        got = O.rank_sum(xs)
        for i in range(got.size):
            terms = [Fraction(float(x[i])) for x in xs]
            prefix, exact = terms[0], True
            for t in terms[1:]:
                prefix += t
                exact &= _fp32_exact(prefix)
            if prefix == 0:
                assert (int(got[i]) & 0x7FFF) == 0
                continue
            want = bx.round_rne(prefix)
            if exact:
                n_exact += 1
                assert int(got[i]) == want, (W, i, hex(int(got[i])), hex(want))
            else:
                assert bx.ulp_diff(int(got[i]), want) <= 1
    assert n_exact > 200


def pin_f32_partials_equal_bf16_path_on_bf16_values(O):
    """fp32 partials that hold bf16 values give exactly the bf16 path's
    outputs (same fp32 arithmetic on the same values)."""
    rng = np.random.default_rng(23)
    T, H, W = 5, 96, 6
    xb = [(rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(W)]
    xf = [bx.to_f64(x).astype(np.float32) for x in xb]
    res = (rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w = (rng.normal(1, .1, H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    a = O.forward(xb, res, w, 1e-6)
    b = O.forward(xf, res, w, 1e-6)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ------------------------------------------------------- E4M3 quantisation
E4M3_MAX = Fraction(448)


def e4m3_exact(q) -> int:
    """Exact rational (or float special) -> E4M3 pattern, nearest even,
    magnitudes above 448 (and infinities) saturated, from the format
    definition (1 sign, 4 exponent bits bias 7, 3 fraction bits, S.1111.111
    NaN, subnormal step 2^-9)."""
    if isinstance(q, float):
        if np.isnan(q):
            return 0x7F
        if np.isinf(q):
            return 0xFE if q < 0 else 0x7E
        if q == 0.0:
            return 0x80 if np.signbit(q) else 0x00
        q = Fraction(q)
    sign = 0x80 if q < 0 else 0
    a = abs(q)
    if a > E4M3_MAX:
        return sign | 0x7E
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -6)
    step = Fraction(2) ** (e - 3)
    n = a / step
    k = n.numerator // n.denominator
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    v = k * step
    if v > E4M3_MAX:
        v = E4M3_MAX
    if v == 0:
        return sign
    if v < Fraction(2) ** -6:
        return sign | int(v / Fraction(2) ** -9)
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    mant = (v / Fraction(2) ** e - 1) * 8
    assert mant.denominator == 1
    return sign | ((e + 7) << 3) | int(mant)


def pin_e4m3_decode_all_patterns(O):
    for b in range(256):
        got = O.e4m3_to_f32(b)
        e, m = (b >> 3) & 0xF, b & 7
        if e == 0xF and m == 7:
            assert np.isnan(got)
            continue
        want = (Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
        want = -want if b & 0x80 else want
        assert Fraction(got) == want, hex(b)
    assert O.e4m3_to_f32(0x7E) == 448.0 and O.e4m3_to_f32(0x01) == 2.0 ** -9


def pin_e4m3_rounding_vs_exact(O):
    rng = np.random.default_rng(29)
    vals = list((rng.normal(size=3000) * np.exp2(rng.integers(-14, 11, 3000))).astype(np.float32))
    # ties and neighbours at every binade, subnormal ties, saturation edges
    for e in range(-9, 9):
        for m in range(8):
            base = (1 + m / 8) * 2.0 ** e if e >= -6 else m * 2.0 ** -9
            step = 2.0 ** (max(e, -6) - 3)
            vals += [np.float32(base + step / 2), np.float32(base + step / 2) * np.float32(1 + 2 ** -20),
                     np.float32(base + step / 2) * np.float32(1 - 2 ** -20)]
    vals += [np.float32(v) for v in (448, 455.9, 464, 464.1, 1e30, -1e30, 2.0 ** -10,
                                      3 * 2.0 ** -10, 0.0, -0.0, float("inf"), float("-inf"))]
    for v in vals:
        got = O.f32_to_e4m3(float(v))
        want = e4m3_exact(float(v) if (v == 0 or not np.isfinite(v)) else Fraction(float(v)))
        assert got == want, (float(v), hex(got), hex(want))
    assert O.f32_to_e4m3(float("nan")) & 0x7F == 0x7F


def pin_e4m3_matches_torch_cast(O):
    """The library routine: torch's float8_e4m3fn cast (round to nearest
    even) agrees on finite values within range."""
    import pytest
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("this torch has no float8_e4m3fn dtype: the library cross-check did not run")
    rng = np.random.default_rng(31)
    v = np.clip((rng.normal(size=4000) * np.exp2(rng.integers(-12, 9, 4000))), -448, 448)
    v = v.astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.f32_to_e4m3(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, want)


def pin_quant_row_closed_forms(O):
    one = bx.bits(1)
    # [1, -2, 0.5, 0]: amax 2, scale 2/448, inv 224, values map to 224, -448, 112, 0
    row = np.array([bx.bits(1), bx.bits(-2), bx.bits(0.5), 0], np.uint16)
    q, sc = O.quant_e4m3(row)
    assert abs(sc[0] - np.float32(2) / np.float32(448)) == 0
    assert [O.e4m3_to_f32(int(b)) for b in q[0]] == [224.0, -448.0, 112.0, 0.0]
    # all-zero row: scale 1, q zero
    q, sc = O.quant_e4m3(np.zeros(8, np.uint16))
    assert sc[0] == 1.0 and not q.any()
    # a NaN element is ignored by amax and quantises to NaN
    row = np.array([bx.QNAN, bx.bits(4), bx.bits(-1)], np.uint16)
    q, sc = O.quant_e4m3(row)
    assert sc[0] == np.float32(4) / np.float32(448) and (q[0][0] & 0x7F) == 0x7F
    assert O.e4m3_to_f32(int(q[0][1])) == 448.0
    # the amax element always lands on +-448
    rng = np.random.default_rng(37)
    rows = (rng.normal(size=(20, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q, sc = O.quant_e4m3(rows)
    for t in range(20):
        vals = bx.to_f64(rows[t])
        i = int(np.argmax(np.abs(vals)))
        assert abs(O.e4m3_to_f32(int(q[t][i]))) == 448.0
    del one


def pin_quant_row_power_of_two_invariance(O):
    """Scaling a row by 2^k scales its scale by 2^k and leaves q unchanged."""
    rng = np.random.default_rng(41)
    x = rng.normal(size=(6, 96)).astype(np.float32)
    base = (x.view(np.uint32) >> 16).astype(np.uint16)
    q0, s0 = O.quant_e4m3(base)
    for k in (-3, 1, 5):
        xs = ((x * np.float32(2.0 ** k)).view(np.uint32) >> 16).astype(np.uint16)
        q1, s1 = O.quant_e4m3(xs)
        assert np.array_equal(q0, q1) and np.array_equal(s1, s0 * np.float32(2.0 ** k))


def pin_quant_row_vs_exact_rounding(O):
    """q = E4M3(x * inv), inv = 448 / amax rounded to fp32, the product
    rounded to fp32 first; scale = amax / 448 rounded to fp32."""
    rng = np.random.default_rng(43)
    rows = (rng.normal(size=(8, 48)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q, sc = O.quant_e4m3(rows)
    for t in range(8):
        vals = bx.to_f64(rows[t])
        amax = np.float32(np.abs(vals).max())
        scale = np.float32(amax / np.float32(448))
        inv = np.float32(np.float32(448) / amax)
        assert sc[t] == scale
        for h in range(48):
            d = np.float32(np.float32(vals[h]) * inv)
            assert int(q[t][h]) == e4m3_exact(Fraction(float(d)) if d != 0 else float(d))


# ------------------------------------------------------ NVFP4 quantisation
# E2M1 magnitudes by code (bits: exponent 2, fraction 1, bias 1), written
# out from the format definition: 0, the subnormal 0.5, then 2^(e-1)(1+m/2).
E2M1_GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
             Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def e2m1_exact(q) -> int:
    """Exact rational (or float special) -> E2M1 code by exhaustive search
    of the eight magnitudes: the nearest, a tie going to the code with an
    even fraction bit; magnitudes above 6 and infinities give 6; NaN gives
    +6 (the reading: E2M1 has no NaN)."""
    if isinstance(q, float):
        if np.isnan(q):
            return 0x7
        if np.isinf(q):
            return 0xF if q < 0 else 0x7
        if q == 0.0:
            return 0x8 if np.signbit(q) else 0x0
        q = Fraction(q)
    sign = 0x8 if q < 0 else 0
    a = abs(q)
    best = None
    for code, g in enumerate(E2M1_GRID):
        d = abs(a - g)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return sign | best[1]


def pin_e2m1_decode_all_patterns(O):
    for c in range(16):
        want = E2M1_GRID[c & 7]
        want = -want if c & 8 else want
        got = O.e2m1_to_f32(c)
        assert Fraction(got) == want and (np.signbit(got) == bool(c & 8)), hex(c)


def pin_e2m1_rounding_vs_exact(O):
    rng = np.random.default_rng(61)
    vals = list((rng.normal(size=2000) * np.exp2(rng.integers(-4, 4, 2000))).astype(np.float32))
    # every midpoint between neighbours and its two fp32 neighbours, saturation edges
    for lo, hi in zip(E2M1_GRID[:-1], E2M1_GRID[1:]):
        mid = np.float32(float((lo + hi) / 2))
        for sgn in (1, -1):
            vals += [np.float32(sgn * mid), np.float32(sgn * np.nextafter(mid, np.float32(0))),
                     np.float32(sgn * np.nextafter(mid, np.float32(10)))]
    vals += [np.float32(v) for v in (6, 6.5, 7, 8, 1e30, -1e30, 2.0 ** -126, 0.0, -0.0,
                                      float("inf"), float("-inf"), 0.2499999, 5.0000005)]
    for v in vals:
        got = O.f32_to_e2m1(float(v))
        want = e2m1_exact(float(v) if (v == 0 or not np.isfinite(v)) else Fraction(float(v)))
        assert got == want, (float(v), hex(got), hex(want))
    assert O.f32_to_e2m1(float("nan")) == 0x7


def _nvfp4_decode(O, q, s, g, H):
    """Dequantised values e2m1(q) * e4m3(s) / g in exact rationals."""
    out = []
    for h in range(H):
        byte = int(q[h // 2])
        code = (byte >> 4) if h % 2 else (byte & 0xF)
        out.append(Fraction(O.e2m1_to_f32(code)) * Fraction(O.e4m3_to_f32(int(s[h // 16])))
                   / Fraction(float(np.float32(g))))
    return out


def pin_nvfp4_block_closed_forms(O):
    B = bx.bits
    # g = 1, amax 6: the block scale is E4M3(1) and the values are their own codes
    row = np.array([B(6), B(-3), B(1.5), B(0.5), B(1), B(-0.5), B(4), B(2)] + [0] * 8, np.uint16)
    q, s = O.quant_nvfp4(row, 1.0)
    assert s[0][0] == 0x38                              # 1.0 = 2^0: exponent field 7
    assert list(q[0][:4]) == [0x7 | (0xD << 4), 0x3 | (0x1 << 4),
                              0x2 | (0x9 << 4), 0x6 | (0x4 << 4)]
    assert not q[0][4:].any()
    # amax 12 with g = 1: scale 2, every value halved before rounding
    row = np.array([B(12), B(-5), B(3), B(1)] + [0] * 12, np.uint16)
    q, s = O.quant_nvfp4(row, 1.0)
    assert O.e4m3_to_f32(int(s[0][0])) == 2.0
    assert [Fraction(v) for v in _nvfp4_decode(O, q[0], s[0], 1.0, 4)] == [12, -4, 3, 1]
    # the tensor scale g multiplies the block scale and cancels on decode
    q2, s2 = O.quant_nvfp4(row, 64.0)
    assert O.e4m3_to_f32(int(s2[0][0])) == 128.0 and np.array_equal(q, q2)
    # an all-zero block: scale 0, codes 0; a block whose scale underflows: codes 0
    tiny = np.array([B(2.0 ** -20)] * 16, np.uint16)
    q, s = O.quant_nvfp4(np.concatenate([np.zeros(16, np.uint16), tiny]), 1.0)
    assert not s.any() and not q.any()
    # NaN: ignored by the block amax, written as +6; infinity saturates
    row = np.array([bx.QNAN, B(3), B(-6), 0xFF80] + [0] * 12, np.uint16)   # 0xFF80 = -inf
    q, s = O.quant_nvfp4(row, 1.0)
    assert O.e4m3_to_f32(int(s[0][0])) == 448.0          # (inf / 6) * 1 saturates
    assert (q[0][0] & 0xF) == 0x7 and (q[0][1] >> 4) == 0xF
    # blocks are independent: a large block leaves its neighbour alone
    a = np.array([B(1)] * 16, np.uint16)
    b = np.array([B(1000)] * 16, np.uint16)
    qa, sa = O.quant_nvfp4(a, 1.0)
    qab, sab = O.quant_nvfp4(np.concatenate([a, b]), 1.0)
    assert np.array_equal(qab[0][:8], qa[0]) and sab[0][0] == sa[0][0]


def pin_nvfp4_vs_exact_rounding(O):
    """s = E4M3(fp32(fp32(amax / 6) * g)), inv = fp32(g / e4m3(s)),
    q = E2M1(fp32(v * inv)), each conversion taken exactly from rationals."""
    rng = np.random.default_rng(67)
    for trial in range(6):
        H = 16 * int(rng.integers(1, 6))
        mag = np.exp2(rng.integers(-6, 6, size=(3, H // 16))).repeat(16, axis=1)
        x = (rng.normal(size=(3, H)) * mag).astype(np.float32)
        rows = (x.view(np.uint32) >> 16).astype(np.uint16)
        g = np.float32(np.exp2(rng.uniform(-4, 8)))
        q, s = O.quant_nvfp4(rows, float(g))
        for t in range(3):
            vals = bx.to_f64(rows[t])
            for b in range(H // 16):
                blk = vals[16 * b:16 * b + 16]
                amax = np.float32(np.abs(blk).max())
                sc = e4m3_exact(Fraction(float(np.float32(np.float32(amax / np.float32(6)) * g))))
                assert int(s[t][b]) == sc, (trial, t, b)
                sv = Fraction(O.e4m3_to_f32(sc))
                for i in range(16):
                    h = 16 * b + i
                    code = (int(q[t][h // 2]) >> 4) if h % 2 else (int(q[t][h // 2]) & 0xF)
                    if sv == 0:
                        assert code == 0
                        continue
                    inv = np.float32(g / np.float32(float(sv)))
                    d = np.float32(np.float32(blk[i]) * inv)
                    want = e2m1_exact(Fraction(float(d)) if d != 0 else float(d))
                    assert code == want, (trial, t, h, hex(code), hex(want))


def pin_nvfp4_power_of_two_invariance(O):
    """Scaling a row (or g) by 2^k scales every decoded block scale by 2^k
    and leaves the codes unchanged, while the scales stay normal E4M3."""
    rng = np.random.default_rng(71)
    x = rng.normal(size=(4, 64)).astype(np.float32)
    base = (x.view(np.uint32) >> 16).astype(np.uint16)
    q0, s0 = O.quant_nvfp4(base, 16.0)
    d0 = np.array([[O.e4m3_to_f32(int(v)) for v in r] for r in s0])
    for k in (-2, 3):
        xs = ((x * np.float32(2.0 ** k)).view(np.uint32) >> 16).astype(np.uint16)
        q1, s1 = O.quant_nvfp4(xs, 16.0)
        d1 = np.array([[O.e4m3_to_f32(int(v)) for v in r] for r in s1])
        assert np.array_equal(q0, q1) and np.array_equal(d1, d0 * 2.0 ** k)
        q2, s2 = O.quant_nvfp4(base, 16.0 * 2.0 ** k)
        d2 = np.array([[O.e4m3_to_f32(int(v)) for v in r] for r in s2])
        assert np.array_equal(q0, q2) and np.array_equal(d2, d0 * 2.0 ** k)


# ---------------------------------------------------------------- MoE combine
def _f32(q: Fraction) -> Fraction:
    """Exact rational rounded to the nearest fp32 (ties to even)."""
    return Fraction(float(np.float32(float(q)))) if q != 0 else Fraction(0)


def pin_moe_combine_hand_case(O):
    """Two tokens, K = 3: gates 0.5 / 0.25 / 2, one slot skipped (-1), one
    out of range (7 >= 4 slots)."""
    one = bx.bits(1)
    ex = np.array([[bx.bits(4), bx.bits(1)], [bx.bits(8), bx.bits(-2)],
                   [bx.bits(0.5), bx.bits(3)], [bx.bits(-1), bx.bits(0)]], np.uint16)
    idx = np.array([[0, 1, -1], [2, 7, 3]], np.int32)
    g = np.array([[0.5, 0.25, 9.0], [2.0, 5.0, 1.0]], np.float32)
    res = np.zeros((2, 2), np.uint16)
    red, ro, _ = O.moe_combine(ex, idx, g, res, np.array([one, one], np.uint16), 1e-6)
    # token 0: 0.5*4 + 0.25*8 = 4, 0.5*1 + 0.25*(-2) = 0; token 1: 2*0.5 - 1 = 0, 2*3 + 0 = 6
    assert [bx.decode(int(v)) for v in red[0]] == [4, 0]
    assert [bx.decode(int(v)) for v in red[1]] == [0, 6]


def pin_moe_combine_unit_gates_is_rank_sum(O):
    """With every gate 1 and index[t,k] = the row of partial k, the combine
    is exactly the rank sum of the partials (same fp32 order and roundings,
    1 * x being exact)."""
    rng = np.random.default_rng(47)
    T, H, K = 6, 40, 5
    xs = [(rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(K)]
    res = (rng.normal(size=(T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w = (rng.normal(1, .1, H).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ex = np.concatenate(xs, axis=0)                       # slot k*T + t
    idx = np.array([[k * T + t for k in range(K)] for t in range(T)], np.int32)
    a = O.moe_combine(ex, idx, np.ones((T, K), np.float32), res, w, 1e-6)
    b = O.forward(xs, res, w, 1e-6)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def pin_moe_combine_fp32_accumulator(O):
    """The fp32 accumulator itself against exact rationals rounded to fp32
    after every product and every sum (a fused multiply-add, a reordering or
    a dropped term changes it)."""
    rng = np.random.default_rng(59)
    S, H, K = 16, 32, 7
    ex = (rng.normal(size=(S, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for trial in range(12):
        idx = rng.integers(-1, S + 1, size=K).astype(np.int32)
        g = rng.uniform(0, 1, size=K).astype(np.float32)
        for h in range(H):
            acc = Fraction(0)
            for k in range(K):
                s_ = int(idx[k])
                if 0 <= s_ < S:
                    acc = _f32(acc + _f32(Fraction(float(g[k])) * bx.decode(int(ex[s_, h]))))
            got = O.moe_combine_acc(ex, idx, g, h)
            assert Fraction(got) == acc, (trial, h, got, float(acc))


def pin_moe_combine_exact_rounding(O):
    """Against exact rationals with each product and each sum rounded to
    fp32 in k order (no fused multiply-add): bit for bit."""
    rng = np.random.default_rng(53)
    T, H, K, S = 4, 24, 6, 20
    ex = (rng.normal(size=(S, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    idx = rng.integers(-1, S + 2, size=(T, K)).astype(np.int32)
    g = rng.uniform(0, 1, size=(T, K)).astype(np.float32)
    res = np.zeros((T, H), np.uint16)
    red, _, _ = O.moe_combine(ex, idx, g, res, np.full(H, bx.bits(1), np.uint16), 1e-6)
    for t in range(T):
        for h in range(H):
            acc, any_term = Fraction(0), False
            for k in range(K):
                s_ = int(idx[t, k])
                if s_ < 0 or s_ >= S:
                    continue
                prod = _f32(Fraction(float(g[t, k])) * bx.decode(int(ex[s_, h])))
                acc = _f32(acc + prod)
                any_term = True
            got = int(red[t, h])
            if acc == 0:
                assert (got & 0x7FFF) == 0
            else:
                assert got == bx.round_rne(acc), (t, h, hex(got), hex(bx.round_rne(acc)))


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

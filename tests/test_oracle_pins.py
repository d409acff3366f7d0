"""Pins of the float64 oracle to facts outside itself.

Each check ties an oracle function to a closed form, an invariant, a
brute-force enumeration or a central finite difference, chosen so that a
plausible slip (a dropped term, a wrong sign, a wrong index, a transposed
operand) fails at least one of them.  No GPU is involved.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

from _golden import kv

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.fixture(scope="module")
def O(oracle_lib):
    return oracle_lib


# ------------------------------------------------------------ bf16 rounding

def _bf16_table():
    """All finite non-negative bfloat16 values, ascending, by enumeration."""
    vals = []
    for bits in range(0, 0x7F80):  # 0x7F80 is +inf
        vals.append((struct.unpack(">f", struct.pack(">I", bits << 16))[0], bits))
    return vals


def _brute_round(v, table):
    """Nearest bfloat16 to v by exact comparison; ties go to the even pattern."""
    if v == 0.0:
        return v
    a = abs(v)
    fa = Fraction(a)
    maxv, maxbits = table[-1]
    # Overflow: beyond max + half spacing (the tie goes to the even pattern,
    # i.e. to 2^128, which is infinity).
    half_gap = (Fraction(2) ** 128 - Fraction(maxv)) / 2
    if fa >= Fraction(maxv) + half_gap:
        return math.copysign(math.inf, v)
    lo, hi = 0, len(table) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if Fraction(table[mid][0]) <= fa:
            lo = mid
        else:
            hi = mid
    cands = [table[lo]] if lo == hi else [table[lo], table[hi]]
    best = min(cands, key=lambda c: (abs(Fraction(c[0]) - fa), c[1] & 1))
    return math.copysign(best[0], v)


def test_bf16_rounding_matches_brute_force(O):
    table = _bf16_table()
    rng = np.random.default_rng(7)
    vals = []
    # random magnitudes across the whole bfloat16 range, incl. subnormals
    for e in range(-140, 129, 3):
        vals += list(rng.uniform(0.5, 1.0, 4) * 2.0 ** e)
    # exact midpoints and their neighbours, in several binades
    for bits in list(range(0x3F80, 0x3F90)) + [0x0001, 0x0002, 0x0080, 0x7F7E, 0x7F7F, 0x0C35]:
        lo = struct.unpack(">f", struct.pack(">I", bits << 16))[0]
        hi = struct.unpack(">f", struct.pack(">I", (bits + 1) << 16))[0]
        if math.isinf(hi):
            hi = 2.0 ** 128  # the spacing continues past the largest finite value
        midv = (lo + hi) / 2  # exact in float64
        vals += [midv, math.nextafter(midv, 0), math.nextafter(midv, math.inf)]
        # a value that float32 would round onto the midpoint first (double rounding)
        vals.append(midv + (hi - lo) * 2.0 ** -20)
    vals += [2.0 ** -134, 2.0 ** -135, 3 * 2.0 ** -135, 1e-300, 3.5e38, 3.4e38, 1e39]
    vals += [-v for v in vals[::5]]
    for v in vals:
        want = _brute_round(v, table)
        got = O.round_bf16(v)
        assert got == want or (math.isinf(want) and math.isinf(got) and (got > 0) == (want > 0)), \
            (v, got, want)
    assert math.isnan(O.round_bf16(math.nan))


# ------------------------------------------------------- binary16 rounding

def _f16_table():
    """All finite non-negative IEEE binary16 values, ascending, by enumeration
    of the bit patterns (decoded from the format's definition, not a library)."""
    vals = []
    for bits in range(0, 0x7C00):  # 0x7C00 is +inf
        e, f = bits >> 10, bits & 0x3FF
        v = math.ldexp(f, -24) if e == 0 else math.ldexp(f | 0x400, e - 25)
        vals.append((v, bits))
    return vals


def _brute_round_f16(v, table):
    if v == 0.0:
        return v
    fa = Fraction(abs(v))
    maxv = table[-1][0]
    if fa >= Fraction(maxv) + (Fraction(2) ** 16 - Fraction(maxv)) / 2:
        return math.copysign(math.inf, v)
    lo, hi = 0, len(table) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if Fraction(table[mid][0]) <= fa:
            lo = mid
        else:
            hi = mid
    best = min([table[lo], table[hi]], key=lambda c: (abs(Fraction(c[0]) - fa), c[1] & 1))
    return math.copysign(best[0], v)


def test_f16_rounding_matches_brute_force(O):
    table = _f16_table()
    assert table[-1][0] == 65504.0 and table[1][0] == 2.0 ** -24
    rng = np.random.default_rng(11)
    vals = []
    for e in range(-27, 17):
        vals += list(rng.uniform(0.5, 1.0, 6) * 2.0 ** e)
    # exact midpoints and neighbours: normal, subnormal, binade edges, overflow
    for bits in list(range(0x3C00, 0x3C10)) + [0x0000, 0x0001, 0x0002, 0x03FF, 0x0400, 0x7BFE]:
        lo = table[bits][0]
        hi = table[bits + 1][0]
        midv = (lo + hi) / 2
        vals += [midv, math.nextafter(midv, 0), math.nextafter(midv, math.inf)]
    vals += [65504.0, 65519.99, 65520.0, 65536.0, 1e-9, 2.0 ** -25, 3 * 2.0 ** -26, 1e300]
    vals += [-v for v in vals[::4]]
    for v in vals:
        want = _brute_round_f16(v, table)
        got = O.round_f16(v)
        assert got == want or (math.isinf(want) and math.isinf(got) and (got > 0) == (want > 0)), \
            (v, got, want)
    assert math.isnan(O.round_f16(math.nan))


def test_f16_rounding_matches_numpy(O):
    """Against a library routine: numpy's float64 -> float16 conversion."""
    rng = np.random.default_rng(12)
    v = rng.standard_normal(200000) * np.exp(rng.uniform(-20, 11.5, 200000))
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(O.round_f16_array(v), want)


def test_f16_inputs_widen_exactly(O):
    """A binary16 activation array gives the same results as the float64
    array of the same values (decoding is exact)."""
    rng = np.random.default_rng(13)
    xh = (rng.standard_normal((5, 12)) * 3).astype(np.float16)
    xh[0, 0] = np.float16(2.0 ** -24)  # a subnormal
    dyh = rng.standard_normal((5, 12)).astype(np.float16)
    x64, dy64 = xh.astype(np.float64), dyh.astype(np.float64)
    g, b = rng.standard_normal(12), rng.standard_normal(12)
    for fn in (lambda x: O.ln_fwd(x, 1e-5, g, b)[0], lambda x: O.dyt_fwd(x, 0.7, g, b)[0],
               lambda x: O.rms_fwd(x, 1e-6, g, O.MATH)[0]):
        np.testing.assert_array_equal(fn(xh), fn(x64))
    ch = O.ln_bwd_cols(xh, dyh, *O.ln_fwd(xh, 1e-5, g, b)[2:4])
    c64 = O.ln_bwd_cols(x64, dy64, *O.ln_fwd(x64, 1e-5, g, b)[2:4])
    for k in ch:
        np.testing.assert_array_equal(ch[k], c64[k])


def test_bf16_array_matches_scalar(O):
    v = np.random.default_rng(3).standard_normal(1000) * 10
    a = O.round_bf16_array(v)
    assert all(a[i] == O.round_bf16(v[i]) for i in range(v.size))


def test_near_tie_flag(O):
    mid = 1.0 + 2.0 ** -8  # midpoint between 1 and 1 + 2^-7
    assert O.bf16_near_tie(mid)
    assert O.bf16_near_tie(mid * (1 + 2.0 ** -20))
    assert not O.bf16_near_tie(1.0)
    assert not O.bf16_near_tie(1.0 + 2.0 ** -9)


# ------------------------------------------------------------------- DyT

def _L_dyt(O, x, dy, alpha, g, b):
    y, _ = O.dyt_fwd(x, alpha, g, b)
    return float(np.sum(dy * y))


def test_dyt_fwd_closed_form_tanh_of_log(O):
    # tanh(ln a) = (a^2 - 1) / (a^2 + 1)
    a = np.array([1.5, 2.0, 3.0, 7.0, 1.0 / 3.0])
    x = np.log(a)[None, :]
    y, _ = O.dyt_fwd(x, 1.0, np.ones(5), np.zeros(5))
    np.testing.assert_allclose(y[0], (a * a - 1) / (a * a + 1), rtol=4e-16, atol=0)
    # alpha and x enter only through their product; gamma scales, beta shifts
    y2, _ = O.dyt_fwd(x / 4.0, 4.0, 3.0 * np.ones(5), 0.5 * np.ones(5))
    np.testing.assert_allclose(y2[0], 3.0 * (a * a - 1) / (a * a + 1) + 0.5, rtol=4e-16)


def test_dyt_fwd_limits(O):
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 6))
    g = rng.standard_normal(6); b = rng.standard_normal(6)
    # alpha -> +inf: gamma * sign(x) + beta
    y, _ = O.dyt_fwd(x, math.inf, g, b)
    np.testing.assert_array_equal(y, g * np.sign(x) + b)
    # alpha -> 0: beta + gamma alpha x to first order
    al = 1e-7
    y, _ = O.dyt_fwd(x, al, g, b)
    np.testing.assert_allclose(y, b + g * al * x, rtol=0, atol=1e-19 + 1e-15 * np.abs(b).max())
    # tanh is odd
    y1, _ = O.dyt_fwd(x, 0.7, np.ones(6), np.zeros(6))
    y2, _ = O.dyt_fwd(-x, 0.7, np.ones(6), np.zeros(6))
    np.testing.assert_array_equal(y1, -y2)


def test_dyt_bwd_finite_differences(O):
    rng = np.random.default_rng(1)
    M, N = 4, 7
    x = rng.standard_normal((M, N)); dy = rng.standard_normal((M, N))
    g = 1 + 0.3 * rng.standard_normal(N); b = rng.standard_normal(N)
    al = 0.8
    dx = O.dyt_bwd_rows(x, dy, al, g)
    c = O.dyt_bwd_cols(x, dy, al, g)

    def fd(f, v):
        h = 1e-6 * max(1.0, abs(v))
        return (f(v + h) - f(v - h)) / (2 * h)

    for i in range(M):
        for j in range(N):
            def f(v, i=i, j=j):
                xx = x.copy(); xx[i, j] = v
                return _L_dyt(O, xx, dy, al, g, b)
            assert abs(fd(f, x[i, j]) - dx[i, j]) <= 1e-7 * max(1, abs(dx[i, j]))
    for j in range(N):
        def fg(v, j=j):
            gg = g.copy(); gg[j] = v
            return _L_dyt(O, x, dy, al, gg, b)

        def fb(v, j=j):
            bb = b.copy(); bb[j] = v
            return _L_dyt(O, x, dy, al, g, bb)
        assert abs(fd(fg, g[j]) - c["dgamma"][j]) <= 1e-7 * max(1, abs(c["dgamma"][j]))
        assert abs(fd(fb, b[j]) - c["dbeta"][j]) <= 1e-7 * max(1, abs(c["dbeta"][j]))
    fa = fd(lambda v: _L_dyt(O, x, dy, v, g, b), al)
    assert abs(fa - c["dalpha"]) <= 1e-7 * max(1, abs(c["dalpha"]))


def test_dyt_dbeta_is_column_sum_and_sumsq(O):
    rng = np.random.default_rng(2)
    # values on a 1/8 grid: every float64 sum is exact in any order
    dy = rng.integers(-64, 64, (50, 9)) / 8.0
    x = rng.standard_normal((50, 9))
    c = O.dyt_bwd_cols(x, dy, 0.5, np.ones(9))
    np.testing.assert_array_equal(c["dbeta"], dy.sum(axis=0))
    np.testing.assert_array_equal(c["dbeta_ss"], (dy * dy).sum(axis=0))


def test_dyt_sech2_identity(O):
    rng = np.random.default_rng(4)
    x = rng.uniform(-2, 2, (3, 5)); dy = np.ones((3, 5))
    dx = O.dyt_bwd_rows(x, dy, 1.3, np.ones(5))
    t = np.tanh(1.3 * x)
    np.testing.assert_allclose(dx, 1.3 * (1 - t * t), rtol=1e-13)


def test_dyt_alpha_inf_and_padding_rows(O):
    rng = np.random.default_rng(5)
    M, N = 6, 8
    x = rng.standard_normal((M, N)); dy = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    c = O.dyt_bwd_cols(x, dy, math.inf, g)
    assert np.all(np.isfinite(c["dgamma"])) and np.all(np.isfinite(c["dbeta"]))
    assert c["dalpha"] == 0.0
    np.testing.assert_allclose(c["dgamma"], (dy * np.sign(x)).sum(axis=0), rtol=1e-15)
    dx = O.dyt_bwd_rows(x, dy, math.inf, g)
    assert np.all(np.isnan(dx))  # dy * gamma * inf * 0 under IEEE rules
    # rows with dy = 0 appended: no parameter gradient changes
    xp = np.vstack([x, rng.standard_normal((3, N))]); dyp = np.vstack([dy, np.zeros((3, N))])
    for al in (0.6, math.inf):
        c0 = O.dyt_bwd_cols(x, dy, al, g)
        c1 = O.dyt_bwd_cols(xp, dyp, al, g)
        for k in ("dgamma", "dbeta"):
            np.testing.assert_array_equal(c0[k], c1[k])
        assert c0["dalpha"] == c1["dalpha"]


def test_dyt_rows_subset_and_dtypes(O):
    rng = np.random.default_rng(6)
    x32 = rng.standard_normal((5, 4)).astype(np.float32)
    g = rng.standard_normal(4); b = rng.standard_normal(4)
    full, _ = O.dyt_fwd(x32, 0.9, g, b)
    sub, _ = O.dyt_fwd(x32, 0.9, g, b, rows=[3, 1])
    np.testing.assert_array_equal(sub, full[[3, 1]])
    # bf16 bit patterns widen exactly: compare against the float32 path
    bf = (x32.view(np.uint32) >> 16).astype(np.uint16)
    as32 = (bf.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(O.dyt_fwd(bf, 0.9, g, b)[0], O.dyt_fwd(as32, 0.9, g, b)[0])


# -------------------------------------------------------------- LayerNorm

def test_ln_fwd_invariants(O):
    rng = np.random.default_rng(10)
    M, N = 5, 33
    x = 3 + 2 * rng.standard_normal((M, N))
    eps = 1e-3
    y, _, mu, rs = O.ln_fwd(x, eps)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-14)
    var = ((x - x.mean(axis=1, keepdims=True)) ** 2).mean(axis=1)
    np.testing.assert_allclose((y * y).mean(axis=1), var / (var + eps), rtol=1e-13)
    # shift invariance, and scale invariance at eps = 0
    y2, *_ = O.ln_fwd(x + 17.0, eps)
    np.testing.assert_allclose(y2, y, atol=1e-12)
    ya, *_ = O.ln_fwd(x, 0.0)
    yb, *_ = O.ln_fwd(2.5 * x, 0.0)
    np.testing.assert_allclose(ya, yb, atol=1e-13)
    # affine applied per column
    g = rng.standard_normal(N); b = rng.standard_normal(N)
    y3, *_ = O.ln_fwd(x, eps, g, b)
    np.testing.assert_allclose(y3, y * g + b, atol=1e-13)


def test_ln_fwd_degenerate(O):
    b = np.array([0.25])
    y, _, mu, rs = O.ln_fwd(np.array([[3.0], [-2.0]]), 1e-5, np.array([2.0]), b)
    np.testing.assert_array_equal(y, [[0.25], [0.25]])  # width one: y = beta
    y, *_ = O.ln_fwd(np.full((1, 6), 4.0), 1e-5, np.ones(6), np.arange(6.0))
    np.testing.assert_array_equal(y[0], np.arange(6.0))  # constant row: y = beta


def _L_ln(O, x, dy, eps, g, b):
    y, *_ = O.ln_fwd(x, eps, g, b)
    return float(np.sum(dy * y))


def test_ln_bwd_invariants_and_closed_form(O):
    rng = np.random.default_rng(11)
    M, N = 4, 19
    x = rng.standard_normal((M, N)); dy = rng.standard_normal((M, N))
    g = 1 + 0.2 * rng.standard_normal(N); eps = 0.05
    _, _, mu, rs = O.ln_fwd(x, eps, g)
    dx, _ = O.ln_bwd_rows(x, dy, mu, rs, g)
    np.testing.assert_allclose(dx.sum(axis=1), 0, atol=1e-13)
    xh = (x - mu[:, None]) * rs[:, None]
    gg = dy * g
    m = (gg * xh).mean(axis=1)
    var = ((x - mu[:, None]) ** 2).mean(axis=1)
    want = rs * N * m * eps / (var + eps)
    np.testing.assert_allclose((dx * xh).sum(axis=1), want, rtol=1e-11, atol=1e-13)
    # width one: dx = 0
    x1 = rng.standard_normal((3, 1)); _, _, m1, r1 = O.ln_fwd(x1, eps)
    d1, _ = O.ln_bwd_rows(x1, rng.standard_normal((3, 1)), m1, r1)
    np.testing.assert_array_equal(d1, 0.0)


def test_ln_bwd_finite_differences(O):
    rng = np.random.default_rng(12)
    M, N = 3, 6
    x = rng.standard_normal((M, N)); dy = rng.standard_normal((M, N))
    g = 1 + 0.3 * rng.standard_normal(N); b = rng.standard_normal(N); eps = 0.1
    _, _, mu, rs = O.ln_fwd(x, eps, g, b)
    dx, _ = O.ln_bwd_rows(x, dy, mu, rs, g)
    c = O.ln_bwd_cols(x, dy, mu, rs)

    def fd(f, v):
        h = 1e-6 * max(1.0, abs(v))
        return (f(v + h) - f(v - h)) / (2 * h)

    for i in range(M):
        for j in range(N):
            def f(v, i=i, j=j):
                xx = x.copy(); xx[i, j] = v
                return _L_ln(O, xx, dy, eps, g, b)
            assert abs(fd(f, x[i, j]) - dx[i, j]) <= 1e-7 * max(1, abs(dx[i, j]))
    for j in range(N):
        def fg(v, j=j):
            gg = g.copy(); gg[j] = v
            return _L_ln(O, x, dy, eps, gg, b)

        def fb(v, j=j):
            bb = b.copy(); bb[j] = v
            return _L_ln(O, x, dy, eps, g, bb)
        assert abs(fd(fg, g[j]) - c["dgamma"][j]) <= 1e-7 * max(1, abs(c["dgamma"][j]))
        assert abs(fd(fb, b[j]) - c["dbeta"][j]) <= 1e-7 * max(1, abs(c["dbeta"][j]))


def test_ln_dbeta_and_padding(O):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((20, 5)); dy = rng.integers(-40, 40, (20, 5)) / 4.0
    _, _, mu, rs = O.ln_fwd(x, 1e-5)
    c = O.ln_bwd_cols(x, dy, mu, rs)
    np.testing.assert_array_equal(c["dbeta"], dy.sum(axis=0))
    xp = np.vstack([x, rng.standard_normal((2, 5))]); dyp = np.vstack([dy, np.zeros((2, 5))])
    _, _, mup, rsp = O.ln_fwd(xp, 1e-5)
    cp = O.ln_bwd_cols(xp, dyp, mup, rsp)
    np.testing.assert_array_equal(c["dgamma"], cp["dgamma"])
    np.testing.assert_array_equal(c["dbeta"], cp["dbeta"])


# ---------------------------------------------------------------- RMSNorm

def test_rms_fwd_invariants(O):
    rng = np.random.default_rng(20)
    x = rng.standard_normal((4, 23)); w = 1 + 0.1 * rng.standard_normal(23)
    ya, *_ = O.rms_fwd(x, 0.0, w, O.MATH)
    yb, *_ = O.rms_fwd(3.7 * x, 0.0, w, O.MATH)
    np.testing.assert_allclose(ya, yb, rtol=1e-14)
    eps = 0.3
    y, _, rs, _ = O.rms_fwd(x, eps, np.ones(23), O.MATH)
    ms = (x * x).mean(axis=1)
    np.testing.assert_allclose((y * y).mean(axis=1), ms / (ms + eps), rtol=1e-13)
    np.testing.assert_allclose(rs, 1 / np.sqrt(ms + eps), rtol=1e-15)
    yw, *_ = O.rms_fwd(x, eps, w, O.MATH)
    np.testing.assert_allclose(yw, y * w, rtol=1e-15)


def test_rms_width_one(O):
    eps = kv("rmsnorm_width_one.txt")["eps"]
    x = np.array([[-2.0], [-0.3], [0.1], [0.5], [1.7]])
    w = np.array([1.25])
    y, *_ = O.rms_fwd(x, eps, w, O.MATH)
    np.testing.assert_allclose(y[:, 0], w[0] * x[:, 0] / np.sqrt(x[:, 0] ** 2 + eps), rtol=1e-15)
    dy = np.array([[0.7], [-1.1], [2.0], [1.0], [-0.4]])
    dx, *_ = O.rms_bwd_rows(x, dy, eps, w, O.F32, O.MATH)
    dn = dy[:, 0] * w[0]
    want = dn * eps / (x[:, 0] ** 2 + eps) ** 1.5  # the page's closed form
    np.testing.assert_allclose(dx[:, 0], want, rtol=1e-14)


def test_rms_bwd_closed_form_and_fd(O):
    rng = np.random.default_rng(21)
    M, N = 3, 7
    x = rng.standard_normal((M, N)); dy = rng.standard_normal((M, N))
    w = 1 + 0.2 * rng.standard_normal(N); eps = 0.2
    dx, *_ = O.rms_bwd_rows(x, dy, eps, w, O.F32, O.MATH)
    ms = (x * x).mean(axis=1); r = 1 / np.sqrt(ms + eps)
    dn = dy * w
    lhs = (dx * x).sum(axis=1)
    rhs = eps * r * r * (dn * x * r[:, None]).sum(axis=1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-14)
    dw, *_ = O.rms_bwd_cols(x, dy, eps, O.F32, O.MATH)

    def L(xx, ww):
        y, *_ = O.rms_fwd(xx, eps, ww, O.MATH)
        return float(np.sum(dy * y))

    def fd(f, v):
        h = 1e-6 * max(1.0, abs(v))
        return (f(v + h) - f(v - h)) / (2 * h)

    for i in range(M):
        for j in range(N):
            def f(v, i=i, j=j):
                xx = x.copy(); xx[i, j] = v
                return L(xx, w)
            assert abs(fd(f, x[i, j]) - dx[i, j]) <= 1e-7 * max(1, abs(dx[i, j]))
    for j in range(N):
        def fw(v, j=j):
            ww = w.copy(); ww[j] = v
            return L(x, ww)
        assert abs(fd(fw, w[j]) - dw[j]) <= 1e-7 * max(1, abs(dw[j]))


def test_rms_parity_rounding_points(O):
    rng = np.random.default_rng(22)
    x32 = rng.standard_normal((6, 16)).astype(np.float32)
    bf = (x32.view(np.uint32) >> 16).astype(np.uint16)
    xw = (bf.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    eps = 1e-6
    # parity mode with unit weight: y is the normalized value rounded to bf16
    y, _, rs, amb = O.rms_fwd(bf, eps, np.ones(16), O.PARITY)
    ym, *_ = O.rms_fwd(bf, eps, np.ones(16), O.MATH)
    np.testing.assert_array_equal(y, O.round_bf16_array(ym))
    assert not np.array_equal(y, ym)
    # float64 activations: parity mode has no rounding points
    y64, *_ = O.rms_fwd(xw, eps, np.ones(16), O.PARITY)
    np.testing.assert_array_equal(y64, ym)
    # dw: with a bf16 weight each term dy*n is rounded; with unit dy the term
    # is n itself, already a bf16 value, so both weight dtypes agree
    ones = np.full_like(bf, 0x3F80)  # bf16 1.0
    d_b, *_ = O.rms_bwd_cols(bf, ones, eps, O.BF16, O.PARITY)
    d_f, *_ = O.rms_bwd_cols(bf, ones, eps, O.F32, O.PARITY)
    np.testing.assert_array_equal(d_b, d_f)
    np.testing.assert_allclose(d_b, y.sum(axis=0), rtol=1e-15)
    # a dy with a 3-bit significand times n (8 bits) needs 11 bits: the bf16
    # weight path rounds each term, the float32 weight path does not
    three = np.full_like(bf, 0x3FE0)  # bf16 1.75
    t_b, *_ = O.rms_bwd_cols(bf, three, eps, O.BF16, O.PARITY)
    t_f, *_ = O.rms_bwd_cols(bf, three, eps, O.F32, O.PARITY)
    np.testing.assert_allclose(t_f, 1.75 * y.sum(axis=0), rtol=1e-15)
    np.testing.assert_allclose(t_b, O.round_bf16_array(1.75 * y).sum(axis=0), rtol=1e-15)
    assert not np.array_equal(t_b, t_f)


def test_rms_parity_rounding_points_f16(O):
    """The same rounding points with binary16 activations: n rounds to
    binary16, and a binary16 weight rounds each dw term."""
    rng = np.random.default_rng(24)
    xh = rng.standard_normal((6, 16)).astype(np.float16)
    eps = 1e-6
    y, *_ = O.rms_fwd(xh, eps, np.ones(16), O.PARITY)
    ym, *_ = O.rms_fwd(xh, eps, np.ones(16), O.MATH)
    np.testing.assert_array_equal(y, O.round_f16_array(ym))
    assert not np.array_equal(y, ym)
    # dy = 1.75 has a 3-bit significand; n has 11: each product needs 13 bits
    three = np.full((6, 16), 1.75, dtype=np.float16)
    t_h, *_ = O.rms_bwd_cols(xh, three, eps, O.F16, O.PARITY)
    t_f, *_ = O.rms_bwd_cols(xh, three, eps, O.F32, O.PARITY)
    np.testing.assert_allclose(t_f, 1.75 * y.sum(axis=0), rtol=1e-15)
    np.testing.assert_allclose(t_h, O.round_f16_array(1.75 * y).sum(axis=0), rtol=1e-15)
    assert not np.array_equal(t_h, t_f)
    # dn = round(dy w) in binary16
    w = rng.standard_normal(16)
    dyh = rng.standard_normal((6, 16)).astype(np.float16)
    dx, *_ = O.rms_bwd_rows(xh, dyh, eps, w, O.F32, O.PARITY)
    dxm, *_ = O.rms_bwd_rows(xh, dyh, eps, w, O.F32, O.MATH)
    assert not np.array_equal(dx, dxm)
    np.testing.assert_allclose(dx, dxm, rtol=0, atol=2.0 ** -8 * np.abs(dxm).max())


def _as16(vals, act):
    """float64 values that are bfloat16 (or binary16) values -> the stored
    16-bit array the oracle takes (raw bf16 patterns, or float16)."""
    v = np.asarray(vals, dtype=np.float64)
    if act == "bf16":
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return v.astype(np.float16)


def _round16(O, vals, act):
    return O.round_bf16_array(vals) if act == "bf16" else O.round_f16_array(vals)


@pytest.mark.parametrize("act", ["bf16", "f16"])
@pytest.mark.parametrize("wkind", ["f32", "act"])
def test_rms_parity_dn_is_the_only_backward_rounding(O, act, wkind):
    """Where the parity backward rounds (DS 8645 "Semantics"): dn = round_x(dy*w)
    and nothing else before dx.  Pinned by two structural facts:
    (a) with w = 1, dy*w = dy is already a 16-bit value, so parity dx must be
        math dx bit for bit; a rounding misplaced onto xhat or onto dn*xhat
        would change it;
    (b) with w = 1.75 (3 significant bits, so dy*w needs up to 11 or 14 and
        is rounded), parity dx on (dy, w) must be math dx on
        (dy' = round_x(1.75 dy), w = 1) bit for bit, while math dx on
        (dy, 1.75) differs: skipping the rounding fails (b), and rounding
        anything but the product fails (a) or (b).
    The weight's dtype code (f32 or the activation's) must not move it."""
    rng = np.random.default_rng(40 if act == "bf16" else 41)
    M, N = 8, 32
    xs = _as16(_round16(O, rng.standard_normal((M, N)), act), act)
    dys = _as16(_round16(O, rng.standard_normal((M, N)), act), act)
    dyv = (dys.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if act == "bf16" \
        else dys.astype(np.float64)
    wcode = O.F32 if wkind == "f32" else (O.BF16 if act == "bf16" else O.F16)
    eps = 1e-6
    one = np.ones(N)
    # (a) an exact product: nothing to round before dx
    dp, *_ = O.rms_bwd_rows(xs, dys, eps, one, wcode, O.PARITY)
    dm, *_ = O.rms_bwd_rows(xs, dys, eps, one, wcode, O.MATH)
    np.testing.assert_array_equal(dp, dm)
    # (b) the product rounded where the page rounds it
    w = np.full(N, 1.75)
    dyr = _as16(_round16(O, 1.75 * dyv, act), act)
    assert not np.array_equal(_round16(O, 1.75 * dyv, act), 1.75 * dyv)  # roundings happen
    dp, *_ = O.rms_bwd_rows(xs, dys, eps, w, wcode, O.PARITY)
    want, *_ = O.rms_bwd_rows(xs, dyr, eps, one, wcode, O.MATH)
    np.testing.assert_array_equal(dp, want)
    skipped, *_ = O.rms_bwd_rows(xs, dys, eps, w, wcode, O.MATH)
    assert not np.array_equal(dp, skipped)


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_rms_parity_forward_rounds_n_before_the_weight(O, act):
    """The parity forward rounds n = x r, then multiplies by w (DS 8645
    "Semantics"): y(w) = w * y(1) exactly for w = 1.75 (a 3-bit value times
    a 16-bit n is exact in float64), which a rounding of w * xhat, or none,
    would not give."""
    rng = np.random.default_rng(42 if act == "bf16" else 43)
    xs = _as16(_round16(O, rng.standard_normal((6, 24)), act), act)
    y1, *_ = O.rms_fwd(xs, 1e-6, np.ones(24), O.PARITY)
    yw, *_ = O.rms_fwd(xs, 1e-6, np.full(24, 1.75), O.PARITY)
    np.testing.assert_array_equal(yw, 1.75 * y1)
    ym, *_ = O.rms_fwd(xs, 1e-6, np.full(24, 1.75), O.MATH)
    assert not np.array_equal(yw, ym)
    assert not np.array_equal(yw, _round16(O, ym, act))


def test_rms_variants_math_and_fd(O):
    """In math mode the weight-first expression is the Llama one (only the
    rounding points differ), and Gemma's is the Llama one with w -> 1 + w;
    Gemma's gradients also match central finite differences."""
    rng = np.random.default_rng(25)
    M, N = 3, 7
    x = rng.standard_normal((M, N)); dy = rng.standard_normal((M, N))
    w = 0.2 * rng.standard_normal(N); eps = 0.2
    V0, V1, V2 = O.RMS_CAST_FIRST, O.RMS_WEIGHT_FIRST, O.RMS_GEMMA
    y0, *_ = O.rms_fwd(x, eps, w, O.MATH, variant=V0)
    y1, *_ = O.rms_fwd(x, eps, w, O.MATH, variant=V1)
    y2, *_ = O.rms_fwd(x, eps, w, O.MATH, variant=V2)
    y0p, *_ = O.rms_fwd(x, eps, 1 + w, O.MATH, variant=V0)
    np.testing.assert_array_equal(y1, y0)
    np.testing.assert_array_equal(y2, y0p)
    dx2, *_ = O.rms_bwd_rows(x, dy, eps, w, O.F32, O.MATH, variant=V2)
    dx0p, *_ = O.rms_bwd_rows(x, dy, eps, 1 + w, O.F32, O.MATH, variant=V0)
    np.testing.assert_array_equal(dx2, dx0p)
    dw2, *_ = O.rms_bwd_cols(x, dy, eps, O.F32, O.MATH, variant=V2)
    dw0, *_ = O.rms_bwd_cols(x, dy, eps, O.F32, O.MATH, variant=V0)
    np.testing.assert_array_equal(dw2, dw0)  # d(1 + w)/dw = 1

    def L(xx, ww):
        y, *_ = O.rms_fwd(xx, eps, ww, O.MATH, variant=V2)
        return float(np.sum(dy * y))

    def fd(f, v):
        h = 1e-6 * max(1.0, abs(v))
        return (f(v + h) - f(v - h)) / (2 * h)

    for i in range(M):
        for j in range(N):
            def f(v, i=i, j=j):
                xx = x.copy(); xx[i, j] = v
                return L(xx, w)
            assert abs(fd(f, x[i, j]) - dx2[i, j]) <= 1e-7 * max(1, abs(dx2[i, j]))
    for j in range(N):
        def fw(v, j=j):
            ww = w.copy(); ww[j] = v
            return L(x, ww)
        assert abs(fd(fw, w[j]) - dw2[j]) <= 1e-7 * max(1, abs(dw2[j]))


def test_rms_variants_rounding_points(O):
    """Weight-first and Gemma round only at the outputs, except Gemma's
    float32 1 + w."""
    rng = np.random.default_rng(26)
    x32 = rng.standard_normal((5, 16)).astype(np.float32)
    bf = (x32.view(np.uint32) >> 16).astype(np.uint16)
    dyb = (rng.standard_normal((5, 16)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    eps = 1e-6
    w = 1 + 0.1 * rng.standard_normal(16)
    for v in (O.RMS_WEIGHT_FIRST, O.RMS_GEMMA):
        wv = w - 1 if v == O.RMS_GEMMA else w
        wv = wv.astype(np.float32).astype(np.float64)
        yp, *_ = O.rms_fwd(bf, eps, wv, O.PARITY, variant=v)
        ym, *_ = O.rms_fwd(bf, eps, wv, O.MATH, variant=v)
        # no rounding of the normalized value: parity differs from math only
        # through Gemma's float32 1 + w
        if v == O.RMS_WEIGHT_FIRST:
            np.testing.assert_array_equal(yp, ym)
        dxp, *_ = O.rms_bwd_rows(bf, dyb, eps, wv, O.BF16, O.PARITY, variant=v)
        dxm, *_ = O.rms_bwd_rows(bf, dyb, eps, wv, O.BF16, O.MATH, variant=v)
        dwp, *_ = O.rms_bwd_cols(bf, dyb, eps, O.BF16, O.PARITY, variant=v)
        dwm, *_ = O.rms_bwd_cols(bf, dyb, eps, O.BF16, O.MATH, variant=v)
        np.testing.assert_array_equal(dwp, dwm)  # no per-term rounding
        if v == O.RMS_WEIGHT_FIRST:
            np.testing.assert_array_equal(dxp, dxm)
    # Gemma: 1 + w in float32 swallows a weight below float32's resolution
    tiny = np.full(16, 2.0 ** -30)
    yg, *_ = O.rms_fwd(bf, eps, tiny, O.PARITY, variant=O.RMS_GEMMA)
    yg1, *_ = O.rms_fwd(bf, eps, np.zeros(16), O.PARITY, variant=O.RMS_GEMMA)
    ygm, *_ = O.rms_fwd(bf, eps, tiny, O.MATH, variant=O.RMS_GEMMA)
    np.testing.assert_array_equal(yg, yg1)
    assert not np.array_equal(yg, ygm)


def test_rms_padding_rows(O):
    rng = np.random.default_rng(23)
    x = rng.standard_normal((9, 6)); dy = rng.standard_normal((9, 6))
    xp = np.vstack([x, rng.standard_normal((4, 6))]); dyp = np.vstack([dy, np.zeros((4, 6))])
    a, *_ = O.rms_bwd_cols(x, dy, 1e-6, O.F32, O.MATH)
    b, *_ = O.rms_bwd_cols(xp, dyp, 1e-6, O.F32, O.MATH)
    np.testing.assert_array_equal(a, b)


def test_rms_near_tie_allowance(O):
    # The allowance is nonzero exactly where the normalized value sits within
    # 2^-17 (relative) of a bfloat16 midpoint, and equals |w| times the
    # bfloat16 spacing there.
    rng = np.random.default_rng(24)
    x32 = rng.standard_normal((400, 64)).astype(np.float32)
    bf = (x32.view(np.uint32) >> 16).astype(np.uint16)
    xv = (bf.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = 1 + 0.1 * rng.standard_normal(64)
    _, _, rs, allow = O.rms_fwd(bf, 1e-6, w, O.PARITY)
    v = xv * rs[:, None]
    tie = np.vectorize(O.bf16_near_tie)(v)
    assert tie.sum() > 0
    np.testing.assert_array_equal(allow > 0, tie)
    a = np.abs(v[tie])
    spacing = 2.0 ** (np.floor(np.log2(a)) - 7)
    np.testing.assert_allclose(allow[tie], np.abs(np.broadcast_to(w, v.shape)[tie]) * spacing, rtol=0)
    # a bfloat16 weight makes dy*w exact in float32: no dn allowance
    dy = bf[::-1].copy()
    _, _, al_b = O.rms_bwd_rows(bf, dy, 1e-6, w, O.BF16, O.PARITY)
    assert np.all(al_b == 0)
    _, _, al_f = O.rms_bwd_rows(bf, dy, 1e-6, w, O.F32, O.PARITY)
    assert np.any(al_f > 0)


# ------------------------------------------- linearity and equivariance
# Facts of every layer's backward as a function of its inputs: the gradients
# are linear in dy; permuting rows permutes the row outputs and leaves the
# column sums unchanged; permuting columns (with the per-column parameters)
# permutes every per-column output.  A wrong row or column index, a parameter
# applied to the wrong column, or dy entering non-linearly fails one of them.

def _backwards(O, x, dy, g, b, eps):
    """Every backward output of the three layers (math mode, float64)."""
    out = {}
    out["dyt dx"] = O.dyt_bwd_rows(x, dy, 0.9, g)
    c = O.dyt_bwd_cols(x, dy, 0.9, g)
    out["dyt dgamma"], out["dyt dbeta"] = c["dgamma"], c["dbeta"]
    out["dyt dalpha"] = np.array([c["dalpha"]])
    _, _, mu, rs = O.ln_fwd(x, eps, g, b)
    out["ln dx"] = O.ln_bwd_rows(x, dy, mu, rs, g)[0]
    c = O.ln_bwd_cols(x, dy, mu, rs)
    out["ln dgamma"], out["ln dbeta"] = c["dgamma"], c["dbeta"]
    out["rms dx"] = O.rms_bwd_rows(x, dy, eps, g, O.F32, O.MATH)[0]
    out["rms dw"] = O.rms_bwd_cols(x, dy, eps, O.F32, O.MATH)[0]
    return out


def test_backwards_linear_in_dy(O):
    rng = np.random.default_rng(40)
    M, N = 6, 11
    x = rng.standard_normal((M, N))
    d1, d2 = rng.standard_normal((M, N)), rng.standard_normal((M, N))
    g, b = 1 + 0.3 * rng.standard_normal(N), rng.standard_normal(N)
    a1, a2 = 0.75, -2.5
    o1 = _backwards(O, x, d1, g, b, 0.01)
    o2 = _backwards(O, x, d2, g, b, 0.01)
    o12 = _backwards(O, x, a1 * d1 + a2 * d2, g, b, 0.01)
    for k in o12:
        np.testing.assert_allclose(o12[k], a1 * o1[k] + a2 * o2[k], rtol=1e-12, atol=1e-12,
                                   err_msg=k)


def test_backwards_equivariant_under_row_and_column_permutations(O):
    rng = np.random.default_rng(41)
    M, N = 7, 9
    x = rng.standard_normal((M, N)) + 0.5
    dy = rng.standard_normal((M, N))
    g, b = 1 + 0.3 * rng.standard_normal(N), rng.standard_normal(N)
    base = _backwards(O, x, dy, g, b, 0.02)
    pr, pc = rng.permutation(M), rng.permutation(N)
    rows = _backwards(O, x[pr], dy[pr], g, b, 0.02)
    cols = _backwards(O, x[:, pc], dy[:, pc], g[pc], b[pc], 0.02)
    for k in base:
        if k.endswith(" dx"):
            np.testing.assert_allclose(rows[k], base[k][pr], rtol=1e-13, atol=1e-14, err_msg=k)
            np.testing.assert_allclose(cols[k], base[k][:, pc], rtol=1e-12, atol=1e-13,
                                       err_msg=k)
        elif k == "dyt dalpha":
            np.testing.assert_allclose(rows[k], base[k], rtol=1e-12, err_msg=k)
            np.testing.assert_allclose(cols[k], base[k], rtol=1e-12, err_msg=k)
        else:
            np.testing.assert_allclose(rows[k], base[k], rtol=1e-12, atol=1e-13, err_msg=k)
            np.testing.assert_allclose(cols[k], base[k][pc], rtol=1e-12, atol=1e-13,
                                       err_msg=k)

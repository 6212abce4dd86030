"""Pin of the oracle quantizer's two IEEE divisions (CPU only).

The quantizer ("4.4 KV Cache 量化", section 3.1: min/max asymmetric mapping)
is read as s = fl(fl(max - min) / levels) and c = rne(fl(fl(x - min) / s)),
every step one binary32 operation rounded to nearest-even. This file computes
those roundings exactly, from integers and rationals, with no use of a
floating-point divide, and compares the oracle's codes, scales and minima bit
for bit. It also builds inputs on which the plausible slips give different
codes or scales, and checks that such inputs really occur in the test:
  * multiplying by a rounded reciprocal, x * fl(1/s) or range * fl(1/levels);
  * skipping the binary32 rounding of the quotient before the integer
    rounding (rounding the exact, or double-precision, quotient instead).
"""
from fractions import Fraction

import numpy as np

import oracle


# ------------------------------------------------------ exact binary32 helpers --
def fl32(q: Fraction) -> np.float32:
    """Round a rational to binary32, nearest with ties to even (normal and
    subnormal range; the tests never reach overflow)."""
    if q == 0:
        return np.float32(0.0)
    neg = q < 0
    a = -q if neg else q
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2^e <= a < 2^(e+2)
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                       # below 2^-126 the quantum stays 2^-149
    quantum = Fraction(2) ** (e - 23)
    n = round(a / quantum)                 # Fraction.__round__: half to even
    v = float(n * quantum)                 # exact: n has at most 24 bits
    return np.float32(-v if neg else v)


def rne_int(t: Fraction) -> int:
    """Nearest integer, ties to the even one, written out."""
    f = t.numerator // t.denominator
    d = t - f
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def exact_group(x: np.ndarray, bits: int):
    """The quantizer with every binary32 rounding done exactly."""
    levels = (1 << bits) - 1
    xs = [Fraction(float(v)) for v in x]
    lo, hi = min(xs), max(xs)
    s = fl32(Fraction(float(fl32(hi - lo))) / levels)
    sf = Fraction(float(s))
    codes = []
    for v in xs:
        if sf == 0:
            codes.append(0)
            continue
        t = fl32(Fraction(float(fl32(v - lo))) / sf)
        codes.append(min(max(rne_int(Fraction(float(t))), 0), levels))
    return np.array(codes, np.uint8), s, fl32(lo)


# ----------------------------------------- the same, vectorised on integers --
def _split(a):
    """a = m * 2^e with m a 24-bit integer in [2^23, 2^24) (a > 0, normal)."""
    f, e = np.frexp(a.astype(np.float64))
    return (f * (1 << 24)).astype(np.int64), e.astype(np.int64) - 24


def div_rne(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Correctly rounded binary32 quotient a / b for a >= 0 and b > 0 (both
    normal binary32, quotient normal), by integer long division: the 24-bit
    significands give a quotient of 25 or 26 significant bits plus a
    remainder, rounded to 24 bits with ties to even."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    out = np.zeros(a.shape, np.float32)
    nz = a != 0
    ia, ea = _split(a[nz])
    ib, eb = _split(b[nz])
    num = ia << 26                          # < 2^50
    q, r = num // ib, num % ib              # q in (2^25, 2^27)
    sh = np.where(q >= (1 << 26), 3, 2)
    keep = q >> sh
    dropped = q & ((1 << sh) - 1)
    half = 1 << (sh - 1)
    up = (dropped > half) | ((dropped == half) & ((r != 0) | ((keep & 1) == 1)))
    keep = keep + up
    val = np.ldexp(keep.astype(np.float64), (sh + ea - eb - 26).astype(np.int32))
    assert np.all(val >= 2.0 ** -126), "quotients in the normal range only"
    out[nz] = val.astype(np.float32)        # exact: keep has at most 24 bits (or is 2^24)
    return out


def sub_rne(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """binary32 x - y, rounded once. The float64 difference is checked to be
    error-free (two-sum), so rounding it to binary32 is the single rounding."""
    a, b = x.astype(np.float64), -y.astype(np.float64)
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    assert np.all(err == 0), "float64 difference not exact for these inputs"
    return s.astype(np.float32)


def rne_int_vec(t: np.ndarray) -> np.ndarray:
    t = t.astype(np.float64)
    f = np.floor(t)
    d = t - f                               # exact: t has 24 significant bits
    up = (d > 0.5) | ((d == 0.5) & (np.mod(f, 2) == 1))
    return (f + up).astype(np.int64)


def exact_groups_vec(X: np.ndarray, n: np.ndarray, bits: int):
    """X [groups, 32] float32, the first n[g] entries of row g used."""
    levels = (1 << bits) - 1
    mask = np.arange(X.shape[1])[None, :] < n[:, None]
    lo = np.where(mask, X, np.inf).min(axis=1).astype(np.float32) + np.float32(0)
    hi = np.where(mask, X, -np.inf).max(axis=1).astype(np.float32) + np.float32(0)
    rng = sub_rne(hi, lo)
    s = np.zeros_like(rng)
    pos = rng > 0
    s[pos] = div_rne(rng[pos], np.full(pos.sum(), levels, np.float32))
    a = sub_rne(np.where(mask, X, lo[:, None]), np.broadcast_to(lo[:, None], X.shape))
    t = np.zeros_like(a)
    live = pos[:, None] & mask & (a > 0)
    t[live] = div_rne(a[live], np.broadcast_to(s[:, None], X.shape)[live])
    codes = np.clip(rne_int_vec(t), 0, levels)
    codes[~(pos[:, None] & mask)] = 0
    return codes.astype(np.uint8), s, lo


# --------------------------------------------------------------------- tests --
def test_vectorised_division_matches_exact_rationals():
    """The integer long division used below agrees with Fraction arithmetic."""
    rng = np.random.default_rng(5)
    a = (rng.uniform(0.5, 1.0, 4000) * 2.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    b = (rng.uniform(0.5, 1.0, 4000) * 2.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    got = div_rne(a, b)
    for x, y, z in zip(a, b, got):
        assert z.view(np.uint32) == fl32(Fraction(float(x)) / Fraction(float(y))).view(np.uint32)


def test_oracle_equals_exact_roundings_on_random_groups():
    """10^5 random groups (sizes 1..32, fp16- and bf16-valued inputs over six
    decades, 4- and 2-bit codes): codes, scale and min bit for bit."""
    rng = np.random.default_rng(17)
    G = 100_000
    n = rng.integers(1, 33, G)
    scale = 10.0 ** rng.uniform(-3, 3, G)
    X = rng.normal(size=(G, 32)) * scale[:, None] + rng.normal(size=(G, 1)) * scale[:, None]
    X16 = X.astype(np.float16).astype(np.float32)
    Xb = X.astype(np.float32)
    Xb = (Xb.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)   # bf16 values (truncated)
    X = np.where((np.arange(G) % 2 == 0)[:, None], X16, Xb)
    bits = np.where(np.arange(G) % 4 == 3, 2, 4)
    for b in (4, 2):
        sel = np.nonzero(bits == b)[0]
        ec, es, el = exact_groups_vec(X[sel], n[sel], b)
        for j, gi in enumerate(sel):
            c, s, mn = oracle.quantize_group(X[gi, :n[gi]], bits=b)
            assert np.array_equal(c, ec[j, :n[gi]]), (gi, b)
            assert np.float32(s).view(np.uint32) == es[j].view(np.uint32), (gi, b)
            assert np.float32(mn).view(np.uint32) == el[j].view(np.uint32), (gi, b)


def _near_half_cases(bits: int, seed: int, want: int):
    """Groups [0, range, a_1, ...] whose quotients a_i / s fall next to a
    half-integer, where the wrong divisions round the other way."""
    levels = (1 << bits) - 1
    rng = np.random.default_rng(seed)
    recip_diff, noround_diff, scale_diff = [], [], []
    groups = []
    while len(recip_diff) < want or len(noround_diff) < want:
        R = np.float32(rng.uniform(0.5, 1.0) * 2.0 ** rng.integers(-12, 12))
        s = fl32(Fraction(float(R)) / levels)
        if s.view(np.uint32) != np.float32(np.float32(R) * fl32(Fraction(1, levels))).view(np.uint32):
            scale_diff.append(R)
        sF = Fraction(float(s))
        inv = fl32(1 / sF)
        xs = []
        for k in range(levels):
            a0 = fl32((k + Fraction(1, 2)) * sF)
            for j in range(-6, 7):
                # positive binary32: adding j to the bit pattern moves j ulps
                a = np.array([a0.view(np.uint32) + np.uint32(j + 8)], np.uint32)
                a = (a - np.uint32(8)).view(np.float32)[0]
                if not (0 < a < R):
                    continue
                Q = Fraction(float(a)) / sF
                c_exact = rne_int(Fraction(float(fl32(Q))))
                c_recip = rne_int(Fraction(float(fl32(Fraction(float(a)) * Fraction(float(inv))))))
                c_noround = rne_int(Q)
                hit = False
                if c_recip != c_exact:
                    recip_diff.append((R, a))
                    hit = True
                if c_noround != c_exact:
                    noround_diff.append((R, a))
                    hit = True
                if hit:
                    xs.append(a)
        for i in range(0, len(xs), 30):
            groups.append(np.array([0.0, R] + xs[i:i + 30], np.float32))
    return groups, recip_diff, noround_diff, scale_diff


def test_divisions_on_inputs_that_tell_the_slips_apart():
    for bits in (4, 2):
        groups, recip_diff, noround_diff, scale_diff = _near_half_cases(bits, 40 + bits, 200)
        assert len(recip_diff) >= 200 and len(noround_diff) >= 200
        for x in groups:
            c, s, mn = oracle.quantize_group(x, bits=bits)
            ec, es, el = exact_group(x, bits)
            assert np.array_equal(c, ec), (x, bits)
            assert np.float32(s).view(np.uint32) == es.view(np.uint32)
            assert np.float32(mn).view(np.uint32) == el.view(np.uint32)


def test_scale_division_on_ranges_where_the_reciprocal_differs():
    """s = fl(range / levels), not fl(range * fl(1 / levels)): ranges where the
    two differ occur, and the oracle's scale is the correctly rounded one."""
    rng = np.random.default_rng(23)
    for levels, bits in ((15, 4), (3, 2)):
        R = (rng.uniform(0.5, 1.0, 20000) * 2.0 ** rng.integers(-20, 20, 20000)).astype(np.float32)
        exact = div_rne(R, np.full(R.shape, levels, np.float32))
        recip = R * fl32(Fraction(1, levels))
        differ = np.nonzero(exact.view(np.uint32) != recip.view(np.uint32))[0]
        assert differ.size > 100
        for i in differ[:400]:
            _, s, _ = oracle.quantize_group(np.array([0.0, R[i]], np.float32), bits=bits)
            assert np.float32(s).view(np.uint32) == exact[i].view(np.uint32)
            assert np.float32(s).view(np.uint32) != recip[i].view(np.uint32)


def test_range_subtraction_is_one_rounding():
    """fl(max - min) with an inexact difference (operands of far-apart
    magnitudes): the oracle's scale equals fl(fl(max - min) / 15)."""
    rng = np.random.default_rng(29)
    for _ in range(2000):
        hi = np.float32(rng.uniform(1, 2) * 2.0 ** rng.integers(0, 20))
        lo = np.float32(-rng.uniform(1, 2) * 2.0 ** rng.integers(-30, -5))
        x = np.array([hi, lo, np.float32(0.5) * hi], np.float32)
        c, s, mn = oracle.quantize_group(x)
        ec, es, el = exact_group(x, 4)
        assert np.float32(s).view(np.uint32) == es.view(np.uint32)
        assert np.array_equal(c, ec)

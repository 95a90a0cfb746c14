"""Pins for the FP64 oracle: things fixed by the pages and by mathematics, not
by the oracle itself.

* the pages' printed FP32 -> BF16 conversions (sec. 6.2, Fig. 5),
* torch's bf16 conversion as an independent library routine,
* exact-rational brute force on tiny shapes (Python `fractions`),
* closed forms: rank 1 / K 1, one-hot rows, zero weights, no-adapter tokens,
* small-integer inputs, where every sum is exact,
* planted mistakes: mutated copies of the oracle must fail at least one pin.
"""
from fractions import Fraction
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers that do not use the oracle
# --------------------------------------------------------------------------

def torch_bf16_bits(values_f32) -> np.ndarray:
    t = torch.from_numpy(np.asarray(values_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_value(bits) -> np.ndarray:
    """bf16 bits -> float64 through torch (independent of oracle.bf16_to_f64)."""
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def rand_bf16(rng, shape, scale=1.0):
    return torch_bf16_bits(rng.standard_normal(shape) * scale)


def frac_of_bits(b):
    return Fraction(float(bits_value(np.array([b]))[0]))


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def _read_golden_rounding():
    singles, pairs = [], []
    with open(os.path.join(GOLDEN, "bf16_rounding_pages.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p = line.split()
            if p[0] == "pair":
                pairs.append((float(p[1]), float(p[2]), float(p[4])))
            else:
                singles.append((float(p[0]), None if p[1] == "-" else float(p[1])))
    return singles, pairs


def test_golden_values_are_fp32():
    singles, _ = _read_golden_rounding()
    for v, _ in singles:
        assert float(np.float32(v)) == v


def test_bf16_round_pages_examples():
    singles, pairs = _read_golden_rounding()
    for v, want in singles:
        got = oracle.bf16_to_f64(oracle.bf16_round([v]))[0]
        if want is not None:
            assert got == want, (v, got, want)
    for a, b, gap in pairs:
        ga, gb = oracle.bf16_to_f64(oracle.bf16_round([a, b]))
        assert ga != gb
        # printed to three significant digits
        assert abs(abs(ga - gb) - gap) <= 5e-3 * gap + 1e-12, (a, b, ga, gb, gap)


def test_bf16_round_midpoints_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even neighbour is 1.
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    cases = [(1 + 2**-8, 1.0), (1 + 3 * 2**-8, 1 + 2**-6),
             (-(1 + 2**-8), -1.0), (2**-130 * 1.5, 2**-130 * 1.5),
             (2**-134, 0.0), (3 * 2**-134, 2**-132)]
    for v, want in cases:
        got = oracle.bf16_to_f64(oracle.bf16_round([v]))[0]
        assert got == want, (v, got, want)


def test_bf16_round_matches_torch_on_fp32():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormals
        np.clip(rng.standard_normal(2000) * 1e38, -3.4e38, 3.4e38).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4e38], np.float32),
    ])
    # exact midpoints of random bf16 neighbours
    hi = (rng.integers(0, 2**15, 4000, dtype=np.uint32) << 16) | 0x8000
    v = np.concatenate([v, hi.view(np.float32)])
    v = v[np.isfinite(v) | np.isinf(v)]
    got = oracle.bf16_round(v.astype(np.float64))
    want = torch_bf16_bits(v)
    assert np.array_equal(got, want)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    a = oracle.bf16_to_f64(bits)
    b = bits_value(bits)
    same = (a == b) | (np.isnan(a) & np.isnan(b))
    assert same.all()


def test_eq4_nonassociativity_fp32():
    with open(os.path.join(GOLDEN, "eq4_nonassociativity.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for a, b, c, left, right in rows:
        a, b, c = np.float32(a), np.float32(b), np.float32(c)
        assert float((a + b) + c) == float(left)
        assert float(a + (b + c)) == float(right)


# --------------------------------------------------------------------------
# pins on shrink / expand, written against any implementation so that the
# planted-mistake test can run them on mutants
# --------------------------------------------------------------------------

def _tiny(seed, M=3, K=24, r=4, N=5, L=2, slices=2):
    rng = np.random.default_rng(seed)
    x = rand_bf16(rng, (M, K))
    A = rand_bf16(rng, (L, slices, r, K), 0.3)
    B = rand_bf16(rng, (L, slices, N, r), 0.5)
    y = rand_bf16(rng, (M, slices * N))
    idx = rng.integers(-1, L, M).astype(np.int32)
    idx[0] = 1
    return x, A, B, y, idx


def pin_shrink_bruteforce(shrink):
    """Exact rationals: z equals the true sum to float64 accuracy."""
    for seed in range(4):
        x, A, B, y, idx = _tiny(seed)
        scale = 1.75
        z, bound = shrink(x, A, idx, scale)
        L, slices, r, K = A.shape
        M = x.shape[0]
        for sl in range(slices):
            for m in range(M):
                for j in range(r):
                    if idx[m] < 0:
                        exact = Fraction(0)
                        absb = Fraction(0)
                    else:
                        terms = [frac_of_bits(x[m, k]) * frac_of_bits(A[idx[m], sl, j, k])
                                 for k in range(K)]
                        exact = Fraction(scale) * sum(terms, Fraction(0))
                        absb = abs(Fraction(scale)) * sum((abs(t) for t in terms), Fraction(0))
                    err = abs(Fraction(float(z[sl, m, j])) - exact)
                    if err > absb * Fraction(K + 2, 2**52):
                        return False
                    if abs(Fraction(float(bound[sl, m, j])) - absb) > absb * Fraction(K + 2, 2**52):
                        return False
    return True


def pin_shrink_integers(shrink):
    """Small integers: every sum is exact, compare with int64 matmul."""
    rng = np.random.default_rng(11)
    M, K, r, L, slices = 7, 64, 8, 3, 2
    xi = rng.integers(-4, 5, (M, K))
    Ai = rng.integers(-4, 5, (L, slices, r, K))
    idx = np.array([0, 2, 1, -1, 2, 0, 1], np.int32)
    z, _ = shrink(torch_bf16_bits(xi), torch_bf16_bits(Ai), idx, 2.0)
    for sl in range(slices):
        for m in range(M):
            want = np.zeros(r, np.int64) if idx[m] < 0 else 2 * (Ai[idx[m], sl] @ xi[m])
            if not np.array_equal(z[sl, m], want.astype(np.float64)):
                return False
    return True


def pin_shrink_closed_forms(shrink):
    rng = np.random.default_rng(5)
    # K = 1, r = 1: z = s * x * a
    x = rand_bf16(rng, (4, 1))
    A = rand_bf16(rng, (2, 1, 1, 1))
    idx = np.array([0, 1, 1, 0], np.int32)
    z, _ = shrink(x, A, idx, 2.0)
    want = 2.0 * bits_value(x)[:, 0] * bits_value(A)[idx, 0, 0, 0]
    if not np.array_equal(z[0, :, 0], want):
        return False
    # one-hot A rows: z[m, j] = s * x[m, k_j]
    K, r = 32, 4
    x = rand_bf16(rng, (3, K))
    kj = [5, 0, 31, 17]
    A = np.zeros((1, 1, r, K), np.uint16)
    for j, k in enumerate(kj):
        A[0, 0, j, k] = torch_bf16_bits([1.0])[0]
    z, _ = shrink(x, A, np.zeros(3, np.int32), 0.5)
    if not np.array_equal(z[0], 0.5 * bits_value(x)[:, kj]):
        return False
    # adapter -1: zero row
    z, _ = shrink(x, A, np.array([-1, 0, -1], np.int32), 0.5)
    if not (np.all(z[0, 0] == 0) and np.all(z[0, 2] == 0)):
        return False
    return True


def pin_expand_bruteforce(expand):
    for seed in range(4):
        x, A, B, y, idx = _tiny(seed)
        L, slices, N, r = B.shape
        M = y.shape[0]
        rng = np.random.default_rng(100 + seed)
        z32 = (rng.standard_normal((slices, M, r)) * 3).astype(np.float32)
        y_exact, bound, out = expand(z32, B, idx, y)
        zb = bits_value(torch_bf16_bits(z32))          # torch's rounding of Z
        for m in range(M):
            for sl in range(slices):
                for n in range(N):
                    col = sl * N + n
                    yv = frac_of_bits(y[m, col])
                    if idx[m] < 0:
                        if out[m, col] != y[m, col]:
                            return False
                        continue
                    terms = [Fraction(float(zb[sl, m, j])) * frac_of_bits(B[idx[m], sl, n, j])
                             for j in range(r)]
                    exact = yv + sum(terms, Fraction(0))
                    # the exact value fits a double here (few terms, close exponents)
                    if Fraction(float(y_exact[m, col])) != exact:
                        return False
                    absb = abs(yv) + sum((abs(t) for t in terms), Fraction(0))
                    if Fraction(float(bound[m, col])) != absb:
                        return False
                    # the output is one of the two bf16 neighbours of exact,
                    # and the nearer one
                    got = Fraction(float(bits_value(out[m:m + 1, col])[0]))
                    alt = torch_bf16_bits([float(exact)])[0]   # exact fits float32?
                    if float(np.float32(float(exact))) == float(exact):
                        if out[m, col] != alt:
                            return False
                    if abs(got - exact) > abs(exact) / 256 + Fraction(1, 2**140):
                        return False
    return True


def pin_expand_closed_forms(expand):
    rng = np.random.default_rng(9)
    M, N, r = 4, 6, 8
    y = rand_bf16(rng, (M, N))
    z = (rng.standard_normal((1, M, r))).astype(np.float32)
    # zero B: y unchanged
    B = np.zeros((1, 1, N, r), np.uint16)
    _, _, out = expand(z, B, np.zeros(M, np.int32), y)
    if not np.array_equal(out, y):
        return False
    # one-hot B: y[m, n] = bf16(y + bf16(z[m, j_n]))
    jn = [0, 3, 7, 1, 2, 5]
    B = np.zeros((1, 1, N, r), np.uint16)
    for n, j in enumerate(jn):
        B[0, 0, n, j] = torch_bf16_bits([1.0])[0]
    _, _, out = expand(z, B, np.zeros(M, np.int32), y)
    zb = bits_value(torch_bf16_bits(z))
    for m in range(M):
        for n, j in enumerate(jn):
            s = float(bits_value(y[m:m + 1, n])[0]) + float(zb[0, m, j])
            if float(np.float32(s)) != s:
                continue
            if out[m, n] != torch_bf16_bits([s])[0]:
                return False
    # no adapter: row untouched even with nonzero weights
    B = rand_bf16(rng, (1, 1, N, r))
    _, _, out = expand(z, B, np.array([-1, 0, -1, 0], np.int32), y)
    if not (np.array_equal(out[0], y[0]) and np.array_equal(out[2], y[2])):
        return False
    return True


def pin_expand_integers(expand):
    rng = np.random.default_rng(3)
    M, N, r, L = 5, 16, 8, 2
    zi = rng.integers(-300, 300, (1, M, r))
    Bi = rng.integers(-4, 5, (L, 1, N, r))
    yi = rng.integers(-4, 5, (M, N))
    idx = np.array([0, 1, 1, 0, -1], np.int32)
    zb = bits_value(torch_bf16_bits(zi.astype(np.float32))).astype(np.int64)  # bf16(z), integers
    _, _, out = expand(zi.astype(np.float32), torch_bf16_bits(Bi), idx, torch_bf16_bits(yi))
    for m in range(M):
        if idx[m] < 0:
            want = yi[m]
        else:
            want = yi[m] + Bi[idx[m], 0] @ zb[0, m]
        if not np.array_equal(out[m], torch_bf16_bits(want.astype(np.float32))):
            return False
    return True


SHRINK_PINS = [pin_shrink_bruteforce, pin_shrink_integers, pin_shrink_closed_forms]
EXPAND_PINS = [pin_expand_bruteforce, pin_expand_closed_forms, pin_expand_integers]


@pytest.mark.parametrize("pin", SHRINK_PINS, ids=lambda f: f.__name__)
def test_oracle_shrink_pins(pin):
    assert pin(oracle.shrink)


@pytest.mark.parametrize("pin", EXPAND_PINS, ids=lambda f: f.__name__)
def test_oracle_expand_pins(pin):
    assert pin(oracle.expand)


def test_oracle_expand_fp32_z_bruteforce():
    """round_z=False: y_exact = y + sum_j z_j B_nj with the FP32 z values as
    they are (exact rationals, tiny shapes)."""
    for seed in range(3):
        x, A, B, y, idx = _tiny(seed)
        L, slices, N, r = B.shape
        M = y.shape[0]
        rng = np.random.default_rng(50 + seed)
        z32 = (rng.standard_normal((slices, M, r)) * 3).astype(np.float32)
        y_exact, bound, out = oracle.expand(z32, B, idx, y, round_z=False)
        for m in range(M):
            if idx[m] < 0:
                continue
            for sl in range(slices):
                for n in range(N):
                    exact = frac_of_bits(y[m, sl * N + n]) + sum(
                        (Fraction(float(z32[sl, m, j])) * frac_of_bits(B[idx[m], sl, n, j])
                         for j in range(r)), Fraction(0))
                    got = Fraction(float(y_exact[m, sl * N + n]))
                    assert abs(got - exact) <= abs(exact) * Fraction(1, 2**50) + Fraction(1, 2**200)


def test_oracle_apply_chains_stages():
    x, A, B, y, idx = _tiny(21)
    z32, y_exact, bound, out = oracle.apply(x, y, idx, A, B, 2.0)
    z, _ = oracle.shrink(x, A, idx, 2.0)
    assert np.array_equal(z32, z.astype(np.float32))
    y2, b2, o2 = oracle.expand(z32, B, idx, y)
    assert np.array_equal(out, o2) and np.array_equal(y_exact, y2)


def test_oracle_rejects_bad_adapter():
    x, A, B, y, idx = _tiny(1)
    idx = idx.copy()
    idx[1] = A.shape[0]
    with pytest.raises(ValueError):
        oracle.shrink(x, A, idx, 1.0)
    idx[1] = -2
    with pytest.raises(ValueError):
        oracle.expand(np.zeros((A.shape[1], x.shape[0], A.shape[2]), np.float32), B, idx, y)


# --------------------------------------------------------------------------
# planted mistakes: each mutant of the oracle must fail some pin
# --------------------------------------------------------------------------

def _mut_shrink(kind):
    f64 = oracle.bf16_to_f64

    def shrink(x_bits, A_bits, idx, scale):
        x = f64(x_bits)
        A = f64(A_bits)
        L, slices, r, K = A.shape
        M = x.shape[0]
        idx = np.asarray(idx).astype(np.int64)
        z = np.zeros((slices, M, r))
        bound = np.zeros((slices, M, r))
        for a in np.unique(idx):
            if a < 0:
                continue
            rows = np.nonzero(idx == a)[0]
            src = (a + 1) % L if kind == "wrong_adapter" else a
            for sl in range(slices):
                Aas = A[src, sl]
                if kind == "dropped_term":
                    Aas = Aas.copy()
                    Aas[:, -1] = 0
                if kind == "transposed":
                    Aas = Aas.reshape(K, r).T
                s = 1.0 if kind == "no_scale" else scale
                if kind == "sign":
                    s = -s
                if kind == "scale_squared":
                    s = scale * scale
                xr = x[np.roll(rows, 1)] if kind == "rows_rolled" else x[rows]
                zz = s * (xr @ Aas.T)
                if kind == "j_reversed":
                    zz = zz[:, ::-1]
                z[sl, rows] = zz
                bound[sl, rows] = abs(scale) * (np.abs(x[rows]) @ np.abs(Aas).T)
        return z, bound
    return shrink


def _mut_expand(kind):
    f64 = oracle.bf16_to_f64

    def expand(z_f32, B_bits, idx, y_bits):
        z = np.asarray(z_f32, dtype=np.float32)
        B = f64(B_bits)
        L, slices, N, r = B.shape
        M = z.shape[1]
        idx = np.asarray(idx).astype(np.int64)
        if kind == "no_z_rounding":
            zb = z.astype(np.float64)
        elif kind == "z_truncated":
            zb = f64((z.view(np.uint32) >> 16).astype(np.uint16))
        else:
            zb = f64(oracle.bf16_round(z.astype(np.float64)))
        y = f64(y_bits)
        y_exact = y.copy()
        bound = np.abs(y)
        for a in np.unique(idx):
            if a < 0:
                if kind == "none_touched":
                    y_exact[idx == a] = y[idx == a] + 1
                continue
            rows = np.nonzero(idx == a)[0]
            for sl in range(slices):
                Bas = B[(a + 1) % L if kind == "wrong_adapter" else a, sl]
                cols = slice(sl * N, (sl + 1) * N)
                if kind == "slice_swapped":
                    Bas = B[a, (sl + 1) % slices]
                if kind == "b_strided":     # B read as [r][N] instead of [N][r]
                    Bas = Bas.reshape(r, N).T
                add = zb[sl, rows] @ Bas.T
                if kind == "scaled_twice":
                    add = 2.0 * add
                if kind == "n_reversed":
                    add = add[:, ::-1]
                if kind == "y_dropped":
                    y_exact[rows, cols] = add
                else:
                    y_exact[rows, cols] = y[rows, cols] + add
                bound[rows, cols] = np.abs(y[rows, cols]) + np.abs(zb[sl, rows]) @ np.abs(Bas).T
        out = np.asarray(y_bits).astype(np.uint16).copy()
        if kind == "none_touched":
            out = oracle.bf16_round(y_exact)
        elif kind == "y_truncated":   # final conversion drops the low bits
            act = idx >= 0
            out[act] = (y_exact[act].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        else:
            act = idx >= 0
            out[act] = oracle.bf16_round(y_exact[act])
        return y_exact, bound, out
    return expand


@pytest.mark.parametrize("kind", ["wrong_adapter", "dropped_term", "transposed",
                                  "no_scale", "sign", "j_reversed", "scale_squared",
                                  "rows_rolled"])
def test_planted_shrink_mistakes_are_caught(kind):
    mut = _mut_shrink(kind)
    caught = []
    for pin in SHRINK_PINS:
        try:
            caught.append(not pin(mut))
        except Exception:
            caught.append(True)
    assert any(caught), kind


@pytest.mark.parametrize("kind", ["no_z_rounding", "z_truncated", "none_touched",
                                  "slice_swapped", "y_dropped", "wrong_adapter",
                                  "b_strided", "scaled_twice", "n_reversed", "y_truncated"])
def test_planted_expand_mistakes_are_caught(kind):
    mut = _mut_expand(kind)
    caught = []
    for pin in EXPAND_PINS:
        try:
            caught.append(not pin(mut))
        except Exception:
            caught.append(True)
    assert any(caught), kind

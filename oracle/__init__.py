"""FP64 CPU oracle for the multi-adapter LoRA shrink/expand path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports or calls this
package: only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` use it. It shares no code with the CUDA library.

It is a plain restatement of what "Reproducible LoRA Inference Through
Deterministic Split-K Reduction" (Balusamy & Mohan) defines, written with
numpy in float64:

* Eq. 1: a LoRA linear layer adds s * (X A^T) B^T to the base output, with
  A in R^{r x H} and B in R^{Hout x r}. The shrink is X A^T (sec. 2).
* Eq. 3: Split-K only regroups the sum over the reduction index; every split
  count S reaches the same mathematical value, so the oracle evaluates the
  plain sum and does not emulate partitions (sec. 2.2, Algorithm 1).
* Algorithm 1 / Fig. 2: the scale factor is applied to the combined shrink
  output ("x alpha/r"), giving an FP32 tensor Z.
* Sec. 6.2 / Fig. 5: Z is converted FP32 -> BF16 with round-to-nearest before
  the expand consumes it.

Exact arithmetic claims:
* bf16 inputs widen to float64 exactly, and each bf16 x bf16 product is exact
  in float64 (8 + 8 significant bits).
* The sums use float64 matmul, whose error (K * 2^-53 relative to the sum of
  absolute terms, < 4e-12 for K <= 28672) is far below every tolerance the
  tests use. On small-integer inputs all sums are exact.

Readings where the pages are silent (also listed in the design notes):
* Tokens with adapter index -1 get a zero Z row and an untouched y row.
* The expand adds the bf16-rounded Z times B to f32(y) and rounds once to
  bf16 (no intermediate rounding of the LoRA delta).
* Rounding to bf16 is round-to-nearest, ties to even.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f64",
    "bf16_round",
    "shrink",
    "expand",
    "apply",
]


# --------------------------------------------------------------------------
# bf16 encoding (bit patterns are carried as uint16)
# --------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns: the high 16 bits of an IEEE binary32."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


_BF16_MIN_EXP = -133          # exponent of the smallest bf16 subnormal, 2^-126 * 2^-7
_BF16_OVERFLOW = 2.0 ** 128   # first value past the largest finite bf16


def bf16_round(v) -> np.ndarray:
    """Round real values (given as float64) to bf16, nearest with ties to even.

    bf16 keeps 8 significant bits. For v = m * 2^e with 0.5 <= |m| < 1
    (np.frexp), the spacing of bf16 values near v is 2^(e-8), floored at the
    subnormal spacing 2^-133. Scaling by that power of two is exact, np.rint
    rounds half to even, and scaling back is exact. Results of magnitude
    2^128 or more overflow to infinity. Returns uint16 bit patterns.

    Sec. 6.2 and Fig. 5 print FP32 values on both sides of bf16 rounding
    midpoints with the bf16 values they convert to; the tests pin this
    function to those examples.
    """
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(v)
        q_exp = np.maximum(e.astype(np.int64) - 8, _BF16_MIN_EXP)
        q = np.ldexp(v, -q_exp)
        rv = np.ldexp(np.rint(q), q_exp)
        rv = np.where(np.abs(rv) >= _BF16_OVERFLOW, np.copysign(np.inf, v), rv)
        f = rv.astype(np.float32)
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(v)
    if nan.any():
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits


# --------------------------------------------------------------------------
# the path
# --------------------------------------------------------------------------

def _check_idx(idx, L):
    idx = np.asarray(idx).astype(np.int64)
    if idx.size and (idx.min() < -1 or idx.max() >= L):
        raise ValueError("adapter index outside [-1, L)")
    return idx


def shrink(x_bits, A_bits, idx, scale):
    """Z[sl, m, j] = scale * sum_k x[m, k] * A[idx[m], sl, j, k]   (Eq. 1, Eq. 3).

    x_bits  uint16 [M][K]            bf16 activations
    A_bits  uint16 [L][slices][r][K] bf16 stacked shrink weights
    idx     int    [M]               adapter per token, -1 = none
    Returns (z, bound), both float64 [slices][M][r]:
      z     the value in float64 (exact up to float64 rounding)
      bound |scale| * sum_k |x[m,k] * A[idx[m],sl,j,k]|, the scale of the terms,
            used to size the FP32 tolerance
    """
    x = bf16_to_f64(x_bits)
    A = bf16_to_f64(A_bits)
    L, slices, r, K = A.shape
    M = x.shape[0]
    assert x.shape == (M, K)
    idx = _check_idx(idx, L)
    z = np.zeros((slices, M, r))
    bound = np.zeros((slices, M, r))
    for a in np.unique(idx):
        if a < 0:
            continue
        rows = np.nonzero(idx == a)[0]
        xa = x[rows]
        for sl in range(slices):
            Aas = A[a, sl]                      # [r][K]
            z[sl, rows] = scale * (xa @ Aas.T)
            bound[sl, rows] = abs(scale) * (np.abs(xa) @ np.abs(Aas).T)
    return z, bound


def expand(z_f32, B_bits, idx, y_bits, round_z=True):
    """y[m, sl*N + n] += sum_j bf16(Z[sl, m, j]) * B[idx[m], sl, n, j]   (Eq. 1).

    z_f32   float32 [slices][M][r]   shrink output as stored (FP32)
    B_bits  uint16  [L][slices][N][r] bf16 stacked expand weights
    idx     int     [M]
    y_bits  uint16  [M][slices*N]    bf16 base output, updated
    Z is first rounded to bf16 (sec. 6.2: the FP32 shrink output reaches the
    next operation in bf16); with round_z=False the FP32 values are used as
    they are (the precision variant that keeps Z in FP32).
    Returns (y_exact, bound, y_bits_out):
      y_exact    float64 value y + sum_j zb_j * B_nj, before the final rounding
      bound      |y| + sum_j |zb_j * B_nj|
      y_bits_out bf16_round(y_exact) for rows with an adapter, y unchanged else
    """
    z = np.asarray(z_f32, dtype=np.float32)
    B = bf16_to_f64(B_bits)
    L, slices, N, r = B.shape
    M = z.shape[1]
    assert z.shape == (slices, M, r)
    y_bits = np.asarray(y_bits).astype(np.uint16)
    assert y_bits.shape == (M, slices * N)
    idx = _check_idx(idx, L)
    if round_z:
        zb = bf16_to_f64(bf16_round(z.astype(np.float64)))
    else:
        zb = z.astype(np.float64)
    y = bf16_to_f64(y_bits)
    y_exact = y.copy()
    bound = np.abs(y)
    for a in np.unique(idx):
        if a < 0:
            continue
        rows = np.nonzero(idx == a)[0]
        for sl in range(slices):
            Bas = B[a, sl]                          # [N][r]
            cols = slice(sl * N, (sl + 1) * N)
            zr = zb[sl, rows]                       # [rows][r]
            y_exact[rows, cols] = y[rows, cols] + zr @ Bas.T
            bound[rows, cols] = np.abs(y[rows, cols]) + np.abs(zr) @ np.abs(Bas).T
    out = y_bits.copy()
    active = idx >= 0
    out[active] = bf16_round(y_exact[active])
    return y_exact, bound, out


def apply(x_bits, y_bits, idx, A_bits, B_bits, scale):
    """Shrink then expand, all in the oracle: Z is rounded FP64 -> FP32 (numpy's
    round-to-nearest cast, the FP32 output type of sec. 4.3) and then handed to
    `expand`. Returns (z_f32, y_exact, bound, y_bits_out)."""
    z, _ = shrink(x_bits, A_bits, idx, scale)
    z32 = z.astype(np.float32)
    y_exact, bound, out = expand(z32, B_bits, idx, y_bits)
    return z32, y_exact, bound, out

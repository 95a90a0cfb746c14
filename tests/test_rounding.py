"""The expand's single bf16 rounding, bit for bit, on every path.

"Reproducible LoRA Inference Through Deterministic Split-K Reduction", sec. 6.2
and Fig. 5: FP32 values that sit on either side of a bf16 rounding midpoint
convert to different bf16 values, so the rounding itself has to be right,
not just close. Here the inputs make y = bf16_rn(f32(y) + D) the only
rounding: B is one-hot (B[n][0] = 1, every other j zero), so D = bf16(z_0)
exactly, and y and bf16(z_0) are bf16 values whose exponents differ by 16 or
less, so f32(y) + D is exact in FP32. The results must then equal the
oracle's bf16_round of the exact sum (pinned to the pages' printed
conversions and to torch's conversion) for

  * ties: y = +-(1 + k 2^-7), D = j 2^-8, odd multiples of 2^-8 halfway
    between two bf16 values (ties to even), plus the non-tie neighbours;
  * random exact sums: y and D of random sign and exponent in [-6, 4];
  * the overflow boundary: y = +-max bf16 (odd last bit) or its even
    neighbour, D = +-2^119 (a half unit in the last place: a tie that rounds
    to infinity from the odd value and stays from the even one) or 2^118.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import oracle
from helpers import bits, need_gpu

pytestmark = pytest.mark.gpu


def _bf16(v) -> np.ndarray:
    """Exactly representable values -> bf16 bit patterns (checked exact)."""
    v = np.asarray(v, dtype=np.float64)
    b = oracle.bf16_round(v)
    assert np.array_equal(oracle.bf16_to_f64(b), v), "value not representable in bf16"
    return b


def _cases(N: int, seed: int):
    """Rows of y (bf16 bits [M][N]) and the per-row D value (float64 [M])."""
    rng = np.random.default_rng(seed)
    ys, ds = [], []
    k = np.arange(N) % 128
    # ties and their neighbours
    for j in range(-7, 8):
        for sign in (1.0, -1.0):
            ys.append(_bf16(sign * (1.0 + k * 2.0 ** -7)))
            ds.append(j * 2.0 ** -8)
    # random exact sums
    for _ in range(96):
        e = rng.integers(-4, 5, size=N)
        f = rng.integers(0, 128, size=N)
        s = rng.choice([-1.0, 1.0], size=N)
        ys.append(_bf16(s * (1.0 + f / 128.0) * np.exp2(e)))
        ds.append(float(rng.choice([-1.0, 1.0]) * (1.0 + rng.integers(0, 128) / 128.0) *
                        2.0 ** int(rng.integers(-6, 5))))
    # the overflow boundary
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127          # largest finite bf16, last bit odd
    even = (2.0 - 2.0 ** -6) * 2.0 ** 127         # its neighbour, last bit even
    for d in (2.0 ** 119, 2.0 ** 118):
        for sign in (1.0, -1.0):
            ys.append(_bf16(sign * np.where(np.arange(N) % 2 == 0, big, even)))
            ds.append(sign * d)
    y = np.stack(ys).astype(np.uint16)
    d = np.asarray(ds, dtype=np.float64)
    _bf16(d)
    return y, d


@pytest.mark.parametrize("path,r", [(ig.PATH_WARP, 16), (ig.PATH_WARP, 8), (ig.PATH_FMA, 16),
                                    (ig.PATH_MMA, 32)])
def test_expand_rounding_bit_exact(path, r):
    need_gpu()
    N = 512
    y_bits, d = _cases(N, seed=20 + r)
    M = y_bits.shape[0]
    z = np.zeros((1, M, r), dtype=np.float32)
    z[0, :, 0] = d.astype(np.float32)
    B = np.zeros((1, 1, N, r), dtype=np.uint16)
    B[..., 0] = _bf16(1.0)
    idx = np.zeros(M, dtype=np.int32)
    _, _, y_ref = oracle.expand(z, B, idx, y_bits)

    sh = ig.make_shape(M, 64, N, r, num_adapters=1, split_k=1, path=path)
    ws = ig.workspace(sh)
    dev = "cuda"
    idx_t = torch.from_numpy(idx).to(dev)
    z_t = torch.from_numpy(z).to(dev)
    B_t = torch.from_numpy(B.view(np.int16)).to(dev).view(torch.bfloat16)
    y_t = torch.from_numpy(y_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    ig.map_tokens(sh, idx_t, ws)
    ig.lora_expand(sh, z_t, B_t, None, y_t, ws)
    assert ig.check_status(ws) == 0
    got = bits(y_t)
    bad = got != y_ref
    if bad.any():
        m, n = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} of {bad.size} differ; first at ({m}, {n}): "
                             f"gpu {got[m, n]:#06x} oracle {y_ref[m, n]:#06x} "
                             f"(y {y_bits[m, n]:#06x}, D {d[m]!r})")
    # the cases do reach ties, infinities and both rounding directions
    y_exact = oracle.bf16_to_f64(y_bits) + d[:, None]
    assert np.isinf(oracle.bf16_to_f64(y_ref)).any()
    assert (oracle.bf16_to_f64(y_ref) != y_exact).any()

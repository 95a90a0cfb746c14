"""Shared helpers for the GPU tests: run the CUDA path through the C ABI and
compare against the FP64 oracle with the tolerances of the path.

Tolerances:
  shrink  |z_gpu - z_ref| <= 1e-5 * |s| * sum_k |x_k A_jk|
  expand  |y_gpu - y_ref| <= 2^-8 |y_ref| + 1e-5 (|y| + sum_j |zb_j B_nj|)
          with y_ref the unrounded float64 value (2^-8 is the bf16 rounding
          bound; the second term covers FP32 accumulation over r <= 256).
  integer inputs: z equal to float32(z_ref), y equal to bf16_round(y_ref).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import oracle

SHRINK_TOL = 1e-5
EXPAND_REL = 2.0 ** -8
EXPAND_ABS = 1e-5


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ig.lib()  # raises if the library is missing


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def shape_of(prob, mode=ig.MODE_DET, split_k=8, path=ig.PATH_AUTO, M=None):
    return ig.make_shape(prob.M if M is None else M, prob.K, prob.N, prob.r,
                         slices=prob.slices, num_adapters=prob.L, split_k=split_k,
                         mode=mode, path=path)


def run_apply(prob, mode=ig.MODE_DET, split_k=8, path=ig.PATH_AUTO, ws=None, z=None,
              y=None, check=True, shape=None):
    """lora_apply on copies of the problem's device tensors; returns (z, y)."""
    sh = shape_of(prob, mode, split_k, path) if shape is None else shape
    if ws is None:
        ws = ig.workspace(sh)
    if z is None:
        z = torch.full((prob.slices, prob.M, prob.r), float("nan"), dtype=torch.float32,
                       device="cuda")
    if y is None:
        y = prob.y.clone()
    ig.lora_apply(sh, prob.x, y, prob.idx, prob.A, prob.B, prob.scale, z, ws)
    if check:
        assert ig.check_status(ws) == 0
    return z, y


def check_shrink(prob_cpu, z_gpu: torch.Tensor, rows=None, exact=False):
    """z_gpu [slices][M][r] (device or host) against the oracle on `rows`."""
    x = bits(prob_cpu.x)
    idx = prob_cpu.idx.cpu().numpy()
    A = bits(prob_cpu.A)
    z = z_gpu.detach().cpu().numpy()
    if rows is not None:
        x, idx, z = x[rows], idx[rows], z[:, rows]
    z_ref, bound = oracle.shrink(x, A, idx, prob_cpu.scale)
    if exact:
        np.testing.assert_array_equal(z, z_ref.astype(np.float32))
        return
    err = np.abs(z.astype(np.float64) - z_ref)
    tol = SHRINK_TOL * bound
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"shrink: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={z[tuple(i)]!r} ref={z_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")


def check_expand(prob_cpu, z_gpu: torch.Tensor, y_gpu: torch.Tensor, rows=None, exact=False,
                 y_in=None):
    """Stage-wise: the oracle expands the GPU's own Z."""
    B = bits(prob_cpu.B)
    idx = prob_cpu.idx.cpu().numpy()
    y0 = bits(prob_cpu.y if y_in is None else y_in)
    z = z_gpu.detach().cpu().numpy().astype(np.float32)
    y = bits(y_gpu)
    if rows is not None:
        idx, y0, z, y = idx[rows], y0[rows], z[:, rows], y[rows]
    y_exact, bound, y_rne = oracle.expand(z, B, idx, y0)
    if exact:
        np.testing.assert_array_equal(y, y_rne)
        return
    yv = oracle.bf16_to_f64(y)
    err = np.abs(yv - y_exact)
    tol = EXPAND_REL * np.abs(y_exact) + EXPAND_ABS * bound
    bad = ~(err <= tol)
    none = idx < 0
    if none.any():
        np.testing.assert_array_equal(y[none], y0[none])
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"expand: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
            f"gpu={yv[tuple(i)]!r} ref={y_exact[tuple(i)]!r} bound={bound[tuple(i)]!r}")

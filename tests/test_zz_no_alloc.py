"""lora_shrink_noalloc: the shrink for callers that cannot allocate device
memory (no workspace argument; the scratch is a fixed 4 MiB array inside the
library). Its output must match lora_shrink's within the shrink tolerance, on
two calls in a row (the second sees whatever the first left in the shared
array). The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import oracle
import synth
from helpers import SHRINK_TOL, bits, need_gpu, shape_of

pytestmark = pytest.mark.gpu


def _existing(p, sh):
    ws = ig.workspace(sh)
    z = torch.full((p.slices, p.M, p.r), float("nan"), dtype=torch.float32, device="cuda")
    ig.lora_shrink(sh, p.x, p.A, p.idx, p.scale, z, ws)
    assert ig.check_status(ws) == 0
    return z


def _noalloc(p, sh):
    z = torch.full((p.slices, p.M, p.r), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = ig.lib().lora_shrink_noalloc(ctypes.byref(sh), p.x.data_ptr(), p.A.data_ptr(),
                                      p.idx.data_ptr(), ctypes.c_float(p.scale),
                                      z.data_ptr(), stream)
    assert rc == 0, ig.status_string(rc)
    torch.cuda.synchronize()
    return z


def _close(p, z_new, z_old):
    _, bound = oracle.shrink(bits(p.x), bits(p.A), p.idx.cpu().numpy(), p.scale)
    a = z_new.cpu().numpy().astype(np.float64)
    b = z_old.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(a - b) <= SHRINK_TOL * bound)


def test_noalloc_matches_lora_shrink_two_calls():
    need_gpu()
    p1 = synth.make_problem(256, 4096, 4096, 16, L=8, seed=1257, none_frac=0.05, device="cuda")
    p2 = synth.make_problem(77, 4096, 512, 32, slices=3, L=5, seed=1258, device="cuda")
    for p in (p1, p2):
        sh = shape_of(p, ig.MODE_DET, 8)
        _close(p, _noalloc(p, sh), _existing(p, sh))


def test_noalloc_rejects_oversized_shape():
    need_gpu()
    sh = ig.make_shape(8192, 28672, 8192, 128, num_adapters=64, split_k=16)
    assert ig.workspace_bytes(sh) > (4 << 20)
    rc = ig.lib().lora_shrink_noalloc(ctypes.byref(sh), 0x10000, 0x10000, 0x10000,
                                      ctypes.c_float(1.0), 0x10000, None)
    assert rc == -4

"""lora_shrink_noalloc: the shrink for callers that cannot allocate device
memory (no workspace argument; the scratch is a fixed 4 MiB array inside the
library).

It runs the same plan on the same kernels as lora_shrink, so its z must be
bit for bit the same as lora_shrink's on the same inputs; it is also checked
against the FP64 oracle within the shrink tolerance. The calls come in a row,
a shape with a large scratch footprint before a mma_p one, then both again,
so that anything a call leaves in the shared array (token map, counters,
partials) would show in the next one. The file is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

import invariant_gemm_gb300 as ig
import synth
from helpers import check_shrink, need_gpu, shape_of

pytestmark = pytest.mark.gpu


def _existing(p, sh):
    ws = ig.workspace(sh)
    z = torch.full((p.slices, p.M, p.r), float("nan"), dtype=torch.float32, device="cuda")
    ig.lora_shrink(sh, p.x, p.A, p.idx, p.scale, z, ws)
    assert ig.check_status(ws) == 0
    return z


def _call(sh, x, A, idx, scale, z):
    stream = torch.cuda.current_stream().cuda_stream
    return ig.lib().lora_shrink_noalloc(ctypes.byref(sh), x, A, idx, ctypes.c_float(scale), z,
                                        stream)


def _noalloc(p, sh):
    z = torch.full((p.slices, p.M, p.r), float("nan"), dtype=torch.float32, device="cuda")
    rc = _call(sh, p.x.data_ptr(), p.A.data_ptr(), p.idx.data_ptr(), p.scale, z.data_ptr())
    assert rc == 0, ig.status_string(rc)
    torch.cuda.synchronize()
    return z


def _same_bits(a, b):
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_noalloc_bitwise_equals_lora_shrink_in_a_row():
    need_gpu()
    # warp tensor-core path (r = 16), tokens without adapter among them
    warp_p = synth.make_problem(256, 4096, 4096, 16, L=8, seed=1257, none_frac=0.05,
                                device="cuda")
    # tcgen05 path (r = 32, three stacked slices), ragged tile, index -1 rows
    mma_p = synth.make_problem(77, 4096, 512, 32, slices=3, L=5, seed=1258, none_frac=0.1,
                               device="cuda")
    assert (warp_p.idx < 0).any() and (mma_p.idx < 0).any()
    sh_warp, sh_mma = shape_of(warp_p, ig.MODE_DET, 8), shape_of(mma_p, ig.MODE_DET, 8)
    assert ig.plan_query(sh_warp)["path"] == ig.PATH_WARP
    assert ig.plan_query(sh_mma)["path"] == ig.PATH_MMA
    # the call with the larger scratch footprint first (the 128-row tcgen05
    # tiles need more than the 8-row warp-path tiles), then the smaller one,
    # then both again
    runs = sorted(((warp_p, sh_warp), (mma_p, sh_mma)),
                  key=lambda c: -ig.workspace_bytes(c[1]))
    assert ig.workspace_bytes(runs[0][1]) > ig.workspace_bytes(runs[1][1])
    ref = {id(warp_p): _existing(warp_p, sh_warp), id(mma_p): _existing(mma_p, sh_mma)}
    for p, sh in runs + runs:
        z = _noalloc(p, sh)
        _same_bits(z, ref[id(p)])
        check_shrink(p, z)
        zc = z.cpu()
        assert torch.all(zc[:, p.idx.cpu() < 0] == 0)


def test_noalloc_atomic_and_unsplit_match_oracle():
    need_gpu()
    p = synth.make_problem(64, 2048, 512, 16, L=4, seed=1259, none_frac=0.1, device="cuda")
    for mode in (ig.MODE_UNSPLIT, ig.MODE_DET, ig.MODE_ATOMIC):
        sh = shape_of(p, mode, 8)
        z = _noalloc(p, sh)
        check_shrink(p, z)
        if mode != ig.MODE_ATOMIC:
            _same_bits(z, _existing(p, sh))


def test_noalloc_rejects_oversized_shape():
    need_gpu()
    sh = ig.make_shape(8192, 28672, 8192, 128, num_adapters=64, split_k=16)
    assert ig.workspace_bytes(sh) > (4 << 20)
    rc = ig.lib().lora_shrink_noalloc(ctypes.byref(sh), 0x10000, 0x10000, 0x10000,
                                      ctypes.c_float(1.0), 0x10000, None)
    assert rc == -4


def test_noalloc_rejects_bad_pointers_before_enqueueing():
    need_gpu()
    p = synth.make_problem(16, 512, 512, 16, L=2, seed=1260, device="cuda")
    sh = shape_of(p, ig.MODE_DET, 8)
    z = torch.zeros((p.slices, p.M, p.r + 4), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    # misaligned z, null x: rejected on the host, z untouched
    assert _call(sh, p.x.data_ptr(), p.A.data_ptr(), p.idx.data_ptr(), 1.0,
                 z.data_ptr() + 4) == -3
    assert _call(sh, 0, p.A.data_ptr(), p.idx.data_ptr(), 1.0, z.data_ptr()) == -1
    assert _call(sh, p.x.data_ptr(), p.A.data_ptr(), 0, 1.0, z.data_ptr()) == -1
    torch.cuda.synchronize()
    assert torch.count_nonzero(z) == 0
    # and the next valid call is still right
    z2 = _noalloc(p, sh)
    _same_bits(z2, _existing(p, sh))


def test_noalloc_needs_only_the_shrinks_share():
    """ig_workspace_bytes also counts the expand's Z operand that lora_apply
    writes on the tcgen05 path (three bf16 parts per value with FP32 Z); the
    shrink alone never touches it, so a shape whose full workspace is past
    4 MiB but whose shrink share fits still runs here."""
    need_gpu()
    p = synth.make_problem(2048, 1024, 512, 64, slices=3, L=16, seed=1261, none_frac=0.05,
                           device="cuda")
    sh = ig.make_shape(p.M, p.K, p.N, p.r, slices=3, num_adapters=16, split_k=8,
                       mode=ig.MODE_UNSPLIT, flags=ig.FLAG_Z_FP32)
    assert ig.plan_query(sh)["path"] == ig.PATH_MMA
    assert ig.workspace_bytes(sh) > (4 << 20)
    z = _noalloc(p, sh)
    _same_bits(z, _existing(p, sh))
    check_shrink(p, z)

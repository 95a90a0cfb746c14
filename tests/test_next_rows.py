"""The extensions past the core path:

* IG_MODE_DET_TREE: the pages' earlier deterministic design (sec. 4.3):
  partials combined by a second kernel with a fixed pairwise tree;
* the Split-K sweep and a batch-size-dependent Split-K choice like vLLM's
  (sec. 4: S = 64 for M < 128, else 8), shown to break batch invariance;
* IG_FLAG_Z_FP32: the expand reads Z in FP32 (no bf16 boundary, sec. 6.2).
"""
import os

import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import oracle
import synth
from helpers import (EXPAND_ABS, EXPAND_REL, bits, check_expand, check_shrink, need_gpu,
                     run_apply, shape_of)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


# ---------------------------------------------------------------- DET_TREE

@pytest.mark.parametrize("K,S,r", [(4096, 8, 16), (4096, 2, 16), (3072, 3, 16), (8192, 16, 8),
                                   (4096, 8, 64), (11008, 8, 64)])
def test_tree_mode_parity(K, S, r):
    p = synth.make_problem(150, K, 512, r, slices=2, L=4, seed=K + S, none_frac=0.1,
                           device="cuda")
    z, y = run_apply(p, mode=ig.MODE_DET_TREE, split_k=S)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)


@pytest.mark.parametrize("r", [16, 64])
def test_tree_mode_replay_and_batch_invariance(r):
    K, N, L = 4096, 512, 8
    base = synth.make_problem(32, K, N, r, L=L, seed=r, device="cuda")
    sh0 = ig.make_shape(300, K, N, r, num_adapters=L, mode=ig.MODE_DET_TREE)
    ws = ig.workspace(sh0)
    ref = None
    for b in list(range(1, 40)) + [64, 100, 173, 256, 300]:
        x, y, idx, pos = synth.probe_batch(base.x, base.y, base.idx, b, L, seed=300 + b,
                                           device="cuda")
        sh = ig.make_shape(b, K, N, r, num_adapters=L, mode=ig.MODE_DET_TREE)
        z = torch.empty((1, b, r), dtype=torch.float32, device="cuda")
        for _ in range(3):  # replays
            yy = y.clone()
            ig.lora_apply(sh, x, yy, idx, base.A, base.B, base.scale, z, ws)
            pz, py = z[0, pos].view(torch.int32).clone(), yy[pos].view(torch.int16).clone()
            if ref is None or pz.shape[0] > ref[0].shape[0]:
                if ref is not None:
                    assert torch.equal(pz[:ref[0].shape[0]], ref[0])
                    assert torch.equal(py[:ref[1].shape[0]], ref[1])
                ref = (pz, py)
            else:
                assert torch.equal(pz, ref[0][:pz.shape[0]]), b
                assert torch.equal(py, ref[1][:py.shape[0]]), b
    assert ig.check_status(ws) == 0


def test_tree_order_probe():
    """Partials [a, 1, 0, 0, -a, 1, 0, 0], a = 2^100: the pairwise tree
    ((a+1)+(0+0)) + ((-a+1)+(0+0)) absorbs each 1 into +-a before the halves
    meet, as in the pages' a + (b + c) = 0 (Eq. 4); the in-kernel
    increasing-order combine gives (a + b) + c = 1."""
    with open(os.path.join(GOLDEN, "eq4_nonassociativity.txt")) as f:
        row = [l.split() for l in f if l.strip() and not l.startswith("#")][0]
    left, right = float(row[3]), float(row[4])
    S, Ks = 8, 256
    K = S * Ks
    a = 2.0 ** 100
    parts = [a, 1.0, 0.0, 0.0, -a, 1.0, 0.0, 0.0]
    x = torch.zeros((1, K))
    A = torch.zeros((1, 1, 8, K))
    for s in range(S):
        x[0, s * Ks] = 1.0
        A[0, 0, :, s * Ks] = parts[s]
    p = synth.Problem(M=1, K=K, N=8, r=8, slices=1, L=1, scale=1.0,
                      x=x.to(torch.bfloat16).cuda(), A=A.to(torch.bfloat16).cuda(),
                      B=torch.zeros((1, 1, 8, 8), dtype=torch.bfloat16, device="cuda"),
                      y=torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda"),
                      idx=torch.zeros(1, dtype=torch.int32, device="cuda"))
    z_tree, _ = run_apply(p, mode=ig.MODE_DET_TREE, split_k=S)
    z_det, _ = run_apply(p, mode=ig.MODE_DET, split_k=S)
    assert torch.all(z_tree == right)
    assert torch.all(z_det == left)


# ------------------------------------------------ Split-K sweep, S chosen by M

def vllm_like_split(M):
    """Split-K picked from the batch size (sec. 4: 64 below 128 rows, else 8)."""
    return 64 if M < 128 else 8


def test_batch_dependent_split_breaks_invariance():
    """The same 16 rows in a batch of 64 and in a batch of 256: with S fixed
    by the plan their bits agree; with S picked from M (64 vs 8) the
    partition sums regroup and some bits differ. That is why the plan never
    looks at M."""
    K, N, r, L = 4096, 512, 16, 4
    base = synth.make_problem(16, K, N, r, L=L, seed=11, device="cuda")

    def probe(b, S):
        x, y, idx, pos = synth.probe_batch(base.x, base.y, base.idx, b, L, seed=b,
                                           device="cuda")
        sh = ig.make_shape(b, K, N, r, num_adapters=L, split_k=S)
        z = torch.empty((1, b, r), dtype=torch.float32, device="cuda")
        ig.lora_apply(sh, x, y, idx, base.A, base.B, base.scale, z, ig.workspace(sh))
        return z[0, pos].view(torch.int32).clone()

    assert torch.equal(probe(64, 8), probe(256, 8))
    assert not torch.equal(probe(64, vllm_like_split(64)), probe(256, vllm_like_split(256)))


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16, 64])
@pytest.mark.parametrize("mode", [ig.MODE_DET, ig.MODE_DET_TREE, ig.MODE_ATOMIC],
                         ids=["det", "tree", "atomic"])
def test_split_sweep_all_modes(S, mode):
    if mode == ig.MODE_ATOMIC and S == 1:
        pytest.skip("nothing to add atomically")
    p = synth.make_problem(64, 4096, 512, 16, L=4, seed=S, device="cuda")
    z, y = run_apply(p, mode=mode, split_k=S)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)


# ------------------------------------------------------------- FP32 Z input

def check_expand_fp32(prob, z_gpu, y_gpu):
    B = bits(prob.B.cpu())
    idx = prob.idx.cpu().numpy()
    y0 = bits(prob.y.cpu())
    zc = z_gpu.cpu().numpy()
    y_exact, bound, _ = oracle.expand(zc, B, idx, y0, round_z=False)
    yv = oracle.bf16_to_f64(bits(y_gpu))
    err = np.abs(yv - y_exact)
    tol = EXPAND_REL * np.abs(y_exact) + EXPAND_ABS * bound
    assert np.all(err <= tol), float(np.max(err - tol))


@pytest.mark.parametrize("r,path", [(16, ig.PATH_WARP), (64, ig.PATH_MMA), (32, ig.PATH_WARP),
                                    (24, ig.PATH_WARP), (192, ig.PATH_MMA), (80, ig.PATH_MMA),
                                    (256, ig.PATH_AUTO)])
def test_fp32_z_expand(r, path):
    p = synth.make_problem(120, 4096, 520, r, slices=2, L=3, seed=r, none_frac=0.1,
                           device="cuda")
    sh = ig.make_shape(p.M, p.K, p.N, r, slices=2, num_adapters=3, path=path,
                       flags=ig.FLAG_Z_FP32)
    z, y = run_apply(p, shape=sh)
    check_shrink(p.to("cpu"), z)
    check_expand_fp32(p, z, y)
    # the bf16 boundary really is gone: rounding Z first gives other bits somewhere
    sh2 = ig.make_shape(p.M, p.K, p.N, r, slices=2, num_adapters=3, path=path)
    _, y2 = run_apply(p, shape=sh2)
    assert not torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_fp32_z_fused_equals_two_kernel():
    p = synth.make_problem(77, 4096, 1024, 16, L=4, seed=3, device="cuda")
    outs = []
    for fl in (ig.FLAG_Z_FP32, ig.FLAG_Z_FP32 | ig.FLAG_UNFUSED):
        sh = ig.make_shape(p.M, p.K, p.N, 16, num_adapters=4, flags=fl)
        outs.append(run_apply(p, shape=sh))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))
    check_expand_fp32(p, outs[0][0], outs[0][1])

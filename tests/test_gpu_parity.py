"""CUDA path against the FP64 oracle, element by element, through the C ABI.

Shapes follow the workloads of "Reproducible LoRA Inference Through
Deterministic Split-K Reduction" (decode and prefill, ranks 16-128, fused QKV
slices, Split-K 8) and cover several tiles, ragged tails (rows, K partitions
that are not whole k-blocks, output columns), tokens without an adapter, and
the largest sizes on sampled rows.
"""
import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import oracle
import synth
from helpers import (bits, check_expand, check_shrink, need_gpu, run_apply, shape_of)

pytestmark = pytest.mark.gpu

MODES = [ig.MODE_DET, ig.MODE_ATOMIC, ig.MODE_UNSPLIT]
MODE_ID = {ig.MODE_DET: "det", ig.MODE_ATOMIC: "atomic", ig.MODE_UNSPLIT: "unsplit"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def cpu(prob):
    return prob.to("cpu")


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
def test_single_adapter_small_normal(mode):
    p = synth.make_problem(4, 512, 512, 8, L=1, seed=1000, device="cuda")
    z, y = run_apply(p, mode=mode)
    check_shrink(cpu(p), z)
    check_expand(cpu(p), z, y)


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
def test_single_adapter_small_integers_bit_exact(mode):
    p = synth.make_problem(4, 512, 512, 8, L=1, seed=1000, dist="int", device="cuda")
    z, y = run_apply(p, mode=mode)
    check_shrink(cpu(p), z, exact=True)
    check_expand(cpu(p), z, y, exact=True)


@pytest.mark.parametrize("M", [1, 8, 32, 128, 256])
@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
def test_decode_7b(M, mode):
    p = synth.make_problem(M, 4096, 4096, 16, L=8, seed=1001 + M, device="cuda")
    z, y = run_apply(p, mode=mode)
    check_shrink(cpu(p), z)
    check_expand(cpu(p), z, y)


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
def test_decode_7b_integers_bit_exact(mode):
    # |sum| <= 4096 * 16 < 2^24 and every expand sum < 2^24: all orders exact
    p = synth.make_problem(256, 4096, 4096, 16, L=8, seed=77, dist="int", device="cuda")
    z, y = run_apply(p, mode=mode)
    check_shrink(cpu(p), z, exact=True)
    check_expand(cpu(p), z, y, exact=True)


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
def test_ragged_everything(mode):
    # K/S = 1376 (5 whole k-blocks + 96), r = 24 (three 8-column blocks),
    # N = 264 (a partial column tile), 3 slices, 5 adapters, 20% no-adapter rows
    p = synth.make_problem(300, 11008, 264, 24, slices=3, L=5, seed=5, none_frac=0.2,
                           device="cuda")
    z, y = run_apply(p, mode=mode)
    check_shrink(cpu(p), z)
    check_expand(cpu(p), z, y)
    zc = z.cpu().numpy()
    none = p.idx.cpu().numpy() < 0
    assert none.any() and np.all(zc[:, none] == 0)


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16, 64])
def test_split_counts(S):
    p = synth.make_problem(40, 4096, 512, 16, L=3, seed=60 + S, device="cuda")
    z, y = run_apply(p, mode=ig.MODE_DET, split_k=S)
    check_shrink(cpu(p), z)
    check_expand(cpu(p), z, y)


def _sample_rows(M, n, seed):
    g = np.random.default_rng(seed)
    rows = set(g.choice(M, size=min(M, n), replace=False).tolist())
    rows.update({0, M - 1})
    return np.array(sorted(rows))


@pytest.mark.parametrize("which", ["qkv", "down"])
@pytest.mark.parametrize("mode", [ig.MODE_DET, ig.MODE_UNSPLIT], ids=MODE_ID.get)
def test_prefill_sampled_rows(which, mode):
    if which == "qkv":
        p = synth.make_problem(4096, 4096, 4096, 64, slices=3, L=16, ids="segments",
                               segment=256, seed=1002, device="cuda")
    else:
        p = synth.make_problem(4096, 11008, 4096, 64, slices=1, L=16, ids="segments",
                               segment=256, seed=1012, device="cuda")
    z, y = run_apply(p, mode=mode)
    rows = _sample_rows(p.M, 48, 3)
    rows = np.union1d(rows, [255, 256, 257, 4095])
    check_shrink(cpu(p), z, rows=rows)
    check_expand(cpu(p), z, y, rows=rows)


# (K, M, S) of the large-model workload (K = 8192 hidden, K = 28672 down-
# projection; M in {1, 16, 256, 2048, 8192}; Split-K in {1, 4, 8, 16}): every
# M at K = 8192 and at K = 28672, every Split-K at each K.
LARGE = [(8192, 1, 8), (8192, 1, 16), (8192, 16, 4), (8192, 16, 16), (8192, 256, 8),
         (8192, 2048, 4), (8192, 8192, 8), (8192, 8192, 16), (8192, 8192, 1),
         (28672, 1, 4), (28672, 16, 16), (28672, 256, 1), (28672, 2048, 8),
         (28672, 8192, 16), (28672, 8192, 8)]


def _sub_problem(p, rows):
    """The sampled rows of a device problem on the host, with only the
    adapters those rows use (renumbered), so that the oracle stays small."""
    rt = torch.as_tensor(rows, device="cuda")
    idx = p.idx[rt].cpu()
    used = torch.unique(idx[idx >= 0]).long()
    remap = torch.full((p.L,), -1, dtype=torch.int32)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32)
    ud = used.to("cuda")
    return synth.Problem(M=len(rows), K=p.K, N=p.N, r=p.r, slices=p.slices,
                         L=max(1, used.numel()), scale=p.scale, x=p.x[rt].cpu(),
                         A=p.A[ud].cpu(), B=p.B[ud].cpu(), y=p.y[rt].cpu(),
                         idx=torch.where(idx >= 0, remap[idx.clamp(min=0).long()], idx)), rt


@pytest.mark.parametrize("K,M,S", LARGE)
@pytest.mark.parametrize("mode", [ig.MODE_DET, ig.MODE_ATOMIC], ids=MODE_ID.get)
def test_large_model_sampled_rows(K, M, S, mode):
    if S == 1 and mode == ig.MODE_ATOMIC:
        pytest.skip("Split-K = 1 has nothing to add atomically")
    p = synth.make_problem(M, K, 8192, 128, L=64, ids="zipf", seed=1004, device="cuda")
    z, y = run_apply(p, mode=mode, split_k=S)
    sub, rt = _sub_problem(p, _sample_rows(M, 24, K + M))
    check_shrink(sub, z[:, rt])
    check_expand(sub, z[:, rt], y[rt])


@pytest.mark.parametrize("variant", ["det_cluster", "det_counter", "atomic", "unsplit"])
def test_large_model_integers_bit_exact(variant):
    """K = 28672, r = 128 on tcgen05 with small-integer x, A, B, y: every
    partial sum of the shrink is an integer below 28672 * 16 < 2^24, so every
    order gives the exact value and z must equal the oracle's bit for bit;
    the expand's sums are integers too (bf16(z) has at most 8 significant
    bits), and where the oracle's sum of magnitudes stays below 2^24 y must
    equal bf16(y_exact) bit for bit."""
    mode, flags = {"det_cluster": (ig.MODE_DET, 0), "det_counter": (ig.MODE_DET, ig.FLAG_UNFUSED),
                   "atomic": (ig.MODE_ATOMIC, 0), "unsplit": (ig.MODE_UNSPLIT, 0)}[variant]
    p = synth.make_problem(512, 28672, 8192, 128, L=64, ids="zipf", dist="int", seed=1014,
                           device="cuda")
    sh = ig.make_shape(p.M, p.K, p.N, p.r, num_adapters=p.L, split_k=8, mode=mode, flags=flags)
    assert ig.plan_query(sh)["path"] == ig.PATH_MMA
    z, y = run_apply(p, shape=sh)
    sub, rt = _sub_problem(p, _sample_rows(p.M, 40, 28672))
    check_shrink(sub, z[:, rt], exact=True)
    _, bound, _ = oracle.expand(z[:, rt].cpu().numpy(), bits(sub.B), sub.idx.numpy(),
                                bits(sub.y))
    assert float(bound.max()) < 2.0 ** 24
    check_expand(sub, z[:, rt], y[rt], exact=True)


def test_zero_tokens():
    p = synth.make_problem(0, 512, 512, 8, L=1, seed=1, device="cuda")
    z, y = run_apply(p)
    assert z.numel() == 0 and y.numel() == 0


def test_max_adapters_and_all_none():
    p = synth.make_problem(700, 512, 256, 16, L=1023, seed=8, device="cuda")
    z, y = run_apply(p)
    check_shrink(cpu(p), z)
    check_expand(cpu(p), z, y)
    p.idx.fill_(-1)
    z, y = run_apply(p)
    assert torch.all(z == 0)
    assert torch.equal(y, p.y)


@pytest.mark.parametrize("mode", MODES + [ig.MODE_DET_TREE], ids=lambda m: MODE_ID.get(m, "tree"))
@pytest.mark.parametrize("r", [8, 16, 24])
def test_fma_path_parity(r, mode):
    """IG_PATH_FMA (CUDA-core FP32 FMA, warp-shuffle reduction): every mode,
    against the oracle; small integers bit-exact."""
    p = synth.make_problem(150, 11008, 264, r, slices=2, L=5, seed=400 + r, none_frac=0.2,
                           device="cuda")
    z, y = run_apply(p, mode=mode, path=ig.PATH_FMA)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)
    pi = synth.make_problem(40, 4096, 512, r, L=3, seed=500 + r, dist="int", device="cuda")
    z, y = run_apply(pi, mode=mode, path=ig.PATH_FMA)
    check_shrink(pi.to("cpu"), z, exact=True)
    check_expand(pi.to("cpu"), z, y, exact=True)


def test_fma_and_warp_paths_differ_only_within_tolerance():
    """The two small-rank paths sum each partition in a different order
    (FMA chains and a butterfly against tensor-core MMAs); the plan keeps
    them apart in the determinism key, and both meet the oracle's bound."""
    p = synth.make_problem(64, 4096, 1024, 16, L=4, seed=77, device="cuda")
    keys = []
    for path in (ig.PATH_WARP, ig.PATH_FMA):
        sh = ig.make_shape(p.M, p.K, p.N, 16, num_adapters=4, path=path)
        keys.append(ig.plan_query(sh)["determinism_key"])
        z, y = run_apply(p, shape=sh)
        check_shrink(p.to("cpu"), z)
        check_expand(p.to("cpu"), z, y)
    assert keys[0] != keys[1]

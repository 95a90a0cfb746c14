"""Seeded random shapes through lora_apply against the FP64 oracle: every mode
and path on ragged sizes (M, K, N, r, slices, adapters, Split-K, share of
tokens without an adapter), with and without the static-weights and
input-ready flags (copies and, in the fused decode kernel, the shrink issued
before the dependency wait), so that the hand-picked cases of the other
files are not the only ones that hold. Deterministic modes are also replayed
once and must give the same bits."""
import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import synth
from helpers import check_expand, check_shrink, need_gpu, run_apply

pytestmark = pytest.mark.gpu

MODES = [ig.MODE_DET, ig.MODE_ATOMIC, ig.MODE_UNSPLIT, ig.MODE_DET_TREE]


def draw(i):
    """Case i: a valid shape and plan, reproducible from i alone."""
    rng = np.random.default_rng(9100 + i)
    path = [ig.PATH_AUTO, ig.PATH_WARP, ig.PATH_FMA, ig.PATH_MMA][i % 4]
    mode = MODES[(i // 4) % 4]
    if path == ig.PATH_MMA:
        r = int(rng.choice([16, 32, 48, 64, 128]))
    else:
        r = int(rng.choice([8, 16, 24, 32, 48]))
    S = 1 if mode == ig.MODE_UNSPLIT else int(rng.choice([1, 2, 3, 4, 8, 16]))
    step = 16 if path == ig.PATH_MMA else 8          # K/S granularity of the path
    K = S * step * int(rng.integers(1, max(2, 2048 // (S * step)) + 1))
    N = 8 * int(rng.integers(1, 130))
    M = int(rng.integers(0, 260))
    slices = int(rng.integers(1, 4))
    L = int(rng.integers(1, 11))
    none_frac = float(rng.choice([0.0, 0.0, 0.15, 0.5]))
    ids = str(rng.choice(["uniform", "segments", "zipf"]))
    flags = [0, ig.FLAG_STATIC_WEIGHTS, ig.FLAG_STATIC_WEIGHTS | ig.FLAG_INPUT_READY][i % 3]
    return dict(M=M, K=K, N=N, r=r, slices=slices, L=L, S=S, mode=mode, path=path,
                none_frac=none_frac, ids=ids, seed=9100 + i, flags=flags)


CASES = [draw(i) for i in range(36)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M%d_K%d_N%d_r%d_sl%d_L%d_S%d_m%d_p%d_f%d" % (
    c["M"], c["K"], c["N"], c["r"], c["slices"], c["L"], c["S"], c["mode"], c["path"],
    c["flags"]))
def test_random_shapes_against_oracle(case):
    c = case
    L = c["L"] if c["ids"] != "zipf" else max(c["L"], 2)
    p = synth.make_problem(c["M"], c["K"], c["N"], c["r"], slices=c["slices"], L=L,
                           ids=c["ids"], segment=64, seed=c["seed"],
                           none_frac=c["none_frac"], device="cuda")
    sh = ig.make_shape(c["M"], c["K"], c["N"], c["r"], slices=c["slices"], num_adapters=L,
                       split_k=c["S"], mode=c["mode"], path=c["path"], flags=c["flags"])
    z, y = run_apply(p, shape=sh)
    if c["M"] == 0:
        return
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)
    if c["mode"] != ig.MODE_ATOMIC:
        z2, y2 = run_apply(p, shape=sh)
        assert torch.equal(z.view(torch.int32), z2.view(torch.int32))
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))

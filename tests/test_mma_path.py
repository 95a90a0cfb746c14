"""The tcgen05 tensor-core path (ranks of 32 and more by default, or forced
with PATH_MMA) against the FP64 oracle: bit-exact on small-integer inputs
(products exact, sums below 2^24), within tolerance on normal inputs, every
mode, ragged partitions (K/S not a multiple of 64), partial tiles, no-adapter
rows, several slices, and the plan's path choice."""
import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import synth
from helpers import check_expand, check_shrink, need_gpu, run_apply

pytestmark = pytest.mark.gpu

MODES = [ig.MODE_DET, ig.MODE_ATOMIC, ig.MODE_UNSPLIT]
MODE_ID = {ig.MODE_DET: "det", ig.MODE_ATOMIC: "atomic", ig.MODE_UNSPLIT: "unsplit"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def test_plan_picks_tensor_cores_for_large_ranks():
    for r, want in [(16, ig.PATH_WARP), (24, ig.PATH_WARP), (32, ig.PATH_MMA), (64, ig.PATH_MMA),
                    (128, ig.PATH_MMA)]:
        p = ig.plan_query(ig.make_shape(256, 4096, 4096, r, num_adapters=8))
        assert p["path"] == want, r
        if want == ig.PATH_MMA:
            assert p["shrink_bm"] == 128 and p["apply_kernels"] == 2


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
def test_mma_small_integers_bit_exact(mode):
    # |x A| sums <= 4096 * 16 < 2^24; expand sums < 2^24: every order is exact
    p = synth.make_problem(300, 4096, 512, 64, slices=1, L=5, seed=31, dist="int",
                           device="cuda")
    z, y = run_apply(p, mode=mode, path=ig.PATH_MMA)
    check_shrink(p.to("cpu"), z, exact=True)
    check_expand(p.to("cpu"), z, y, exact=True)


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
@pytest.mark.parametrize("r", [32, 64, 128])
def test_mma_normal_inputs(mode, r):
    p = synth.make_problem(200, 2048, 768, r, slices=2, L=3, seed=r, none_frac=0.1,
                           device="cuda")
    z, y = run_apply(p, mode=mode, path=ig.PATH_MMA)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
@pytest.mark.parametrize("r", [16, 48, 64])
def test_mma_ragged_partition_and_small_ranks(mode, r):
    # K/S = 1376: the last k-step of each partition has 32 of 64 columns;
    # r = 16 and 48 are not multiples of one 32-column accumulator read
    p = synth.make_problem(150, 11008, 264, r, L=4, seed=5 + r, device="cuda")
    z, y = run_apply(p, mode=mode, path=ig.PATH_MMA)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)


def test_mma_decode_rows_in_big_tiles():
    # a few tokens per adapter: tiles of 128 rows mostly empty
    for M in (1, 5, 33):
        p = synth.make_problem(M, 8192, 1024, 128, L=4, seed=M, device="cuda")
        z, y = run_apply(p, mode=ig.MODE_DET, split_k=16, path=ig.PATH_MMA)
        check_shrink(p.to("cpu"), z)
        check_expand(p.to("cpu"), z, y)


def test_mma_replay_bitwise():
    p = synth.make_problem(512, 4096, 1024, 64, L=8, seed=9, device="cuda")
    z0, y0 = run_apply(p, mode=ig.MODE_DET)
    for _ in range(50):
        z, y = run_apply(p, mode=ig.MODE_DET)
        assert torch.equal(z.view(torch.int32), z0.view(torch.int32))
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


@pytest.mark.parametrize("mode", MODES, ids=MODE_ID.get)
@pytest.mark.parametrize("r", [64, 128])
def test_mma_contiguous_tiles_with_overhang(mode, r):
    """Tiles whose tokens are consecutive are copied as one 128-row box; the
    last tile of a single-adapter batch of 300 rows reaches past row M (its
    rows go back by row stores; at r = 128 the expand runs two warpgroups)."""
    p = synth.make_problem(300, 4096, 520, r, slices=2, L=1, ids="single", seed=77,
                           device="cuda")
    z, y = run_apply(p, mode=mode, path=ig.PATH_MMA)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)
    # segments of 256 tokens per adapter (the prefill layout) with a ragged end
    p = synth.make_problem(700, 4096, 512, r, L=3, ids="segments", segment=256, seed=78,
                           device="cuda")
    z, y = run_apply(p, mode=mode, path=ig.PATH_MMA)
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)


@pytest.mark.parametrize("r,K,S", [(32, 2048, 8), (64, 11008, 8), (128, 8192, 16), (64, 4096, 4)])
def test_mma_cluster_combine_bitwise_equals_counter(r, K, S):
    """The deterministic tcgen05 shrink combines inside a thread-block cluster
    where it can; IG_FLAG_UNFUSED forces the counter protocol (Algorithm 1).
    Same order of the partition sum, so the same bits for z and y."""
    p = synth.make_problem(300, K, 520, r, slices=2, L=5, seed=r + S, none_frac=0.1,
                           device="cuda")
    outs = []
    for flags in (0, ig.FLAG_UNFUSED):
        sh = ig.make_shape(p.M, K, p.N, r, slices=2, num_adapters=5, split_k=S,
                           mode=ig.MODE_DET, path=ig.PATH_MMA, flags=flags)
        outs.append(run_apply(p, shape=sh))
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))
    check_shrink(p.to("cpu"), outs[0][0])
    check_expand(p.to("cpu"), outs[0][0], outs[0][1])


@pytest.mark.parametrize("mode,flags", [(ig.MODE_DET, 0), (ig.MODE_DET, ig.FLAG_UNFUSED),
                                        (ig.MODE_UNSPLIT, 0), (ig.MODE_DET, ig.FLAG_Z_FP32)],
                         ids=["det_cluster", "det_counter", "unsplit", "det_z_fp32"])
@pytest.mark.parametrize("r,slices", [(32, 3), (48, 2), (128, 1), (192, 1)])
def test_apply_z_operand_equals_separate_calls(mode, flags, r, slices):
    """Inside lora_apply the tcgen05 shrink also writes the expand's Z operand
    (bf16 tiles in the tensor cores' layout) and the expand copies it instead
    of building it from z; lora_shrink then lora_expand build it from z. Same
    rounding of the same z values, so the same bits, on scattered and
    consecutive tiles, partly filled tiles and ranks that end inside an
    atom (r = 48, 192)."""
    for ids, seed in (("uniform", 11), ("segments", 12)):
        p = synth.make_problem(333, 4096, 520, r, slices=slices, L=5, ids=ids, segment=96,
                               seed=seed + r, none_frac=0.1, device="cuda")
        sh = ig.make_shape(p.M, p.K, p.N, r, slices=slices, num_adapters=5, split_k=8,
                           mode=mode, path=ig.PATH_MMA, flags=flags)
        z1, y1 = run_apply(p, shape=sh)
        ws = ig.workspace(sh)
        z2 = torch.full_like(z1, float("nan"))
        y2 = p.y.clone()
        ig.lora_shrink(sh, p.x, p.A, p.idx, p.scale, z2, ws)
        ig.lora_expand(sh, z2, p.B, p.idx, y2, ws)
        assert ig.check_status(ws) == 0
        assert torch.equal(z1.view(torch.int32), z2.view(torch.int32))
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
        if not flags & ig.FLAG_Z_FP32:
            check_expand(p.to("cpu"), z1, y1)

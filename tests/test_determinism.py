"""Determinism invariants of the CUDA path, and the device-side error paths.

"Reproducible LoRA Inference Through Deterministic Split-K Reduction":
  sec. 5.2 / 6.1  identical-input replay: deterministic Split-K and Split-K = 1
                  give bit-identical FP32 shrink outputs on every replay, the
                  atomic variant does not (its mismatch rate is reported);
  Eq. 4           floating-point addition is not associative; the partition
                  order of the combine decides the result;
  Algorithm 1     the completion counter is back at zero after every launch.
Batch invariance (the bits of a row do not depend on the batch it is in) is
checked with fixed probe rows placed at random positions of batches of every
size.
"""
import os

import numpy as np
import pytest
import torch

import invariant_gemm_gb300 as ig
import synth
from helpers import bits, check_expand, check_shrink, need_gpu, run_apply, shape_of

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def replay(p, mode, n, split_k=8):
    """n identical-input replays; returns (#replays differing from replay 0 in
    z, fraction of differing z elements, #replays differing in y)."""
    sh = shape_of(p, mode, split_k)
    ws = ig.workspace(sh)
    z0, y0 = run_apply(p, mode=mode, split_k=split_k, ws=ws)
    z = torch.empty_like(z0)
    y = torch.empty_like(y0)
    diff_runs = torch.zeros((), dtype=torch.int64, device="cuda")
    diff_elems = torch.zeros((), dtype=torch.int64, device="cuda")
    diff_y = torch.zeros((), dtype=torch.int64, device="cuda")
    z0b = z0.view(torch.int32)
    y0b = y0.view(torch.int16)
    for _ in range(n):
        y.copy_(p.y)
        ig.lora_apply(sh, p.x, y, p.idx, p.A, p.B, p.scale, z, ws)
        ne = (z.view(torch.int32) != z0b).sum()
        diff_elems += ne
        diff_runs += (ne > 0).to(torch.int64)
        diff_y += (y.view(torch.int16) != y0b).any().to(torch.int64)
    assert ig.check_status(ws) == 0
    # Algorithm 1 (the last arriver resets its counter): every counter is back at zero
    counters = ws[256:256 + 4 * 65536].view(torch.int32)
    assert int(counters.abs().sum()) == 0
    return int(diff_runs), int(diff_elems) / (n * z0.numel()), int(diff_y)


@pytest.mark.parametrize("M", [1, 8, 32, 128, 256])
@pytest.mark.parametrize("mode", [ig.MODE_DET, ig.MODE_UNSPLIT], ids=["det", "unsplit"])
def test_replay_1000_bitwise(M, mode):
    p = synth.make_problem(M, 4096, 4096, 16, L=8, seed=1001 + M, device="cuda")
    runs, frac, yruns = replay(p, mode, 1000)
    assert runs == 0 and yruns == 0


@pytest.mark.parametrize("M", [8, 256])
def test_replay_atomic_reported(M):
    p = synth.make_problem(M, 4096, 4096, 16, L=8, seed=1001 + M, device="cuda")
    runs, frac, yruns = replay(p, ig.MODE_ATOMIC, 200)
    print(f"\natomic Split-K=8, M={M}: {runs}/200 replays differ in z "
          f"({100 * frac:.3f}% of elements), {yruns}/200 differ in y")


@pytest.mark.parametrize("mode", [ig.MODE_DET, ig.MODE_UNSPLIT], ids=["det", "unsplit"])
def test_batch_invariance_every_size(mode):
    """64 probe rows (K=4096, r=32, N=4096, 32 adapters) at seeded random
    positions in batches of every size 1..1024; the first b probes when b < 64.
    Probe rows of z and y must be bitwise equal across all batches."""
    K, N, r, L = 4096, 4096, 32, 32
    base = synth.make_problem(64, K, N, r, L=L, seed=1003, device="cuda")
    sh0 = shape_of(base, mode, 8, M=1024)
    ws = ig.workspace(sh0)
    ref_z = None
    ref_y = None
    for b in range(1, 1025):
        x, y, idx, pos = synth.probe_batch(base.x, base.y, base.idx, b, L, seed=5000 + b,
                                           device="cuda")
        sh = shape_of(base, mode, 8, M=b)
        z = torch.empty((1, b, r), dtype=torch.float32, device="cuda")
        ig.lora_apply(sh, x, y, idx, base.A, base.B, base.scale, z, ws)
        pz = z[0, pos].view(torch.int32)
        py = y[pos].view(torch.int16)
        n = pos.numel()
        if ref_z is None or n > ref_z.shape[0]:
            if ref_z is not None:
                assert torch.equal(pz[:ref_z.shape[0]], ref_z)
                assert torch.equal(py[:ref_y.shape[0]], ref_y)
            ref_z, ref_y = pz.clone(), py.clone()
        else:
            assert torch.equal(pz, ref_z[:n]), f"batch {b}"
            assert torch.equal(py, ref_y[:n]), f"batch {b}"
    assert ig.check_status(ws) == 0
    # and the probe rows are right
    zfull = torch.empty((1, 64, r), dtype=torch.float32, device="cuda")
    zfull[0] = ref_z.view(torch.float32)
    check_shrink(base.to("cpu"), zfull)


def _eq4_values():
    with open(os.path.join(GOLDEN, "eq4_nonassociativity.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    a, b, c, left, right = rows[0]
    return float(a), float(b), float(c), float(left), float(right)


def test_order_probe_partition_order():
    """Eq. 4: with a = 2^100 (a power of two, exact in bf16, standing in for
    the pages' 1e30), b = -a, c = 1, partition partials [a, c, 0, 0, b, c, 0, 0]
    summed in increasing partition order give fl(fl(fl(a + c) + b) + c) =
    fl(fl(a + b) + c) = 1, the pages' left-to-right value. A pairwise tree
    would give 0."""
    _, _, _, left, right = _eq4_values()
    S, Ks = 8, 256
    K = S * Ks
    a = 2.0 ** 100
    parts = [a, 1.0, 0.0, 0.0, -a, 1.0, 0.0, 0.0]
    x = torch.zeros((1, K), dtype=torch.float32)
    A = torch.zeros((1, 1, 8, K), dtype=torch.float32)
    for s in range(S):
        x[0, s * Ks] = 1.0
        A[0, 0, :, s * Ks] = parts[s]
    p = synth.Problem(M=1, K=K, N=8, r=8, slices=1, L=1, scale=1.0,
                      x=x.to(torch.bfloat16).cuda(), A=A.to(torch.bfloat16).cuda(),
                      B=torch.zeros((1, 1, 8, 8), dtype=torch.bfloat16, device="cuda"),
                      y=torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda"),
                      idx=torch.zeros(1, dtype=torch.int32, device="cuda"))
    z, _ = run_apply(p, mode=ig.MODE_DET, split_k=S)
    assert torch.all(z == left), z
    assert left != right


def test_out_of_range_adapter_flagged():
    p = synth.make_problem(64, 512, 256, 16, L=4, seed=3, device="cuda")
    p.idx[5] = 4
    p.idx[9] = -7
    z, y = run_apply(p, check=False)
    sh = shape_of(p)
    # a fresh workspace was used inside run_apply; re-run on one we keep
    ws = ig.workspace(sh)
    y2 = p.y.clone()
    ig.lora_apply(sh, p.x, y2, p.idx, p.A, p.B, p.scale, z, ws)
    assert ig.check_status(ws) == -7
    assert ig.check_status(ws) == 0         # cleared
    zc = z.cpu()
    assert torch.all(zc[:, 5] == 0) and torch.all(zc[:, 9] == 0)
    assert torch.equal(y2[5], p.y[5]) and torch.equal(y2[9], p.y[9])
    good = p.idx.clone()
    good[5] = -1
    good[9] = -1
    q = synth.Problem(**{**p.__dict__, "idx": good})
    check_shrink(q.to("cpu"), z)
    check_expand(q.to("cpu"), z, y2)


def test_poisoned_counters_detected_and_recovered():
    # the counter protocol runs in the two-kernel path (lora_shrink, or
    # lora_apply with IG_FLAG_UNFUSED)
    p = synth.make_problem(64, 4096, 256, 16, L=2, seed=4, device="cuda")
    sh = ig.make_shape(64, 4096, 256, 16, num_adapters=2, split_k=8, flags=ig.FLAG_UNFUSED)
    ws = ig.workspace(sh)
    ws[256:256 + 4 * 64].fill_(0x5A)        # garbage in the counter region
    z = torch.empty((1, 64, 16), dtype=torch.float32, device="cuda")
    y = p.y.clone()
    ig.lora_apply(sh, p.x, y, p.idx, p.A, p.B, p.scale, z, ws)
    assert ig.check_status(ws) == -6        # IG_ERR_WS_CORRUPT, counters re-zeroed
    y = p.y.clone()
    ig.lora_apply(sh, p.x, y, p.idx, p.A, p.B, p.scale, z, ws)
    assert ig.check_status(ws) == 0
    check_shrink(p.to("cpu"), z)
    check_expand(p.to("cpu"), z, y)


def test_token_map_reuse_across_layers():
    """One ig_map_tokens per batch, then shrink/expand of several layers with
    adapter_idx = NULL, equal to building the map on every call."""
    M, K, N, r, L = 96, 2048, 1024, 16, 6
    g = torch.Generator(device="cuda").manual_seed(9)
    idx = synth.adapter_ids(M, L, "uniform", g, "cuda", none_frac=0.1)
    layers = [synth.make_problem(M, K, N, r, L=L, seed=90 + i, device="cuda") for i in range(3)]
    sh = ig.make_shape(M, K, N, r, num_adapters=L, split_k=8)
    ws = ig.workspace(sh)
    ig.map_tokens(sh, idx, ws)
    for p in layers:
        z = torch.empty((1, M, r), dtype=torch.float32, device="cuda")
        y = p.y.clone()
        ig.lora_shrink(sh, p.x, p.A, None, p.scale, z, ws)
        ig.lora_expand(sh, z, p.B, None, y, ws)
        z2 = torch.empty_like(z)
        y2 = p.y.clone()
        ig.lora_apply(sh, p.x, y2, idx, p.A, p.B, p.scale, z2, ig.workspace(sh))
        assert torch.equal(z.view(torch.int32), z2.view(torch.int32))
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert ig.check_status(ws) == 0


def test_workspace_reused_across_shapes_without_reinit():
    cases = [(512, 8, 32), (7, 4, 16), (300, 16, 32), (1, 8, 16), (512, 8, 32)]
    need = max(ig.workspace_bytes(ig.make_shape(M, 4096, 1024, r, num_adapters=8, split_k=S))
               for M, S, r in cases)
    ws = ig.workspace(ig.make_shape(1, 4096, 1024, 16, num_adapters=8), min_bytes=need)
    for M, S, r in cases:
        p = synth.make_problem(M, 4096, 1024, r, L=8, seed=M * 10 + S, device="cuda")
        z, y = run_apply(p, mode=ig.MODE_DET, split_k=S, ws=ws)
        check_shrink(p.to("cpu"), z)
        check_expand(p.to("cpu"), z, y)


@pytest.mark.parametrize("mode", [ig.MODE_DET, ig.MODE_ATOMIC, ig.MODE_UNSPLIT],
                         ids=["det", "atomic", "unsplit"])
def test_dependent_layers_in_graph(mode):
    """Kernels start early (programmatic dependent launch) but must not read
    data the previous kernel writes before it has finished: chain layers so
    that each layer's x is the previous layer's y, run the chain as one CUDA
    graph with the static-weights flag, and compare with eager calls that
    synchronise after every layer."""
    M, K, L, r, layers = 48, 1024, 4, 16, 6
    probs = [synth.make_problem(M, K, K, r, L=L, seed=700 + i, device="cuda")
             for i in range(layers)]
    idx = probs[0].idx
    x0 = probs[0].x

    def run(flags, graph):
        sh = ig.make_shape(M, K, K, r, num_adapters=L, split_k=8, mode=mode, flags=flags)
        ws = ig.workspace(sh)
        ys = [p.y.clone() for p in probs]
        zs = [torch.empty((1, M, r), dtype=torch.float32, device="cuda") for _ in probs]

        def body(stream):
            ig.map_tokens(sh, idx, ws, stream)
            x = x0
            for l, p in enumerate(probs):
                ig.lora_apply(sh, x, ys[l], None, p.A, p.B, p.scale, zs[l], ws, stream)
                if not graph:
                    torch.cuda.synchronize()
                x = ys[l]

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                body(s)                      # warm-up (also initialises state)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            for l, p in enumerate(probs):
                ys[l].copy_(p.y)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(torch.cuda.current_stream())
            g.replay()
            torch.cuda.synchronize()
        else:
            body(torch.cuda.current_stream())
        assert ig.check_status(ws) == 0
        return zs, ys

    z_g, y_g = run(ig.FLAG_STATIC_WEIGHTS, graph=True)
    if mode == ig.MODE_ATOMIC:
        # no bitwise reference: check every layer against the oracle, with
        # that layer's x being the previous layer's y from the same run
        x = x0
        for l, p in enumerate(probs):
            q = synth.Problem(**{**p.__dict__, "x": x, "idx": idx})
            check_shrink(q.to("cpu"), z_g[l])
            check_expand(q.to("cpu"), z_g[l], y_g[l])
            x = y_g[l]
        return
    z_e, y_e = run(0, graph=False)
    for a, b in zip(y_e, y_g):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(z_e, z_g):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("M", [1, 77, 256])
def test_input_ready_layers_in_graph(M):
    """IG_FLAG_INPUT_READY lets the fused kernel run its shrink, exchange and
    combine while the previous kernel is still running; z and y must still
    be touched only after it completes. Layers with their own x but one
    shared y and one shared z, run as one CUDA graph with the flag, must give
    the same bits as eager calls without it that synchronise after every
    layer (each layer reads the y the previous one wrote)."""
    K, N, r, L, layers = 4096, 4096, 16, 8, 12
    probs = [synth.make_problem(M, K, N, r, L=L, seed=900 + i, device="cuda")
             for i in range(layers)]
    idx = probs[0].idx
    y0 = probs[0].y

    def run(flags, graph):
        sh = ig.make_shape(M, K, N, r, num_adapters=L, split_k=8, mode=ig.MODE_DET, flags=flags)
        assert ig.plan_query(sh)["apply_kernels"] == 1
        ws = ig.workspace(sh)
        y = y0.clone()
        z = torch.empty((1, M, r), dtype=torch.float32, device="cuda")
        zs = []

        def body(stream):
            ig.map_tokens(sh, idx, ws, stream)
            for p in probs:
                ig.lora_apply(sh, p.x, y, None, p.A, p.B, p.scale, z, ws, stream)
                if not graph:
                    torch.cuda.synchronize()
                    zs.append(z.clone())

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                body(s)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            y.copy_(y0)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(torch.cuda.current_stream())
            for _ in range(3):
                y.copy_(y0)
                g.replay()
                torch.cuda.synchronize()
        else:
            body(torch.cuda.current_stream())
        assert ig.check_status(ws) == 0
        return z, y, zs

    z_g, y_g, _ = run(ig.FLAG_STATIC_WEIGHTS | ig.FLAG_INPUT_READY, graph=True)
    z_e, y_e, zs_e = run(0, graph=False)
    assert torch.equal(y_g.view(torch.int16), y_e.view(torch.int16))
    assert torch.equal(z_g.view(torch.int32), z_e.view(torch.int32))
    # the eager chain's first layer against the oracle, and y did change
    check_shrink(probs[0].to("cpu"), zs_e[0])
    assert not torch.equal(y_e, y0)


FUSED_CASES = [
    # M, K, N, r, slices, L, S, none_frac
    (1, 4096, 4096, 16, 1, 8, 8, 0.0),
    (8, 4096, 4096, 16, 1, 8, 8, 0.0),
    (77, 4096, 264, 16, 3, 5, 8, 0.2),     # ragged columns per block, QKV slices
    (256, 4096, 4096, 16, 1, 8, 8, 0.05),
    (40, 512, 512, 8, 1, 1, 8, 0.0),
    (33, 2048, 1024, 16, 1, 4, 1, 0.0),    # cluster of one, 1024 columns per block
    (33, 2048, 1024, 16, 1, 4, 2, 0.0),
    (64, 8192, 1024, 16, 2, 4, 16, 0.1),   # 16-block clusters
    (300, 11008, 4096, 8, 1, 6, 8, 0.0),   # K/S = 1376: ragged k-blocks
    (19, 1032, 520, 16, 1, 3, 3, 0.1),     # K/S = 344: an 8-element last step
    (9, 1032, 256, 8, 2, 2, 1, 0.0),       # K/S = 1032: five k-blocks through four stages
]


@pytest.mark.parametrize("path", [ig.PATH_WARP, ig.PATH_FMA], ids=["warp", "fma"])
@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: "M%d_K%d_N%d_r%d_sl%d_S%d" % (
    c[0], c[1], c[2], c[3], c[4], c[6]))
def test_fused_apply_bitwise_equals_two_kernels(case, path):
    """lora_apply's one-launch cluster kernel (DET) and the two-kernel path
    (Split-K shrink with the counter protocol, then expand) give the same bits
    for z and y, with and without static weights, on the warp-level
    tensor-core path and on the CUDA-core FMA path; and both are within
    tolerance of the oracle."""
    M, K, N, r, slices, L, S, none_frac = case
    p = synth.make_problem(M, K, N, r, slices=slices, L=L, seed=M + K + S,
                           none_frac=none_frac, device="cuda")
    outs = []
    # static weights: the A fragments of short partitions go into registers
    # before the dependency wait (fused and two-kernel shrink alike)
    for flags in (0, ig.FLAG_UNFUSED, ig.FLAG_STATIC_WEIGHTS,
                  ig.FLAG_UNFUSED | ig.FLAG_STATIC_WEIGHTS):
        sh = ig.make_shape(M, K, N, r, slices=slices, num_adapters=L, split_k=S,
                           mode=ig.MODE_DET, path=path, flags=flags)
        if not flags & ig.FLAG_UNFUSED:
            assert ig.plan_query(sh)["apply_kernels"] == 1
        z, y = run_apply(p, mode=ig.MODE_DET, split_k=S, ws=ig.workspace(sh),
                         shape=sh)
        outs.append((z, y))
    for z, y in outs[1:]:
        assert torch.equal(z.view(torch.int32), outs[0][0].view(torch.int32))
        assert torch.equal(y.view(torch.int16), outs[0][1].view(torch.int16))
    check_shrink(p.to("cpu"), outs[0][0])
    check_expand(p.to("cpu"), outs[0][0], outs[0][1])


@pytest.mark.parametrize("path", [ig.PATH_WARP, ig.PATH_FMA], ids=["warp", "fma"])
@pytest.mark.parametrize("flags", [0, ig.FLAG_UNFUSED], ids=["fused", "two_kernel"])
def test_batch_invariance_rank16(flags, path):
    """Batch invariance of 64 probe rows at r = 16 (the fused kernel's rank)
    over batch sizes 1..512, on both small-rank paths."""
    K, N, r, L = 4096, 1024, 16, 8
    base = synth.make_problem(64, K, N, r, L=L, seed=2003, device="cuda")
    sh0 = ig.make_shape(512, K, N, r, num_adapters=L, split_k=8, path=path, flags=flags)
    ws = ig.workspace(sh0)
    ref_z = ref_y = None
    for b in range(1, 513):
        x, y, idx, pos = synth.probe_batch(base.x, base.y, base.idx, b, L, seed=9000 + b,
                                           device="cuda")
        sh = ig.make_shape(b, K, N, r, num_adapters=L, split_k=8, path=path, flags=flags)
        z = torch.empty((1, b, r), dtype=torch.float32, device="cuda")
        ig.lora_apply(sh, x, y, idx, base.A, base.B, base.scale, z, ws)
        pz = z[0, pos].view(torch.int32)
        py = y[pos].view(torch.int16)
        n = pos.numel()
        if ref_z is None or n > ref_z.shape[0]:
            if ref_z is not None:
                assert torch.equal(pz[:ref_z.shape[0]], ref_z)
                assert torch.equal(py[:ref_y.shape[0]], ref_y)
            ref_z, ref_y = pz.clone(), py.clone()
        else:
            assert torch.equal(pz, ref_z[:n]), f"batch {b}"
            assert torch.equal(py, ref_y[:n]), f"batch {b}"
    assert ig.check_status(ws) == 0


@pytest.mark.parametrize("S", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("r", [8, 16, 24])
def test_lora_shrink_cluster_combine_equals_counter(r, S):
    """lora_shrink (IG_MODE_DET, warp path) combines the S partitions inside a
    thread-block cluster where it can (S dividing the tile's outputs, S <=
    16); IG_FLAG_UNFUSED selects the counter protocol (Algorithm 1). Same
    partition order, so the same bits; S = 3 always uses the counter."""
    K = 3096 if S == 3 else 4096          # K/S = 1032 at S = 3: an 8-element last step
    p = synth.make_problem(90, K, 64, r, slices=2, L=5, seed=r * 100 + S, none_frac=0.1,
                           device="cuda")
    zs = []
    for flags in (0, ig.FLAG_UNFUSED):
        sh = ig.make_shape(p.M, K, p.N, r, slices=2, num_adapters=5, split_k=S,
                           mode=ig.MODE_DET, flags=flags)
        ws = ig.workspace(sh)
        z = torch.full((2, p.M, r), float("nan"), dtype=torch.float32, device="cuda")
        ig.lora_shrink(sh, p.x, p.A, p.idx, p.scale, z, ws)
        assert ig.check_status(ws) == 0
        zs.append(z)
    assert torch.equal(zs[0].view(torch.int32), zs[1].view(torch.int32))
    check_shrink(p.to("cpu"), zs[0])

"""The bounded-wait timeout path, made to run on purpose without faulting or
hanging anything.

IG_FLAG_TEST_COPY_TIMEOUT gives the first A-copy wait of every warp-path
shrink block no time: each block checks its first TMA copy once, right after
issuing it, finds it in flight, records IG_ERR_TIMEOUT in the workspace status
word, waits (with the normal bound) for its own copies to land and leaves. The
test checks that ig_check_status reports IG_ERR_TIMEOUT, and that the next
normal call on the same workspace is clean and matches the FP64 oracle (the
counters a failed block left behind are re-zeroed by ig_check_status). The
cluster partial-exchange waits never get a short budget: a peer would still be
storing into a block that had left.
"""
import pytest
import torch

import invariant_gemm_gb300 as ig
import synth
from helpers import check_expand, check_shrink, need_gpu

pytestmark = pytest.mark.gpu

IG_ERR_TIMEOUT = -8

CASES = {
    # name: (entry point, mode, flags)
    "unsplit_shrink": ("shrink", ig.MODE_UNSPLIT, 0),
    "det_counter_shrink": ("shrink", ig.MODE_DET, ig.FLAG_UNFUSED),
    "det_cluster_shrink": ("shrink", ig.MODE_DET, 0),
    "atomic_shrink": ("shrink", ig.MODE_ATOMIC, 0),
    "det_fused_apply": ("apply", ig.MODE_DET, 0),
    "det_fused_apply_static_weights": ("apply", ig.MODE_DET, ig.FLAG_STATIC_WEIGHTS),
    "det_two_kernel_apply": ("apply", ig.MODE_DET, ig.FLAG_UNFUSED),
}


def _flush_l2():
    # more than the 129 MB L2, so that the A copies come from HBM
    buf = torch.empty(320 << 20, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", sorted(CASES))
def test_expired_copy_wait_reports_timeout_and_workspace_recovers(case):
    need_gpu()
    entry, mode, flags = CASES[case]
    p = synth.make_problem(64, 4096, 1024, 16, L=4, seed=1701, none_frac=0.05, device="cuda")
    pc = p.to("cpu")

    def shape(extra):
        return ig.make_shape(p.M, p.K, p.N, p.r, slices=p.slices, num_adapters=p.L,
                             split_k=8, mode=mode, flags=flags | extra)

    sh_bad, sh = shape(ig.FLAG_TEST_COPY_TIMEOUT), shape(0)
    assert ig.plan_query(sh_bad)["determinism_key"] == ig.plan_query(sh)["determinism_key"]
    assert ig.plan_query(sh)["path"] == ig.PATH_WARP
    ws = ig.workspace(sh)
    z = torch.full((p.slices, p.M, p.r), float("nan"), dtype=torch.float32, device="cuda")

    def run(s):
        y = p.y.clone()
        if entry == "shrink":
            ig.lora_shrink(s, p.x, p.A, p.idx, p.scale, z, ws)
        else:
            ig.lora_apply(s, p.x, y, p.idx, p.A, p.B, p.scale, z, ws)
        return y

    _flush_l2()
    run(sh_bad)
    assert ig.check_status(ws) == IG_ERR_TIMEOUT
    assert ig.check_status(ws) == 0          # cleared by the check
    # the next normal calls on the same workspace are clean and right
    for _ in range(2):
        z.fill_(float("nan"))
        y = run(sh)
        assert ig.check_status(ws) == 0
        check_shrink(pc, z)
        if entry == "apply":
            check_expand(pc, z, y)
    if mode == ig.MODE_DET and (flags & ig.FLAG_UNFUSED):
        counters = ws[256:256 + 4 * 65536].view(torch.int32)
        assert int(torch.count_nonzero(counters)) == 0

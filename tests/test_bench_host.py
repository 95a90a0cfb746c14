"""Host-side pieces of the benchmark that its numbers rest on (no GPU).

* The algorithmic bytes of one lora_apply, which every roofline fraction
  divides by, counted element by element for the decode workload and
  compared with the closed form the benchmark uses.
* The hash that ties a recorded ncu capture to a kernel's code: it must
  change with the code and must not change with comments.
"""
from __future__ import annotations

import os

import bench


def test_algorithmic_bytes_of_the_decode_workload():
    W = bench.WORKLOAD
    M, K, N, r, sl, u = W["M"], W["K"], W["N"], W["r"], W["slices"], W["L"]
    b = bench.alg_bytes(M, K, N, r, sl, u)
    bf16, f32, i32 = 2, 4, 4
    x = M * K * bf16                       # read once
    a = u * sl * r * K * bf16              # each adapter present, read once
    z_write = sl * M * r * f32
    z_read = sl * M * r * f32
    bmat = u * sl * N * r * bf16
    y = 2 * M * sl * N * bf16              # read and written
    idx = M * i32                          # read by shrink and by expand
    assert b["shrink"] == x + a + z_write + idx
    assert b["expand"] == z_read + bmat + y + idx
    # the figure quoted with the bench line's roofline
    assert b["total"] == 8_423_424


def test_source_hash_follows_code_not_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "invariant_gemm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = csrc / "k.cu"
    src.write_text("// a kernel\n__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash("k.cu")
    src.write_text("/* reworded\n   comment */\n__global__ void k(int* p) {\n\n  p[0] = 1;\n}\n")
    assert bench.source_hash("k.cu") == h0
    src.write_text("// a kernel\n__global__ void k(int* p) {\n  p[0] = 2;  // store\n}\n")
    assert bench.source_hash("k.cu") != h0
    os.remove(src)
    assert bench.source_hash("k.cu") is None

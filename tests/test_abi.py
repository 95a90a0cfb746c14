"""The C-ABI library without a GPU: it loads, exports exactly what the header
declares, and the host-side plan and validation behave as documented.

No call here reaches a kernel launch: every call either fails host validation
or has M = 0.
"""
import ctypes
import math
import os
import re
import subprocess

import pytest

import invariant_gemm_gb300 as ig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "invariant_gemm.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


def header_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**([a-z_][a-z0-9_]*)\s*\(",
                       txt, flags=re.M)
    return sorted(set(names))


def test_library_exports_header_functions():
    decl = header_functions()
    assert decl == sorted(ig.EXPORTS)
    L = ig.lib()
    for name in decl:
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", ig.lib_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines()
                       if l.split() and re.match(r"^(ig_|lora_)", l.split()[-1])})
    assert exported == decl


def test_version_and_status_strings():
    assert b"sm_103a" in ig.lib().ig_version()
    for code in ig.STATUS:
        assert ig.status_string(code) not in ("", "unknown status")


def shp(**kw):
    d = dict(M=256, K=4096, N=4096, r=16, slices=1, num_adapters=8, split_k=8)
    d.update(kw)
    return ig.make_shape(**d)


def test_plan_independent_of_M():
    keys = set()
    for M in [0, 1, 7, 8, 32, 128, 256, 1000, 4096]:
        p = ig.plan_query(shp(M=M))
        keys.add((p["determinism_key"], p["path"], p["split_k"], p["k_split"],
                  p["shrink_bm"], p["shrink_bn"]))
    assert len(keys) == 1


@pytest.mark.parametrize("field,value", [("K", 8192), ("r", 32), ("split_k", 4),
                                         ("mode", ig.MODE_UNSPLIT), ("slices", 3),
                                         ("mode", ig.MODE_DET_TREE)])
def test_plan_key_changes_with_arithmetic_fields(field, value):
    a = ig.plan_query(shp())["determinism_key"]
    b = ig.plan_query(shp(**{field: value}))["determinism_key"]
    assert a != b


def test_unsplit_forces_one_partition():
    p = ig.plan_query(shp(mode=ig.MODE_UNSPLIT, split_k=8))
    assert p["split_k"] == 1 and p["k_split"] == 4096


def test_eq2_tile_counts():
    """Eq. 2 / Fig. 1 / sec. 2.1: N_tiles = ceil(M/BM) ceil(r/BN) output tiles
    per slice and S blocks per tile. The pages' examples (BM = 32, BN = 16)
    must satisfy it, and the plan's launch grid must cover Eq. 2 with the
    plan's own tile for every single-adapter case."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "eq2_tiles.txt"))
            if l.strip() and not l.startswith("#")]
    for M, r, BM, BN, slices, S, tiles, ctas, _ in rows:
        M, r, BM, BN, slices, S, tiles, ctas = map(int, (M, r, BM, BN, slices, S, tiles, ctas))
        assert math.ceil(M / BM) * math.ceil(r / BN) * slices == tiles
        assert tiles * S == ctas
        mode = ig.MODE_UNSPLIT if S == 1 else ig.MODE_DET
        p = ig.plan_query(shp(M=M, r=r, slices=slices, split_k=S, mode=mode, num_adapters=1))
        own = math.ceil(M / p["shrink_bm"]) * math.ceil(r / p["shrink_bn"]) * slices
        assert p["split_k"] == S
        assert p["shrink_ctas_max"] >= own * S


def test_workspace_bytes():
    assert ig.workspace_bytes(shp(K=4100)) == 0                 # K % 8
    assert ig.workspace_bytes(shp(split_k=3)) == 0              # (K/8) % S
    a = ig.workspace_bytes(shp(M=1))
    b = ig.workspace_bytes(shp(M=4096))
    assert 0 < a < b
    det = ig.workspace_bytes(shp(M=256))
    atom = ig.workspace_bytes(shp(M=256, mode=ig.MODE_ATOMIC))
    assert det > atom                                            # partials only for DET


@pytest.mark.parametrize("kw,code", [
    (dict(K=4100), -2), (dict(N=12), -2), (dict(r=12), -2), (dict(split_k=3), -2),
    (dict(split_k=0), -2), (dict(slices=0), -2), (dict(num_adapters=0), -2),
    (dict(M=-1), -2), (dict(mode=4), -1), (dict(path=7), -1),
    (dict(num_adapters=5000), -9), (dict(r=512), -9),
    (dict(mode=3, split_k=128), -9),
    (dict(r=256, path=2, flags=4), -9),        # three bf16 Z parts do not fit at r = 256
    (dict(K=2**31), -9), (dict(N=2**31), -9),  # 32-bit tensor-map coordinates
])
def test_plan_rejects(kw, code):
    with pytest.raises(ig.IGError) as e:
        ig.plan_query(shp(**kw))
    assert e.value.code == code


def test_fp32_z_large_rank_plan():
    """With FP32 Z the tcgen05 expand holds three bf16 parts of a 128-row Z tile;
    up to r = 192 they fit beside its copy stages, at r = 256 the automatic plan
    takes the warp path instead."""
    assert ig.plan_query(shp(r=192, flags=ig.FLAG_Z_FP32))["path"] == ig.PATH_MMA
    assert ig.plan_query(shp(r=256))["path"] == ig.PATH_MMA
    assert ig.plan_query(shp(r=256, flags=ig.FLAG_Z_FP32))["path"] == ig.PATH_WARP


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def call_shrink(shape, x=FAKE, A=FAKE, idx=FAKE, z=FAKE, ws=FAKE, nbytes=None):
    if nbytes is None:
        nbytes = ig.workspace_bytes(shape)
    return ig.lib().lora_shrink(ctypes.byref(shape), x, A, idx, 1.0, z, ws, nbytes, None)


def test_validation_before_launch():
    s = shp()
    n = ig.workspace_bytes(s)
    assert call_shrink(s, x=None) == -1
    assert call_shrink(s, z=None) == -1
    assert call_shrink(s, ws=None) == -1
    assert call_shrink(s, x=FAKE + 8) == -3
    assert call_shrink(s, idx=FAKE + 4) == -3
    assert call_shrink(s, ws=FAKE + 8) == -3
    assert call_shrink(s, nbytes=n - 1) == -4
    bad = shp(split_k=5)
    assert call_shrink(bad) == -2
    L = ig.lib()
    assert L.lora_expand(ctypes.byref(s), FAKE, None, FAKE, FAKE, FAKE, n, None) == -1
    assert L.lora_apply(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE + 2,
                        FAKE, n, None) == -3
    assert L.ig_map_tokens(ctypes.byref(s), None, FAKE, n, None) == -1
    assert L.ig_plan_query(None, None) == -1
    assert L.ig_check_status(None, 0, None) == -1


def test_zero_tokens_is_a_noop():
    s = shp(M=0)
    n = ig.workspace_bytes(s)
    assert n > 0
    L = ig.lib()
    assert L.lora_apply(ctypes.byref(s), None, None, None, None, None, 1.0, None, FAKE, n,
                        None) == 0
    assert L.lora_shrink(ctypes.byref(s), None, None, None, 1.0, None, FAKE, n, None) == 0

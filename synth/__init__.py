"""Seeded synthetic inputs for the multi-adapter LoRA shrink/expand path.

This module only draws random tensors. It holds none of the method's
arithmetic: no shrink, no expand, no rounding of outputs. Values are drawn
with torch's seeded generators and converted to bf16 with torch's own
conversion, so the values are valid bf16 inputs and nothing more.

Both the CUDA path (through the tests and the bench) and the FP64 oracle
(through the tests) consume what it makes; neither side imports the other.

Workload shapes follow "Reproducible LoRA Inference Through Deterministic
Split-K Reduction": Eq. 1 (A in R^{r x H}, B in R^{Hout x r}), sec. 3.2
(ranks 16 and 32, alpha = 2r so scale = 2), sec. 2.1 (decode, three fused QKV
slices) and sec. 4 (Split-K = 8).

Layouts (row-major, innermost index last):
  x        bf16 [M][K]
  A_stack  bf16 [L][slices][r][K]
  B_stack  bf16 [L][slices][N][r]
  y        bf16 [M][slices*N]
  idx      int32 [M], -1 = token without adapter
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = [
    "Problem",
    "make_problem",
    "adapter_ids",
    "probe_batch",
    "zipf_probs",
]


@dataclasses.dataclass
class Problem:
    M: int
    K: int
    N: int
    r: int
    slices: int
    L: int
    scale: float
    x: torch.Tensor
    A: torch.Tensor
    B: torch.Tensor
    y: torch.Tensor
    idx: torch.Tensor

    def to(self, device) -> "Problem":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
             for k, v in dataclasses.asdict(self).items()}
        return Problem(**f)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def _int_bf16(shape, lo: int, hi: int, g: torch.Generator, device) -> torch.Tensor:
    t = torch.randint(lo, hi + 1, tuple(shape), generator=g, device=device,
                      dtype=torch.int32)
    return t.to(torch.bfloat16)


def zipf_probs(L: int, exponent: float) -> torch.Tensor:
    """Truncated Zipf weights p_i proportional to i**-exponent, i = 1..L."""
    w = torch.tensor([1.0 / (i ** exponent) for i in range(1, L + 1)],
                     dtype=torch.float64)
    return w / w.sum()


def adapter_ids(M: int, L: int, kind: str, g: torch.Generator, device,
                segment: int = 256, zipf_exponent: float = 1.1,
                none_frac: float = 0.0) -> torch.Tensor:
    """Per-token adapter index.

    kind: "uniform" (iid over 0..L-1), "segments" (contiguous blocks of
    `segment` tokens, block b -> adapter b mod L), "zipf" (iid from truncated
    Zipf), "single" (all 0). `none_frac` of the tokens (chosen at random) get
    -1, i.e. no adapter.
    """
    if kind == "uniform":
        ids = torch.randint(0, L, (M,), generator=g, device=device, dtype=torch.int32)
    elif kind == "segments":
        ids = (torch.arange(M, device=device, dtype=torch.int64) // segment) % L
        ids = ids.to(torch.int32)
    elif kind == "zipf":
        p = zipf_probs(L, zipf_exponent).to(torch.float32).to(device)
        if M == 0:
            ids = torch.empty(0, dtype=torch.int32, device=device)
        else:
            ids = torch.multinomial(p, M, replacement=True, generator=g).to(torch.int32)
    elif kind == "single":
        ids = torch.zeros(M, dtype=torch.int32, device=device)
    else:
        raise ValueError(f"unknown adapter-id kind {kind!r}")
    if none_frac > 0 and M > 0:
        mask = torch.rand(M, generator=g, device=device) < none_frac
        ids = torch.where(mask, torch.full_like(ids, -1), ids)
    return ids.contiguous()


def make_problem(M: int, K: int, N: int, r: int, *, slices: int = 1, L: int = 1,
                 scale: float = 2.0, seed: int = 0, dist: str = "normal",
                 ids: str = "uniform", segment: int = 256,
                 none_frac: float = 0.0, device="cpu") -> Problem:
    """One seeded LoRA problem.

    dist="normal": x ~ N(0,1), A ~ N(0,1/K), B ~ N(0,1/r), y ~ N(0,1)
    (variances as written; standard deviations K**-0.5 and r**-0.5).
    dist="int": x, A, B, y uniform integers in [-4, 4] (exact in bf16).
    """
    g = _gen(seed, device)
    if dist == "normal":
        x = _normal_bf16((M, K), 1.0, g, device)
        A = _normal_bf16((L, slices, r, K), 1.0 / math.sqrt(K), g, device)
        B = _normal_bf16((L, slices, N, r), 1.0 / math.sqrt(r), g, device)
        y = _normal_bf16((M, slices * N), 1.0, g, device)
    elif dist == "int":
        x = _int_bf16((M, K), -4, 4, g, device)
        A = _int_bf16((L, slices, r, K), -4, 4, g, device)
        B = _int_bf16((L, slices, N, r), -4, 4, g, device)
        y = _int_bf16((M, slices * N), -4, 4, g, device)
    else:
        raise ValueError(f"unknown dist {dist!r}")
    idx = adapter_ids(M, L, ids, g, device, segment=segment, none_frac=none_frac)
    return Problem(M=M, K=K, N=N, r=r, slices=slices, L=L, scale=scale,
                   x=x, A=A, B=B, y=y, idx=idx)


def probe_batch(probe_x: torch.Tensor, probe_y: torch.Tensor,
                probe_idx: torch.Tensor, batch: int, L: int, seed: int,
                device="cpu"):
    """Place probe rows at seeded random positions of a batch of `batch` rows.

    The other rows are N(0,1) filler with random adapters in 0..L-1. When
    `batch` is smaller than the number of probes, the first `batch` probes fill
    the batch. Returns (x, y, idx, positions) with positions[i] = row of probe i.
    """
    P = probe_x.shape[0]
    K = probe_x.shape[1]
    NY = probe_y.shape[1]
    g = _gen(seed, device)
    nprobe = min(P, batch)
    x = _normal_bf16((batch, K), 1.0, g, device)
    y = _normal_bf16((batch, NY), 1.0, g, device)
    idx = torch.randint(0, L, (batch,), generator=g, device=device, dtype=torch.int32)
    pos = torch.randperm(batch, generator=g, device=device)[:nprobe]
    x[pos] = probe_x[:nprobe].to(device)
    y[pos] = probe_y[:nprobe].to(device)
    idx[pos] = probe_idx[:nprobe].to(device)
    return x.contiguous(), y.contiguous(), idx.contiguous(), pos

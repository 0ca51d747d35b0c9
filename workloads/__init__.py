"""Seeded synthetic inputs for the block-scaled E4M3 GEMM workloads.

This module serves both the CUDA path and the oracle and therefore holds none
of the GEMM's arithmetic: only random draws, clipping, conversion to E4M3 codes
(by torch's own float8 cast) and, for the arbitrary-scale workload, the
per-block absmax quantisation that produces the inputs.  Everything is
generated with an explicit ``torch.Generator`` so a (config, seed, device)
triple always yields the same bytes on a given machine.

Workloads (shapes and value distributions of the FP8 GEMM library article,
hncyxsy.com/news/241433: section 2.1 E4M3 with max 448, section 2.2 32x32
block scales, section 4 grouped decode batches, section 5.1 prefill shapes):

* ``square``   M=N=K (256 or 4096): A, B = E4M3(clip(N(0,1), +-448)); scales
  2^e with e uniform in [-4, 4], one per 32x32 block of A and of B.
* ``prefill``  M=8192, N=28672, K=8192: A = E4M3 of N(0,1) activations; B =
  E4M3 of N(0,0.02) weights renormalised by 1/0.02 (so N(0,1)); scales 2^e,
  e uniform in [-6, 2].
* ``grouped``  G=16 decode groups, M_g uniform in [1, 64], N=4096, K=7168,
  each group with its own B and power-of-two scales (e in [-4, 4]); the A rows
  of all groups are concatenated and an offset array gives each group's first
  row.
* ``outlier``  M=N=K=8192: A from bf16 N(0,1) with 0.5 % of entries (Bernoulli
  per entry) multiplied by 50, B from bf16 N(0,1); each 32x32 block quantised
  with fp32 scale amax/448 (1.0 for an all-zero block), q = E4M3(x/scale)
  saturating at +-448.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def to_e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """fp32 values (already inside +-448) -> uint8 E4M3 codes via torch's cast."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def pow2_scales(rows: int, kb: int, lo: int, hi: int, g: torch.Generator, device) -> torch.Tensor:
    """[ceil(rows/32), kb] fp32 scales 2^e with e uniform in [lo, hi]."""
    e = torch.randint(lo, hi + 1, ((rows + 31) // 32, kb), generator=g, device=device)
    return torch.ldexp(torch.ones_like(e, dtype=torch.float32), e.to(torch.int32))


def normal_codes(rows: int, K: int, g: torch.Generator, device, std: float = 1.0,
                 renorm: float = 1.0) -> torch.Tensor:
    x = torch.randn(rows, K, generator=g, device=device, dtype=torch.float32)
    if std != 1.0 or renorm != 1.0:
        x = (x * std) * renorm
    return to_e4m3_codes(x)


@dataclass
class Problem:
    """One block-scaled GEMM: A [M,K] and B [N,K] E4M3 codes (uint8), sA
    [ceil(M/32),K/32] and sB [ceil(N/32),K/32] fp32 scales."""
    A: torch.Tensor
    sA: torch.Tensor
    B: torch.Tensor
    sB: torch.Tensor
    M: int
    N: int
    K: int
    name: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        return (self.M * self.K + self.N * self.K + 4 * self.sA.numel()
                + 4 * self.sB.numel() + 2 * self.M * self.N)


@dataclass
class GroupedProblem:
    """G independent GEMMs sharing N and K.  ``A`` holds all groups' rows
    concatenated ([sum M_g, K]); ``offsets[g]`` is group g's first row.  Each
    group has its own B_g, sA_g (group-local row blocks) and sB_g."""
    A: torch.Tensor
    sA: list
    B: list
    sB: list
    Ms: list
    offsets: list
    N: int
    K: int
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return len(self.Ms)

    def A_group(self, g: int) -> torch.Tensor:
        o = self.offsets[g]
        return self.A[o:o + self.Ms[g]]

    @property
    def flops(self) -> int:
        return 2 * sum(self.Ms) * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        total_m = sum(self.Ms)
        b = self.G * self.N * self.K + total_m * self.K + 2 * total_m * self.N
        b += sum(4 * s.numel() for s in self.sA) + sum(4 * s.numel() for s in self.sB)
        return b


def square(n: int = 256, seed: int = 0, device="cpu", M: int | None = None) -> Problem:
    """M=N=K=n (M overridable) with power-of-two scales, e in [-4, 4]."""
    g = _gen(seed, device)
    M = n if M is None else M
    N = K = n
    A = normal_codes(M, K, g, device)
    B = normal_codes(N, K, g, device)
    sA = pow2_scales(M, K // 32, -4, 4, g, device)
    sB = pow2_scales(N, K // 32, -4, 4, g, device)
    return Problem(A, sA, B, sB, M, N, K, name=f"square{n}")


def prefill(seed: int = 0, device="cpu", M: int = 8192, N: int = 28672,
            K: int = 8192) -> Problem:
    g = _gen(seed, device)
    A = normal_codes(M, K, g, device)
    B = normal_codes(N, K, g, device, std=0.02, renorm=1.0 / 0.02)
    sA = pow2_scales(M, K // 32, -6, 2, g, device)
    sB = pow2_scales(N, K // 32, -6, 2, g, device)
    return Problem(A, sA, B, sB, M, N, K, name=f"prefill{M}x{N}x{K}")


def grouped(seed: int = 0, device="cpu", G: int = 16, m_lo: int = 1, m_hi: int = 64,
            N: int = 4096, K: int = 7168, Ms: list | None = None) -> GroupedProblem:
    g = _gen(seed, device)
    if Ms is None:
        Ms = torch.randint(m_lo, m_hi + 1, (G,), generator=_gen(seed, "cpu")).tolist()
    Ms = [int(m) for m in Ms]
    offsets, o = [], 0
    for m in Ms:
        offsets.append(o)
        o += m
    A = normal_codes(o, K, g, device)
    sA, B, sB = [], [], []
    for m in Ms:
        sA.append(pow2_scales(m, K // 32, -4, 4, g, device))
    for _ in Ms:
        B.append(normal_codes(N, K, g, device))
        sB.append(pow2_scales(N, K // 32, -4, 4, g, device))
    return GroupedProblem(A, sA, B, sB, Ms, offsets, N, K,
                          name=f"grouped{len(Ms)}x{N}x{K}")


def block_quantize(x: torch.Tensor):
    """Per 32x32 block: scale = amax/448 in fp32 (1.0 when the block is all
    zero), codes = E4M3(x / scale) saturating.  Rows need not be a multiple of
    32 (the last row block is partial); columns must be."""
    R, K = x.shape
    Rp = (R + 31) // 32 * 32
    xp = torch.zeros(Rp, K, dtype=torch.float32, device=x.device)
    xp[:R] = x.float()
    blocks = xp.view(Rp // 32, 32, K // 32, 32)
    amax = blocks.abs().amax(dim=(1, 3))                       # [Rp/32, K/32]
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = blocks / scale[:, None, :, None]
    codes = to_e4m3_codes(q).view(Rp, K)[:R].contiguous()
    return codes, scale.contiguous()


def outlier(n: int = 8192, seed: int = 0, device="cpu", M: int | None = None,
            frac: float = 0.005, factor: float = 50.0) -> Problem:
    """Arbitrary fp32 block scales (amax/448), A with 0.5 % outliers x50."""
    g = _gen(seed, device)
    M = n if M is None else M
    N = K = n
    xa = torch.randn(M, K, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    hit = torch.rand(M, K, generator=g, device=device) < frac
    xa = torch.where(hit, (xa.float() * factor).to(torch.bfloat16), xa)
    xb = torch.randn(N, K, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    A, sA = block_quantize(xa)
    B, sB = block_quantize(xb)
    return Problem(A, sA, B, sB, M, N, K, name=f"outlier{n}")


def prefix_rows(p: Problem, m: int) -> Problem:
    """The first m rows of A (and their row blocks of sA), same B: the
    batch-invariance sweep's smaller launches."""
    return Problem(p.A[:m].contiguous(), p.sA[:(m + 31) // 32].contiguous(), p.B, p.sB,
                   m, p.N, p.K, name=f"{p.name}[:{m}]")


CONFIGS = {
    "c0": dict(kind="square", n=256),
    "c1": dict(kind="square", n=4096),
    "c2": dict(kind="prefill"),
    "c3": dict(kind="grouped"),
    "c4": dict(kind="outlier", n=8192),
}


def make(name: str, seed: int = 0, device="cpu"):
    cfg = dict(CONFIGS[name])
    kind = cfg.pop("kind")
    return {"square": square, "prefill": prefill, "grouped": grouped,
            "outlier": outlier}[kind](seed=seed, device=device, **cfg)

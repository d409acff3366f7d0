"""Seeded synthetic inputs for the benchmark workloads and the parity tests.

This module only draws random numbers in the shapes, dtypes and
distributions of the workloads; it holds none of the layers' arithmetic and
is shared, unchanged, by the CUDA path's tests, the oracle comparisons and
the benchmark.

Conventions
-----------
* N(mu, sigma) means mean mu and standard deviation sigma (torch.normal's
  convention), drawn in float32 and rounded once to the stored dtype.
* Every tensor has its own torch.Generator seeded with
  ``20261202 + 1_000_000 * workload_index + crc32(tensor_name) % 1_000_000``.
  CPU and CUDA generators give different (each reproducible) values; a
  parity test always hands the very same tensor to both sides.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch

SEED_BASE = 20261202
SWEEP_WIDTHS = (16, 24, 64, 128, 256, 512, 1024, 2048, 4096, 8192)
SWEEP_ELEMS = 1 << 28


def seed_for(workload_index: int, name: str) -> int:
    return SEED_BASE + 1_000_000 * workload_index + zlib.crc32(name.encode()) % 1_000_000


def normal(shape, mean: float, std: float, dtype, *, seed: int, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def with_outliers(shape, frac: float, factor: float, dtype, *, seed: int, mask_seed: int,
                  device="cpu") -> torch.Tensor:
    """N(0,1) with a seeded Bernoulli(frac) subset multiplied by `factor`."""
    t = normal(shape, 0.0, 1.0, torch.float32, seed=seed, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(mask_seed)
    hit = torch.rand(shape, generator=g, device=device) < frac
    t = torch.where(hit, t * factor, t)
    return t.to(dtype)


@dataclass
class Workload:
    """One workload: a layer, a shape, dtypes and its input distributions."""
    name: str
    index: int                # workload index (seed namespace)
    op: str                   # "dyt" | "layernorm" | "rmsnorm"
    M: int
    N: int
    xdtype: torch.dtype
    pdtype: torch.dtype
    eps: float = 0.0
    x_std: float = 1.0
    outliers: tuple | None = None      # (fraction, factor)
    alpha: float | None = None         # fixed DyT alpha; None: drawn from param_dist
    param_dist: dict = field(default_factory=dict)   # name -> (mean, std)
    bwd_only: bool = False
    lead: tuple | None = None          # (B, H, S): x and dy head-major, seen as [B, S, H, N]

    def inputs(self, device="cpu") -> dict:
        """x, dy and the parameters, all seeded.  With `lead`, x and dy are
        [B, H, S, N] tensors transposed to [B, S, H, N] views (their storage
        under "x_storage" and "dy_storage")."""
        s = lambda n: seed_for(self.index, f"{self.name}/{n}")  # noqa: E731
        shape = (self.M, self.N) if self.lead is None else (*self.lead, self.N)
        if self.outliers:
            frac, factor = self.outliers
            x = with_outliers(shape, frac, factor, self.xdtype, seed=s("x"), mask_seed=s("x_mask"),
                              device=device)
        else:
            x = normal(shape, 0.0, self.x_std, self.xdtype, seed=s("x"), device=device)
        out = {"x": x, "dy": normal(shape, 0.0, 1.0, self.xdtype, seed=s("dy"), device=device)}
        if self.lead is not None:
            for k in ("x", "dy"):
                out[k + "_storage"] = out[k]
                out[k] = out[k].transpose(1, 2)
        for pname, (mu, sd) in self.param_dist.items():
            n = 1 if pname == "alpha" else self.N
            out[pname] = normal((n,), mu, sd, self.pdtype, seed=s(pname), device=device)
        if self.op == "dyt" and self.alpha is not None:
            out["alpha"] = torch.full((1,), self.alpha, dtype=self.pdtype, device=device)
        return out


def _dyt_params(gm=(1.0, 0.1), bt=(0.0, 0.1)):
    return {"gamma": gm, "beta": bt}


# The five workloads (numbered 1..5 as their seed namespaces).
DYT_F32_SMALL = Workload("dyt_f32_4096x64", 1, "dyt", 4096, 64, torch.float32, torch.float32,
                         alpha=0.5, param_dist=_dyt_params())
LN_BWD_TALL = Workload("layernorm_bwd_401408x24", 2, "layernorm", 25088 * 16, 24, torch.bfloat16,
                       torch.float32, eps=1e-5,
                       param_dist={"gamma": (1.0, 0.1), "beta": (0.0, 0.1)}, bwd_only=True)
DYT_BF16_TALL = Workload("dyt_bf16_1048576x128", 3, "dyt", 1 << 20, 128, torch.bfloat16,
                         torch.float32, x_std=2.0, alpha=0.8, param_dist=_dyt_params())
DYT_BF16_ALPHA_INF = Workload("dyt_bf16_1000x128_alpha_inf", 3, "dyt", 1000, 128, torch.bfloat16,
                              torch.float32, x_std=2.0, alpha=math.inf, param_dist=_dyt_params())
RMS_BF16 = Workload("rmsnorm_bf16_16384x2048", 4, "rmsnorm", 16384, 2048, torch.bfloat16,
                    torch.bfloat16, eps=1e-6, outliers=(0.01, 20.0),
                    param_dist={"weight": (1.0, 0.05)})


def sweep(op: str, N: int, xdtype: torch.dtype = torch.bfloat16) -> Workload:
    """Workload 5: bf16 activations (or xdtype), fp32 parameters ~ N(1, 0.1),
    M = 2^28 // N."""
    M = SWEEP_ELEMS // N
    if op == "dyt":
        params = {"alpha": (1.0, 0.1), "gamma": (1.0, 0.1), "beta": (1.0, 0.1)}
        eps = 0.0
    elif op == "layernorm":
        params = {"gamma": (1.0, 0.1), "beta": (1.0, 0.1)}
        eps = 1e-5
    else:
        params = {"weight": (1.0, 0.1)}
        eps = 1e-6
    tag = "" if xdtype == torch.bfloat16 else "_" + str(xdtype)[6:]
    return Workload(f"sweep{tag}_{op}_{M}x{N}", 5, op, M, N, xdtype, torch.float32, eps=eps,
                    param_dist=params)


def head_major(op: str, B: int, H: int, S: int, D: int) -> Workload:
    """Workload 6: per-head normalization of a head-major [B, H, S, D] bf16
    activation read as [B, S, H, D] rows of D (the query/key norm of
    DeepSpeed PR 8645, whose head-major inputs and upstream gradients come
    straight from attention), fp32 parameters as in the sweep."""
    w = sweep(op, D)
    from dataclasses import replace
    return replace(w, name=f"headmajor_{op}_{B}x{H}x{S}x{D}", index=6, M=B * H * S,
                   lead=(B, H, S))


def sweep_all(xdtype: torch.dtype = torch.bfloat16):
    return [sweep(op, n, xdtype) for n in SWEEP_WIDTHS for op in ("dyt", "layernorm", "rmsnorm")]


def scaled(w: Workload, M: int) -> Workload:
    """The same recipe with fewer rows (small parity cases)."""
    from dataclasses import replace
    return replace(w, M=M, lead=None, name=f"{w.name}@M{M}")

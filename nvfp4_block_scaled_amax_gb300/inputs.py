"""Seeded synthetic inputs for the NVFP4 workloads.

This module holds no NVFP4 arithmetic: it only draws random matrices, so the
CUDA path and the CPU oracle can be fed the same bytes.  Every tensor is
generated on the CPU with a seeded ``torch.Generator`` (the same bytes on any
machine), in FP32 and then rounded to BF16 where the workload is BF16.

Workloads (the shapes and value mixes of the benchmarks on the pages, which
use ``torch.randn`` BF16 inputs with a fixed seed):

* ``randn``            N(0, 1).
* ``row_mix``          N(0, 1) with 1% of rows multiplied by 100 and a disjoint
                       1% of rows set to zero (rows picked by a seeded
                       ``randperm``): the per-token activation mix of the
                       row-scaled recipe.
* ``outliers``         N(0, 1) with 0.1% of elements (seeded ``randperm``
                       positions) replaced by +-50 (seeded signs).
* ``reuse_sequence``   x, x * 0.5, zeros, x * 4: inputs whose maximum
                       decreases, reaches zero and rises again, fed through
                       one reused output ("Write both NVFP4 amax buffers",
                       Changes: the dual-amax test).
"""
from __future__ import annotations

import torch

MASK64 = (1 << 64) - 1


def splitmix64(seed: int) -> int:
    """SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): one output for state
    ``seed``.  Used to derive the 16-bit RHT sign mask from a seed."""
    z = (seed + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def sign_mask_from_seed(seed: int) -> int:
    """16-bit random sign mask for the Hadamard transform: bit i set means
    element i of every 16-element column block is negated."""
    return splitmix64(seed) & 0xFFFF


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def randn(M: int, N: int, seed: int, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """N(0, 1) matrix, drawn in FP32 and rounded to ``dtype``."""
    x = torch.randn((M, N), generator=_gen(seed), dtype=torch.float32)
    return x.to(dtype)


def row_mix(M: int, N: int, seed: int, frac: float = 0.01, big: float = 100.0,
            dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """N(0, 1) with ``frac`` of rows scaled by ``big`` and a disjoint ``frac``
    of rows zeroed."""
    g = _gen(seed)
    x = torch.randn((M, N), generator=g, dtype=torch.float32)
    k = max(1, int(round(M * frac))) if M > 1 else 0
    perm = torch.randperm(M, generator=g)
    x[perm[:k]] *= big
    x[perm[k:2 * k]] = 0.0
    return x.to(dtype)


def outliers(M: int, N: int, seed: int, frac: float = 0.001, value: float = 50.0,
             dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """N(0, 1) with ``frac`` of elements replaced by +-``value``."""
    g = _gen(seed)
    x = torch.randn((M, N), generator=g, dtype=torch.float32)
    n = M * N
    k = int(round(n * frac))
    pos = torch.randperm(n, generator=g)[:k]
    signs = torch.randint(0, 2, (k,), generator=g).to(torch.float32) * 2.0 - 1.0
    x.view(-1)[pos] = signs * value
    return x.to(dtype)


def reuse_sequence(x: torch.Tensor) -> list[torch.Tensor]:
    """The dual-amax reuse sequence: max decreasing, zero, rising."""
    return [x, x * 0.5, torch.zeros_like(x), x * 4.0]


# The five workloads, by name: (mode, M, N, dtype, generator, seed, flags).
WORKLOADS = {
    "1d_1024x1024_bf16": dict(mode="1d", M=1024, N=1024, dtype=torch.bfloat16, gen="randn", seed=0,
                              swizzled=False),
    "2d_8192x5120_bf16": dict(mode="2d", M=8192, N=5120, dtype=torch.bfloat16, gen="randn", seed=1,
                              swizzled=True),
    "rowscaled_16384x4096_bf16": dict(mode="row_scaled", M=16384, N=4096, dtype=torch.bfloat16,
                                      gen="row_mix", seed=2, swizzled=True),
    "rht_8192x8192_bf16": dict(mode="rht", M=8192, N=8192, dtype=torch.bfloat16, gen="outliers",
                               seed=3, swizzled=False),
    "1d_1088x1024_bf16": dict(mode="1d", M=1088, N=1024, dtype=torch.bfloat16, gen="randn", seed=4,
                              swizzled=False),
    "1d_4096x3072_fp32": dict(mode="1d", M=4096, N=3072, dtype=torch.float32, gen="randn", seed=5,
                              swizzled=True),
    "1d_8192x5120_bf16": dict(mode="1d", M=8192, N=5120, dtype=torch.bfloat16, gen="randn", seed=6,
                              swizzled=True),
    "1d_16384x16384_bf16": dict(mode="1d", M=16384, N=16384, dtype=torch.bfloat16, gen="randn",
                                seed=7, swizzled=True),
}


def random_bytes(M: int, N: int, seed: int) -> torch.Tensor:
    """Uniform random bytes (uint8, M x N): the random numbers of
    stochastic rounding, drawn on the host."""
    return torch.randint(0, 256, (M, N), generator=_gen(seed), dtype=torch.int32).to(torch.uint8)


# Stochastic rounding: the 1D 8192x5120 BF16 workload (seed 6) with random
# bytes drawn from seed 9.
SR = dict(mode="1d", M=8192, N=5120, dtype=torch.bfloat16, gen="randn", seed=6, swizzled=True, rbits_seed=9)


# Grouped quantize (tensors stacked along the first dimension, each with its
# own amax): eight members of uneven height, multiples of 128, 8192 rows in
# all, N = 5120; member g is N(0, 1) times 10^e_g, e_g drawn from the seed in
# [-3, 3] (members of different magnitude, like the per-expert inputs of a
# mixture-of-experts layer).
GROUPED = dict(mode="1d", splits=[1280, 768, 1152, 896, 1024, 1408, 640, 1024], N=5120, dtype=torch.bfloat16,
               seed=8, swizzled=True)


def make_grouped(spec=None, splits=None, N: int | None = None) -> torch.Tensor:
    """Builds the stacked input of a grouped workload (optionally with other
    member heights or N)."""
    spec = GROUPED if spec is None else spec
    splits = spec["splits"] if splits is None else list(splits)
    N = spec["N"] if N is None else N
    g = _gen(spec["seed"])
    x = torch.randn((sum(splits), N), generator=g, dtype=torch.float32)
    e = torch.randint(-3, 4, (len(splits),), generator=g)
    r = 0
    for m, k in zip(splits, e.tolist()):
        x[r:r + m] *= float(10.0 ** k)
        r += m
    return x.to(spec["dtype"])


def make(name_or_spec, M: int | None = None, N: int | None = None) -> torch.Tensor:
    """Builds the input of a named workload (optionally at another shape)."""
    spec = WORKLOADS[name_or_spec] if isinstance(name_or_spec, str) else name_or_spec
    M = spec["M"] if M is None else M
    N = spec["N"] if N is None else N
    gen = {"randn": randn, "row_mix": row_mix, "outliers": outliers}[spec["gen"]]
    return gen(M, N, spec["seed"], dtype=spec["dtype"])

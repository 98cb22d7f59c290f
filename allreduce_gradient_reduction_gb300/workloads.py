"""Seeded synthetic inputs for the simulated AllReduce.

This module only draws numbers and describes shapes; it holds none of the
reduction's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.  Every rank buffer is drawn from numpy's PCG64 with seed
``20261202 + 1000 * config + rank``.

bf16 inputs are made by keeping the upper 16 bits of a binary32 draw
(truncation toward zero).  That yields a bf16 value near the draw; it is an
input recipe, not the rounding the reduction itself uses.

Workloads (the pages use no public dataset; these are the synthetic stand-ins
for the configurations the method is measured on):

  small    N=4 ranks, f32, 4096 elements, integers uniform in [-8, 8]
  bucket   N=8, f32, 6,553,600 elements (one 25 MiB DDP bucket), normal(0, 1e-3)
  large    N=8, bf16, 67,108,864 elements (128 MiB per rank), normal(0, 1) with
           an independent 1% of entries scaled by 100
  gpt2     N=8, f32 gradients shaped like GPT-2 small (148 tensors,
           124,439,808 parameters), normal(0, 1e-4)
  sweep    per-rank size 4 KiB .. 1 GiB (powers of two), N in {2,4,8,16,64}
           with N * size <= 64 GiB, f32 and bf16, uniform(-1, 1)
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202

CONFIG_SMALL, CONFIG_BUCKET, CONFIG_LARGE, CONFIG_GPT2, CONFIG_SWEEP = 1, 2, 3, 4, 5

SMALL = {"config": CONFIG_SMALL, "nranks": 4, "count": 4096, "dtype": "f32"}
BUCKET = {"config": CONFIG_BUCKET, "nranks": 8, "count": 6_553_600, "dtype": "f32"}
LARGE = {"config": CONFIG_LARGE, "nranks": 8, "count": 67_108_864, "dtype": "bf16"}
GPT2 = {"config": CONFIG_GPT2, "nranks": 8, "dtype": "f32"}

SWEEP_RANKS = (2, 4, 8, 16, 64)
SWEEP_BYTES = tuple(1 << k for k in range(12, 31))  # 4 KiB .. 1 GiB per rank
SWEEP_CAP_BYTES = 64 << 30                            # N * size <= 64 GiB


def rng(config: int, rank: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(BASE_SEED + 1000 * config + rank))


def f32_to_bf16_bits_truncate(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of each binary32 value, as uint16 bf16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def small_inputs(nranks: int = 4, count: int = 4096, config: int = CONFIG_SMALL) -> np.ndarray:
    """Integers uniform in [-8, 8], stored as binary32 (all sums are exact)."""
    return np.stack([rng(config, r).integers(-8, 9, size=count).astype(np.float32) for r in range(nranks)])


def three_rank_example() -> np.ndarray:
    """Three ranks holding 1, 2 and 3 (one element each)."""
    return np.array([[1.0], [2.0], [3.0]], dtype=np.float32)


def normal_inputs(nranks: int, count: int, sigma: float, config: int) -> np.ndarray:
    return np.stack([(rng(config, r).standard_normal(count, dtype=np.float32) * np.float32(sigma))
                     for r in range(nranks)])


def bucket_inputs(nranks: int = 8, count: int = 6_553_600) -> np.ndarray:
    """Gradient-like f32 values, normal(0, 1e-3)."""
    return normal_inputs(nranks, count, 1e-3, CONFIG_BUCKET)


def large_rank(rank: int, count: int = 67_108_864, config: int = CONFIG_LARGE) -> np.ndarray:
    """One rank of the large bf16 workload: normal(0, 1), an independent 1% of
    entries scaled by 100; returned as uint16 bf16 bit patterns."""
    g = rng(config, rank)
    x = g.standard_normal(count, dtype=np.float32)
    mask = g.random(count, dtype=np.float32) < np.float32(0.01)
    x[mask] *= np.float32(100.0)
    return f32_to_bf16_bits_truncate(x)


def large_inputs(nranks: int = 8, count: int = 67_108_864, config: int = CONFIG_LARGE) -> np.ndarray:
    return np.stack([large_rank(r, count, config) for r in range(nranks)])


def gpt2_small_shapes() -> list[tuple[str, tuple[int, ...]]]:
    """Parameter shapes of GPT-2 small in registration order (148 tensors)."""
    d, v, ctx, layers = 768, 50257, 1024, 12
    shapes: list[tuple[str, tuple[int, ...]]] = [("wte", (v, d)), ("wpe", (ctx, d))]
    for i in range(layers):
        p = f"h.{i}."
        shapes += [
            (p + "ln_1.weight", (d,)), (p + "ln_1.bias", (d,)),
            (p + "attn.c_attn.weight", (d, 3 * d)), (p + "attn.c_attn.bias", (3 * d,)),
            (p + "attn.c_proj.weight", (d, d)), (p + "attn.c_proj.bias", (d,)),
            (p + "ln_2.weight", (d,)), (p + "ln_2.bias", (d,)),
            (p + "mlp.c_fc.weight", (d, 4 * d)), (p + "mlp.c_fc.bias", (4 * d,)),
            (p + "mlp.c_proj.weight", (4 * d, d)), (p + "mlp.c_proj.bias", (d,)),
        ]
    shapes += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    return shapes


def gpt2_small_counts() -> np.ndarray:
    return np.array([int(np.prod(s)) for _, s in gpt2_small_shapes()], dtype=np.int64)


def gpt2_rank_grads(rank: int, counts=None, sigma: float = 1e-4) -> list[np.ndarray]:
    """Rank `rank`'s gradients, one f32 array per tensor, normal(0, sigma)."""
    if counts is None:
        counts = gpt2_small_counts()
    g = rng(CONFIG_GPT2, rank)
    return [g.standard_normal(int(c), dtype=np.float32) * np.float32(sigma) for c in counts]


def sweep_points(dtypes=("f32", "bf16")):
    """(nranks, bytes per rank, dtype) for every sweep point within the cap."""
    pts = []
    for n in SWEEP_RANKS:
        for b in SWEEP_BYTES:
            if n * b <= SWEEP_CAP_BYTES:
                for dt in dtypes:
                    pts.append((n, b, dt))
    return pts


def uniform_rank(rank: int, count: int, dtype: str, config: int = CONFIG_SWEEP) -> np.ndarray:
    """One rank of uniform_inputs (same draws), for buffers too large to stack."""
    x = rng(config, rank).uniform(-1.0, 1.0, size=count).astype(np.float32)
    return f32_to_bf16_bits_truncate(x) if dtype == "bf16" else x


def uniform_rank_device(rank: int, count: int, dtype: str, torch, config: int = CONFIG_SWEEP, device="cuda"):
    """uniform(-1, 1) drawn on the device by torch's seeded generator, for
    buffers too large to draw on the host (not the same values as
    uniform_rank).  f32 as is; bf16 rounded to nearest and returned as int16
    bit patterns."""
    g = torch.Generator(device=device)
    g.manual_seed(BASE_SEED + 1000 * config + rank)
    x = torch.rand(count, generator=g, device=device, dtype=torch.float32).mul_(2.0).sub_(1.0)
    if dtype == "bf16":
        return x.to(torch.bfloat16).view(torch.int16)
    return x


def uniform_inputs(nranks: int, count: int, dtype: str, config: int = CONFIG_SWEEP) -> np.ndarray:
    """uniform(-1, 1) values; bf16 as truncated bit patterns, f16 as numpy's
    binary16 conversion of the binary32 draw."""
    xs = np.stack([rng(config, r).uniform(-1.0, 1.0, size=count).astype(np.float32) for r in range(nranks)])
    if dtype == "bf16":
        return f32_to_bf16_bits_truncate(xs)
    if dtype == "f16":
        return xs.astype(np.float16).view(np.uint16)
    if dtype == "i32":
        return np.stack([rng(config, r).integers(-(1 << 20), 1 << 20, size=count, dtype=np.int32)
                         for r in range(nranks)])
    return xs


def random_bits(nranks: int, count: int, dtype: str, seed: int) -> np.ndarray:
    """Arbitrary bit patterns (including NaN, infinities, subnormals, -0) for
    edge-case tests."""
    g = np.random.Generator(np.random.PCG64(seed))
    if dtype in ("bf16", "f16"):
        return g.integers(0, 1 << 16, size=(nranks, count), dtype=np.uint16)
    bits = g.integers(0, 1 << 32, size=(nranks, count), dtype=np.uint32)
    return bits.view(np.float32) if dtype == "f32" else bits.view(np.int32)

"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the averaging method: it only draws
random gradients and tensor-size lists of the shapes the pages' workloads
have.  Host arrays come from numpy ``default_rng([config, worker])`` (PCG64);
the largest configurations can be drawn on the device instead with a seeded
torch generator (see ``device_normal``), since drawing billions of normals on
the host would take minutes.

Workloads (sizes per worker; "N(0, v)" means variance v):

* ``partition_4mb``  -- P=4, one 4 MB partition (N = 2^20 fp32), N(0, 1), the
  THC microbenchmark's partition size; THC with b = 4.
* ``resnet_fusion``  -- P=8, 300 fp32 tensors with log-uniform sizes in
  [256, 2.4M] scaled to about 45M parameters (a ResNet-101-like many-small-
  tensors model), N(0, 0.01), 64 MB fusion buffers.
* ``vgg_fusion``     -- P=8, 16 fp32 tensors totalling 138M parameters, the
  largest 102,760,448 (a VGG-16-like communication-bound model), N(0, 1e-3).
* ``thc_sweep``      -- N = 2^24 fp32 Student-t(3) x 1e-3, P in {4, 16, 64},
  b in {2, 4, 8}.
* ``large_bf16``     -- P=16, N = 2^28 bf16 N(0, 1e-2) per worker.
"""
from __future__ import annotations

import math

import numpy as np

CONFIG_IDS = {
    "partition_4mb": 1,
    "resnet_fusion": 2,
    "vgg_fusion": 3,
    "thc_sweep": 4,
    "large_bf16": 5,
}

THC_SEED = 0x5EED


def rng(config: int, worker: int) -> np.random.Generator:
    return np.random.default_rng([config, worker])


def normal_f32(n: int, var: float, config: int, worker: int) -> np.ndarray:
    g = rng(config, worker)
    x = g.standard_normal(n, dtype=np.float32)
    if var != 1.0:
        x *= np.float32(math.sqrt(var))
    return x


def student_t_f32(n: int, nu: float, scale: float, config: int, worker: int) -> np.ndarray:
    g = rng(config, worker)
    return (g.standard_t(nu, size=n) * scale).astype(np.float32)


def workers_normal(p: int, n: int, var: float, config: int):
    return [normal_f32(n, var, config, w) for w in range(p)]


def log_uniform_sizes(count: int, lo: int, hi: int, total: int, seed_pair) -> np.ndarray:
    """``count`` sizes drawn log-uniform in [lo, hi], scaled toward ``total``,
    then clamped to [lo, hi] (so the real total is close to, not exactly, it)."""
    g = np.random.default_rng(list(seed_pair))
    raw = np.exp(g.uniform(math.log(lo), math.log(hi), size=count))
    raw = raw * (total / raw.sum())
    return np.clip(np.rint(raw), lo, hi).astype(np.int64)


def resnet_fusion_sizes() -> np.ndarray:
    """300 tensor sizes, about 45M parameters in all."""
    return log_uniform_sizes(300, 256, 2_400_000, 45_000_000, (2, 999))


def vgg_fusion_sizes() -> np.ndarray:
    """16 tensor sizes: 102,760,448 plus 15 log-uniform ones, 138,000,000 in all."""
    big = 102_760_448
    rest_total = 138_000_000 - big
    rest = log_uniform_sizes(15, 1_728, 16_777_216, rest_total, (3, 999))
    # put the remainder on the last small tensor so the total is exact
    rest[-1] += rest_total - int(rest.sum())
    sizes = np.concatenate([rest[:12], [big], rest[12:]]).astype(np.int64)
    return sizes


def tensors_normal(sizes, var: float, config: int, worker: int):
    """One worker's list of gradient tensors: a single stream cut into pieces."""
    flat = normal_f32(int(np.sum(sizes)), var, config, worker)
    out, pos = [], 0
    for s in sizes:
        out.append(flat[pos:pos + int(s)].copy())
        pos += int(s)
    return out


def device_normal(shape, var: float, seed: int, dtype, device):
    """Seeded normal draws made on the device (large workloads only)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if var != 1.0:
        x.mul_(math.sqrt(var))
    return x.to(dtype)


def device_student_t(n: int, nu: int, scale: float, seed: int, device):
    """Seeded Student-t(nu) draws (integer nu) made on the device:
    Z / sqrt(chi2_nu / nu) with chi2_nu a sum of nu squared normals."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(n, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi2.addcmul_(*(2 * [torch.randn(n, generator=g, device=device, dtype=torch.float32)]))
    return (z / torch.sqrt(chi2 / nu) * scale).to(torch.float32)

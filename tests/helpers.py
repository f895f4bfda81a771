"""Shared helpers for the GPU parity tests (marshalling between numpy and torch)."""
import numpy as np
import pytest


def need_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import gradient_allreduce_homomorphic_gb300 as g

    g.load()  # raises if libgar.so is missing: no fallback
    return torch, g


def to_dev(a, torch, dev="cuda"):
    if a.dtype == np.uint16:  # bf16 bit patterns
        return torch.from_numpy(a.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def to_host(t):
    import torch

    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.cpu().numpy().view(np.uint32)
    if t.dtype == torch.int16:
        return t.cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_bits(x32, torch):
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def same_bits(a, b):
    """Bit equality, except that any NaN matches any NaN (payloads are not specified)."""
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape
    if a.dtype == np.float32:
        au, bu = a.view(np.uint32), b.view(np.uint32)
        nan = np.isnan(a) & np.isnan(b)
    elif a.dtype == np.uint16:
        au, bu = a, b
        fa = (a.astype(np.uint32) << 16).view(np.float32)
        fb = (b.astype(np.uint32) << 16).view(np.float32)
        nan = np.isnan(fa) & np.isnan(fb)
    else:
        au, bu, nan = a, b, np.zeros(a.shape, bool)
    bad = (au != bu) & ~nan
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{int(bad.sum())} of {a.size} differ; first at {i}: {a.flat[i]!r} vs {b.flat[i]!r}")

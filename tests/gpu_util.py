"""Helpers for the GPU tests: host <-> device marshalling and comparisons."""
from __future__ import annotations

import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns (any shape) -> contiguous CUDA bfloat16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 CUDA tensor -> uint16 numpy bit patterns."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_float(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.ascontiguousarray(got).ravel()
    want = np.ascontiguousarray(want).ravel()
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    g8, w8 = got.view(np.uint8), want.view(np.uint8)
    if not np.array_equal(g8, w8):
        bad = np.nonzero(got.view(np.uint8 if got.itemsize == 1 else
                                  {2: np.uint16, 4: np.uint32}[got.itemsize]) !=
                         want.view(np.uint8 if want.itemsize == 1 else
                                   {2: np.uint16, 4: np.uint32}[want.itemsize]))[0]
        raise AssertionError(f"{what}: {len(bad)} of {got.size} differ, first at {bad[:5]}: "
                             f"got {got[bad[:5]]} want {want[bad[:5]]}")


# (test, what, elements, max |dy| in units of the oracle's bf16 ulp, bit-exact fraction)
# for every y comparison of the session; conftest.py prints them at the end.
Y_STATS = []


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    """One bf16 ulp at each value: 2^(e - 7) for |y| in [2^e, 2^(e+1)),
    2^-133 (the subnormal spacing) below 2^-126, and 0 at y == 0."""
    y = np.abs(np.asarray(y, np.float64))
    _, ex = np.frexp(y)  # y = m * 2^ex, m in [0.5, 1): e = ex - 1
    e = np.maximum(ex - 1, -126)
    return np.where(y == 0, 0.0, np.ldexp(1.0, e - 7))


def assert_y_close(y_gpu_bits: np.ndarray, y_or_bits: np.ndarray, what="y"):
    """bf16 outputs within one bf16 ulp of the oracle: |dy| <= ulp_bf16(y_oracle),
    the spacing of bf16 values at the oracle's exponent (exact where the oracle
    gives 0).  Records the largest error in ulps and the bit-exact fraction in
    Y_STATS; returns the fraction that is bit-exact."""
    import os
    g = bf16_float(y_gpu_bits).astype(np.float64).ravel()
    w = bf16_float(y_or_bits).astype(np.float64).ravel()
    ulp = bf16_ulp(w)
    err = np.abs(g - w)
    bad = np.nonzero(err > ulp)[0]
    assert len(bad) == 0, (f"{what}: {len(bad)} of {g.size} beyond 1 bf16 ulp, first "
                           f"{bad[:5]}: got {g[bad[:5]]} want {w[bad[:5]]}")
    nz = ulp > 0
    max_ulp = float(np.max(err[nz] / ulp[nz])) if np.any(nz) else 0.0
    exact = float(np.mean(np.asarray(y_gpu_bits).ravel() == np.asarray(y_or_bits).ravel()))
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    Y_STATS.append((test, what, int(g.size), max_ulp, exact))
    return exact

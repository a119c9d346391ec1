"""Comparison helpers for the GPU parity tests (GPU output vs the CPU oracle)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor (any device) -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_tolerance_violations(gpu_bits: np.ndarray, ref: np.ndarray, K: int) -> np.ndarray:
    """Mask of elements outside |C_gpu - R| <= ulp(R) + 1e-4 * sqrt(K), R = bf16_rne(C_ref).

    The bound: every element within one BF16 ulp of the oracle value rounded to BF16, plus
    1e-4 * sqrt(K) absolute (FP32 accumulation order is not specified).
    """
    R = oracle.round_bf16(ref)
    g = oracle.bf16_bits_to_f64(gpu_bits)
    r = oracle.bf16_bits_to_f64(R)
    tol = oracle.ulp_bf16(R) + 1e-4 * math.sqrt(K)
    return ~(np.abs(g - r) <= tol)


def assert_bf16_close(gpu_bits: np.ndarray, ref: np.ndarray, K: int, what: str = "") -> None:
    bad = bf16_tolerance_violations(gpu_bits, ref, K)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        R = oracle.bf16_bits_to_f64(oracle.round_bf16(ref))
        g = oracle.bf16_bits_to_f64(gpu_bits)
        detail = ", ".join(f"{tuple(i)}: gpu {g[tuple(i)]!r} oracle {R[tuple(i)]!r}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; {detail}")


def assert_bf16_exact(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    """Bit-exact by value (+0 == -0) against the oracle rounded to BF16."""
    R = oracle.bf16_bits_to_f64(oracle.round_bf16(ref))
    g = oracle.bf16_bits_to_f64(gpu_bits)
    bad = g != R
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: gpu {g[tuple(i)]!r} oracle {R[tuple(i)]!r}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements differ; {detail}")


def assert_nvfp4_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    """max |C_gpu - C_ref| <= 1e-2 * max |C_ref| over all compared elements."""
    g = oracle.bf16_bits_to_f64(gpu_bits)
    err = float(np.max(np.abs(g - ref))) if ref.size else 0.0
    bound = 1e-2 * float(np.max(np.abs(ref))) if ref.size else 0.0
    if not err <= bound:
        raise AssertionError(f"{what}: max |C_gpu - C_ref| = {err} > 1e-2 * max|C_ref| = {bound}")


def sample_coords(M: int, N: int, n: int, seed: int = 0):
    """n random output coordinates plus the four corners and the last row / column edges."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    edge = [(0, 0), (0, N - 1), (M - 1, 0), (M - 1, N - 1)]
    edge += [(M - 1, int(c)) for c in rng.integers(0, N, 64)] + [(int(r), N - 1) for r in rng.integers(0, M, 64)]
    rows += [e[0] for e in edge]
    cols += [e[1] for e in edge]
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)

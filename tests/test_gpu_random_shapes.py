"""Seeded random shapes and option combinations through the C ABI against the oracle.

Each case draws M, N, K (ragged, within the layout rules: N % 8 == 0, BF16 K % 8 == 0,
NVFP4 K % 256 == 0) and a set of options: the scheduler (static, CLC), the kernel
variant, a cluster cap, one tile per cluster, swap-AB and split-K switches and the tail
split. Together they reach the swapped few-row path with and without K splits (through
the reduction kernel or a cluster of two CTA pairs), split tails, CLC cancellations, the
512 x 256 BF16 tile (plain and fused), few-row NVFP4 GEMMs with and without the padded copy
of A, and ragged edges in every dimension. Sizes stay small enough for the oracle to take about a
second per case.
"""
import numpy as np
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import oracle
import synthetic_inputs as si
from dense_tensor_core_persistent_gb300 import build as gbuild
from parity import assert_bf16_close, assert_nvfp4_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def setup():
    if DEV is None:
        pytest.skip("needs a CUDA GPU")
    gbuild.build()
    oracle.build()
    torch.cuda.set_device(DEV)
    yield
    st, detail = g.get_device_status()
    assert st == g.GEMM_OK, f"a kernel reported status {st} ({detail:#x})"


def bf16_case(seed):
    rng = np.random.default_rng(1000 + seed)
    few_rows = rng.random() < 0.35
    M = int(rng.integers(1, 129)) if few_rows else int(rng.integers(1, 700))
    N = 8 * int(rng.integers(1, 200 if not few_rows else 1025))
    K = 8 * int(rng.integers(1, 257 if not few_rows else 1025))
    opts = dict(
        clc=int(rng.choice([g.GEMM_CLC_AUTO, g.GEMM_CLC_ON, g.GEMM_CLC_OFF])),
        kernel=int(rng.choice([g.GEMM_KERNEL_DEFAULT, g.GEMM_KERNEL_DEFAULT, g.GEMM_KERNEL_BF16_1CTA,
                               g.GEMM_KERNEL_BF16_2CTA_K64, g.GEMM_KERNEL_BF16_2CTA_WIDE])),
        max_clusters=int(rng.choice([0, 0, 0, 1, 3, 7])),
        persistent=int(rng.choice([1, 1, 1, 0])),
        no_swap_ab=int(rng.random() < 0.15),
        no_split_k=int(rng.random() < 0.15),
        no_tail_split=int(rng.random() < 0.15),
    )
    if opts["kernel"] == g.GEMM_KERNEL_BF16_2CTA_WIDE and opts["clc"] == g.GEMM_CLC_ON:
        opts["clc"] = g.GEMM_CLC_AUTO  # the 512 x 256 tile has a static schedule only
    return M, N, K, opts


@pytest.mark.parametrize("seed", range(64))
def test_bf16_random_shape_and_options(seed):
    M, N, K, opts = bf16_case(seed)
    if M * N * K > 1.5e9:  # keep the oracle to about a second
        K = max(8, int(1.5e9 / (M * N)) // 8 * 8)
    A, B = si.bf16_problem(seed, M, N, K)
    C = g.matmul_bf16(A.to(DEV), B.to(DEV), opts=g.options(**opts))
    torch.cuda.synchronize()
    assert_bf16_close(bits(C), oracle.gemm_bf16(A, B), K, f"{M}x{N}x{K} {opts}")


@pytest.mark.parametrize("seed", range(32))
def test_nvfp4_random_shape_and_options(seed):
    rng = np.random.default_rng(2000 + seed)
    M = int(rng.integers(1, 32)) if seed % 4 == 3 else int(rng.integers(1, 600))  # a quarter with few rows
    N = 8 * int(rng.integers(1, 120))
    K = 256 * int(rng.integers(1, 9))
    opts = dict(clc=int(rng.choice([g.GEMM_CLC_AUTO, g.GEMM_CLC_ON])), max_clusters=int(rng.choice([0, 0, 2, 5])),
                persistent=int(rng.choice([1, 1, 0])), no_tail_split=int(rng.random() < 0.2),
                no_pad_a=int(rng.random() < 0.3))
    a, sfa, b, sfb = si.nvfp4_problem(seed, M, N, K)
    C = g.matmul_nvfp4(a.to(DEV), sfa.to(DEV), b.to(DEV), sfb.to(DEV), opts=g.options(**opts))
    torch.cuda.synchronize()
    assert_nvfp4_close(bits(C), oracle.gemm_nvfp4(a, sfa, b, sfb), f"{M}x{N}x{K} {opts}")


@pytest.mark.parametrize("seed", range(16))
def test_bf16_fused_random_shape_and_epilogue(seed):
    from test_gpu_fused import assert_fused_close, bias_bits, prior_c, run_bf16_fused
    rng = np.random.default_rng(3000 + seed)
    M = int(rng.integers(1, 600))
    N = 8 * int(rng.integers(1, 150))
    K = 8 * int(rng.integers(1, 200))
    alpha = float(rng.choice([1.0, 0.5, -1.25]))
    beta = float(rng.choice([0.0, 1.0, -0.5]))
    act = int(rng.choice([g.GEMM_ACT_NONE, g.GEMM_ACT_RELU, g.GEMM_ACT_GELU_TANH]))
    bias = bias_bits(N, 3100 + seed) if rng.random() < 0.5 else None
    c_old = prior_c(M, N, 3200 + seed)
    kernel = int(rng.choice([g.GEMM_KERNEL_DEFAULT, g.GEMM_KERNEL_BF16_2CTA_WIDE]))
    clc = int(rng.choice([g.GEMM_CLC_AUTO, g.GEMM_CLC_ON])) if kernel == g.GEMM_KERNEL_DEFAULT else g.GEMM_CLC_AUTO
    opts = g.options(clc=clc, max_clusters=int(rng.choice([0, 3])), kernel=kernel)
    A, B = si.bf16_problem(3300 + seed, M, N, K)
    got = run_bf16_fused(A, B, c_old, alpha, beta, bias, act, opts=opts)
    assert_fused_close(got, oracle.gemm_bf16(A, B), alpha, beta, c_old, bias, act, K, f"{M}x{N}x{K}")

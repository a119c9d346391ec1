"""Size extremes, checked on every output element through properties that hold at any size.

All-ones operands give C = K exactly (every partial sum is an integer below 2^24, and K is
a power of two, exact in BF16). Deep K runs the stage rings through hundreds of phases;
wide grids run thousands of work items through the static and the CLC schedules; the
few-row path runs with its deepest K splits.
"""
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
from dense_tensor_core_persistent_gb300 import build as gbuild

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def setup():
    if DEV is None:
        pytest.skip("needs a CUDA GPU")
    gbuild.build()
    torch.cuda.set_device(DEV)
    yield
    st, detail = g.get_device_status()
    assert st == g.GEMM_OK, f"a kernel reported status {st} ({detail:#x})"


def ones_bf16(rows, K):
    return torch.ones(rows, K, dtype=torch.bfloat16, device=DEV)


@pytest.mark.parametrize("opts", [dict(), dict(clc=g.GEMM_CLC_ON), dict(kernel=g.GEMM_KERNEL_BF16_1CTA),
                                  dict(kernel=g.GEMM_KERNEL_BF16_2CTA_K64)], ids=["default", "clc", "1cta", "k64"])
def test_bf16_deep_k_all_ones(opts):
    M, N, K = 512, 768, 65536   # 512 stages of 128 K per tile
    C = g.matmul_bf16(ones_bf16(M, K), ones_bf16(N, K), opts=g.options(**opts))
    torch.cuda.synchronize()
    assert torch.all(C == float(K)).item()


@pytest.mark.parametrize("M", [1, 64, 128])
def test_bf16_few_rows_deep_k_all_ones(M):
    N, K = 8192, 65536          # swapped, K split over several clusters (or two pairs per cluster)
    C = g.matmul_bf16(ones_bf16(M, K), ones_bf16(N, K))
    torch.cuda.synchronize()
    assert torch.all(C == float(K)).item()


@pytest.mark.parametrize("clc", [g.GEMM_CLC_OFF, g.GEMM_CLC_ON])
def test_bf16_wide_grid_all_ones(clc):
    M, N, K = 32768, 16384, 64  # 8192 tiles: over 100 waves of the co-resident pairs
    C = g.matmul_bf16(ones_bf16(M, K), ones_bf16(N, K), opts=g.options(clc=clc))
    torch.cuda.synchronize()
    assert torch.all(C == float(K)).item()


def test_nvfp4_deep_k_all_ones():
    M, N, K = 512, 768, 65536   # 256 stages of 256 K; every code 1.0 (0x2), every scale 1.0 (0x38)
    a = torch.full((M, K // 2), 0x22, dtype=torch.uint8, device=DEV)
    b = torch.full((N, K // 2), 0x22, dtype=torch.uint8, device=DEV)
    sfa = torch.full((M, K // 16), 0x38, dtype=torch.uint8, device=DEV)
    sfb = torch.full((N, K // 16), 0x38, dtype=torch.uint8, device=DEV)
    for opts in (None, g.options(clc=g.GEMM_CLC_ON)):
        C = g.matmul_nvfp4(a, sfa, b, sfb, opts=opts)
        torch.cuda.synchronize()
        assert torch.all(C == float(K)).item()

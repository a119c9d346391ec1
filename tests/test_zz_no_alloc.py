"""gemm_nvfp4_noalloc: the NVFP4 GEMM for callers that must not let the library allocate.

Some callers cannot have a library allocate device memory on their behalf (code running
inside their own allocator, or applications that account for every byte of device memory
themselves). gemm_nvfp4 takes its scale workspace from a memory pool; gemm_nvfp4_noalloc
uses a fixed 16 MiB array compiled into the library instead. This file checks, through
the C ABI, that the no-allocation entry point gives the same result as gemm_nvfp4 on two
calls in a row (the second call reuses the array the first one left behind), that both
calls also agree with the CPU oracle (so that a fault shared by the two entry points, which
run the same packing and GEMM kernels, cannot pass), that unit scales give the oracle's
exact result bit for bit, and that a problem too large for the array is refused before
anything is launched.

It sits in a file of its own that pytest collects last, and works both alone in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import oracle
import synthetic_inputs as si
from dense_tensor_core_persistent_gb300 import build as gbuild
from parity import assert_bf16_exact, assert_nvfp4_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def setup():
    if DEV is None:
        pytest.skip("needs a CUDA GPU")
    gbuild.build()
    oracle.build()
    torch.cuda.set_device(DEV)


E4M3_ONE = 0x38


def _both(seed, M, N, K, unit_scales=False):
    a, sfa, b, sfb = si.nvfp4_problem(seed, M, N, K, device=DEV)
    if unit_scales:
        sfa = torch.full((M, K // 16), E4M3_ONE, dtype=torch.uint8, device=DEV)
        sfb = torch.full((N, K // 16), E4M3_ONE, dtype=torch.uint8, device=DEV)
    want = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    g.gemm_nvfp4(a, sfa, b, sfb, want, M, N, K)
    before = g.launch_count()
    g.gemm_nvfp4_noalloc(a, sfa, b, sfb, got, M, N, K)
    torch.cuda.synchronize()
    assert g.launch_count() == before + 2  # scale packing (SFA and SFB together), GEMM
    ref = oracle.gemm_nvfp4(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu())
    return bits(got), want.cpu().double().numpy(), ref


def test_noalloc_matches_gemm_nvfp4_on_two_calls_in_a_row():
    # first call: a larger problem fills more of the scratch array; the second call, with
    # different shapes and ragged M / N, must not be affected by what the first left there
    for seed, (M, N, K) in [(50, (1024, 768, 2048)), (51, (300, 264, 1024))]:
        got, want, ref = _both(seed, M, N, K)
        assert_nvfp4_close(got, want, f"noalloc vs gemm_nvfp4 {M}x{N}x{K}")
        assert_nvfp4_close(got, ref, f"noalloc vs oracle {M}x{N}x{K}")
    assert g.get_device_status()[0] == g.GEMM_OK


def test_noalloc_unit_scales_bit_exact_on_two_calls_in_a_row():
    # all scales 1.0: every product is a multiple of 1/4 and |sums| <= 36 K, exact in FP32,
    # so both calls must equal the oracle's BF16 rounding bit for bit
    for seed, (M, N, K) in [(52, (640, 512, 1024)), (53, (129, 136, 512))]:
        got, _, ref = _both(seed, M, N, K, unit_scales=True)
        assert_bf16_exact(got, ref, f"noalloc unit scales {M}x{N}x{K}")
    assert g.get_device_status()[0] == g.GEMM_OK


def test_noalloc_few_rows_on_two_calls_in_a_row():
    # fewer than 32 rows: A is copied into the array too (after the scales), padded to 32
    # rows; the second call, with fewer rows, finds the first call's rows past its own M
    for seed, (M, N, K) in [(54, (20, 1024, 2048)), (55, (3, 264, 512))]:
        got, want, ref = _both(seed, M, N, K)
        assert np.array_equal(got, bits_of(want)), f"noalloc vs gemm_nvfp4 {M}x{N}x{K}"
        assert_nvfp4_close(got, ref, f"noalloc vs oracle {M}x{N}x{K}")
    assert g.get_device_status()[0] == g.GEMM_OK


def bits_of(values: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of values that are BF16 numbers (exact conversion)."""
    return bits(torch.from_numpy(values).to(torch.bfloat16))


def test_noalloc_rejects_problems_larger_than_its_scratch():
    K = 16384
    # M = N = 8192 at K = 16384 fills the 16 MiB exactly; one more row block does not fit
    M, N = 8192 + 128, 8192
    C = torch.empty(8, dtype=torch.bfloat16, device=DEV)  # never touched: refused on the host
    dummy = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_nvfp4_noalloc(dummy, dummy, dummy, dummy, C, M, N, K)
    assert e.value.status == g.GEMM_ERR_SCRATCH_TOO_SMALL
    blocked = g.nvfp4_blocked_scale_bytes(8192, K) * 2
    assert blocked == g.NVFP4_NOALLOC_SCRATCH_BYTES

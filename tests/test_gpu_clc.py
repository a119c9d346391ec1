"""Cluster launch control (dynamic tile scheduling) through the C ABI against the oracle.

With gemm_options_t.clc = 1 the grid has one cluster per work item; the clusters that run
take the items of clusters they cancel before those start. The shapes here have more items
than co-resident clusters (so cancellations happen), fewer (the first cancellation fails),
tail waves cut into halves and K splits of the swapped path.
"""
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import oracle
import synthetic_inputs as si
from dense_tensor_core_persistent_gb300 import build as gbuild
from parity import assert_bf16_close, assert_bf16_exact, assert_nvfp4_close, bits, sample_coords

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
CLC = g.GEMM_CLC_ON


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


def run(A, B, **opt):
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = g.matmul_bf16(Ad, Bd, opts=g.options(**opt))
    torch.cuda.synchronize()
    return bits(C)


# (M, N, K): 108 tiles of 256 x 256 (more than the co-resident pairs), a ragged edge in
# every dimension, and one wave or less
SHAPES = [(2304, 3072, 192), (2056, 3080, 136), (1000, 1000, 64), (256, 256, 256)]
KERNELS = [g.GEMM_KERNEL_BF16_2CTA, g.GEMM_KERNEL_BF16_2CTA_K64, g.GEMM_KERNEL_BF16_1CTA]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_clc_against_oracle(kernel, shape):
    M, N, K = shape
    A, B = si.bf16_problem(M + N + K, M, N, K)
    assert_bf16_close(run(A, B, kernel=kernel, clc=CLC), oracle.gemm_bf16(A, B), K, f"clc {shape}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_clc_integer_inputs_bit_exact(kernel):
    M, N, K = 2304, 3072, 192
    A, B = si.bf16_problem(5, M, N, K, kind="int")
    assert_bf16_exact(run(A, B, kernel=kernel, clc=CLC), oracle.gemm_bf16(A, B), "clc integer")


def test_clc_and_static_agree_bit_for_bit():
    # the schedule only decides which cluster computes a tile, never how
    M, N, K = 4096, 4352, 512
    A, B = si.bf16_problem(6, M, N, K, device=DEV)
    c_static = bits(g.matmul_bf16(A, B, opts=g.options(clc=g.GEMM_CLC_OFF)))
    c_clc = bits(g.matmul_bf16(A, B, opts=g.options(clc=CLC)))
    torch.cuda.synchronize()
    assert (c_static == c_clc).all()


def test_clc_with_split_tail_wave():
    # 96 tiles on 76 pairs: the last 20 tiles are cut into halves (116 work items)
    M, N, K = 2048, 3072, 128
    assert 96 == (M // 256) * (N // 256)
    A, B = si.bf16_problem(7, M, N, K)
    ref = oracle.gemm_bf16(A, B)
    assert_bf16_close(run(A, B, clc=CLC), ref, K, "clc tail split")
    assert_bf16_close(run(A, B, clc=CLC, no_tail_split=1), ref, K, "clc no tail split")


@pytest.mark.parametrize("shape", [(64, 40960, 256), (16, 1024, 8192), (100, 2048, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_clc_few_rows_swapped(shape):
    # 160 swapped tiles of 256 rows; K splits (work items = tiles x splits, one wave)
    M, N, K = shape
    A, B = si.bf16_problem(M + N, M, N, K)
    assert_bf16_close(run(A, B, clc=CLC), oracle.gemm_bf16(A, B), K, f"clc swapped {shape}")


def test_clc_fused_epilogue():
    from test_gpu_fused import assert_fused_close, bias_bits, prior_c, run_bf16_fused
    M, N, K = 2304, 3072, 192
    A, B = si.bf16_problem(8, M, N, K)
    bias, c_old = bias_bits(N, 9), prior_c(M, N, 10)
    got = run_bf16_fused(A, B, c_old, 0.5, -1.0, bias, g.GEMM_ACT_RELU, opts=g.options(clc=CLC))
    static = run_bf16_fused(A, B, c_old, 0.5, -1.0, bias, g.GEMM_ACT_RELU, opts=g.options(clc=g.GEMM_CLC_OFF))
    assert (got == static).all()
    assert_fused_close(got, oracle.gemm_bf16(A, B), 0.5, -1.0, c_old, bias, g.GEMM_ACT_RELU, K, "clc fused")


def test_clc_full_size_sampled():
    M = N = K = 8192
    A, B = si.bf16_problem(2, M, N, K, device=DEV)
    C = g.matmul_bf16(A, B, opts=g.options(clc=CLC))
    torch.cuda.synchronize()
    rows, cols = sample_coords(M, N, 4096, 2)
    ref = oracle.gemm_bf16_at(A.cpu(), B.cpu(), rows, cols)
    assert_bf16_close(bits(C)[rows, cols], ref, K, "clc 8192^3")


def test_clc_nvfp4_against_oracle():
    M, N, K = 2304, 3072, 512
    a, sfa, b, sfb = si.nvfp4_problem(11, M, N, K)
    C = g.matmul_nvfp4(a.to(DEV), sfa.to(DEV), b.to(DEV), sfb.to(DEV), opts=g.options(clc=CLC))
    torch.cuda.synchronize()
    assert_nvfp4_close(bits(C), oracle.gemm_nvfp4(a, sfa, b, sfb), "clc nvfp4")


def test_clc_nvfp4_fused_and_static_agree():
    from test_gpu_fused import bias_bits, prior_c, to_dev_bf16
    M, N, K = 2304, 3072, 512
    a, sfa, b, sfb = (t.to(DEV) for t in si.nvfp4_problem(13, M, N, K))
    bias = to_dev_bf16(bias_bits(N, 14))
    c_old = to_dev_bf16(prior_c(M, N, 15))
    outs = []
    for mode in (CLC, g.GEMM_CLC_OFF):
        C = c_old.clone()
        g.gemm_nvfp4_fused(a, sfa, b, sfb, C, M, N, K, g.epilogue(0.75, 0.5, bias, g.GEMM_ACT_GELU_TANH),
                           opts=g.options(clc=mode))
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_clc_nvfp4_deep_k_sampled():
    # K = 16384 (64 stages per item) with more tiles than co-resident pairs
    M, N, K = 2304, 3072, 16384
    a, sfa, b, sfb = si.nvfp4_problem(16, M, N, K)
    C = g.matmul_nvfp4(a.to(DEV), sfa.to(DEV), b.to(DEV), sfb.to(DEV), opts=g.options(clc=CLC))
    torch.cuda.synchronize()
    rows, cols = sample_coords(M, N, 2048, 16)
    assert_nvfp4_close(bits(C)[rows, cols], oracle.gemm_nvfp4_at(a, sfa, b, sfb, rows, cols), "nvfp4 deep K")


def test_clc_bf16_deep_k_default_schedule():
    # the default options take the CLC order here (BF16, 108 tiles, K = 16384)
    M, N, K = 2304, 3072, 16384
    assert g.clc_rule(108, 76, K)
    A, B = si.bf16_problem(18, M, N, K, device=DEV)
    C = g.matmul_bf16(A, B)
    C_static = g.matmul_bf16(A, B, opts=g.options(clc=g.GEMM_CLC_OFF))
    torch.cuda.synchronize()
    assert torch.equal(C, C_static)
    rows, cols = sample_coords(M, N, 2048, 18)
    assert_bf16_close(bits(C)[rows, cols], oracle.gemm_bf16_at(A.cpu(), B.cpu(), rows, cols), K, "bf16 deep K")


def test_clc_nvfp4_bounded_wait_reports_timeout():
    g.get_device_status()
    M, N, K = 2304, 3072, 512
    a, sfa, b, sfb = (t.to(DEV) for t in si.nvfp4_problem(17, M, N, K))
    g.matmul_nvfp4(a, sfa, b, sfb, opts=g.options(clc=CLC, wait_limit_us=100_000, debug_flags=1))
    st, _ = g.get_device_status()
    assert st == g.GEMM_ERR_TIMEOUT
    C = g.matmul_nvfp4(a, sfa, b, sfb, opts=g.options(clc=CLC))
    C_static = g.matmul_nvfp4(a, sfa, b, sfb, opts=g.options(clc=g.GEMM_CLC_OFF))
    torch.cuda.synchronize()
    assert torch.equal(C, C_static)
    assert g.get_device_status()[0] == g.GEMM_OK


def test_clc_back_to_back_on_one_stream():
    M, N, K = 2304, 3072, 192
    A, B = si.bf16_problem(12, M, N, K, device=DEV)
    ref = g.matmul_bf16(A, B, opts=g.options(clc=g.GEMM_CLC_OFF))
    outs = [g.matmul_bf16(A, B, opts=g.options(clc=CLC)) for _ in range(20)]
    torch.cuda.synchronize()
    for C in outs:
        assert torch.equal(C, ref)


def test_clc_bounded_wait_reports_timeout_and_context_survives():
    """The MMA issuer waits on a barrier nothing arrives on (debug flag 1), in a grid with
    more clusters than can run at once: every wait is bounded, the status records the
    timeout, and the next GEMM on the context is correct."""
    g.get_device_status()
    A, B = si.bf16_problem(0, 2304, 3072, 192, device=DEV)
    g.matmul_bf16(A, B, opts=g.options(clc=CLC, wait_limit_us=100_000, debug_flags=1))
    st, detail = g.get_device_status()
    assert st == g.GEMM_ERR_TIMEOUT
    A2, B2 = si.bf16_problem(1, 2304, 3072, 192)
    assert_bf16_close(run(A2, B2, clc=CLC), oracle.gemm_bf16(A2, B2), 192, "after timeout")
    assert g.get_device_status()[0] == g.GEMM_OK


def test_clc_option_defers_to_capped_and_one_tile_per_cluster_grids():
    # CLC applies to uncapped persistent grids; with a cluster cap or one cluster per tile
    # the request is ignored and the static walk runs
    M, N, K = 2304, 3072, 192
    A, B = si.bf16_problem(19, M, N, K)
    ref = oracle.gemm_bf16(A, B)
    assert_bf16_close(run(A, B, clc=CLC, max_clusters=5), ref, K, "clc with a cluster cap")
    assert_bf16_close(run(A, B, clc=CLC, persistent=0), ref, K, "clc with one cluster per tile")


def test_clc_call_is_one_launch():
    A, B = si.bf16_problem(20, 2304, 3072, 192, device=DEV)
    torch.cuda.synchronize()
    before = g.launch_count()
    g.matmul_bf16(A, B, opts=g.options(clc=CLC))
    torch.cuda.synchronize()
    assert g.launch_count() == before + 1

"""The C-ABI library without a GPU: exports, argument checks, tile order (no compute)."""
import itertools
import os
import re

import pytest

import dense_tensor_core_persistent_gb300 as g
from dense_tensor_core_persistent_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "gemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w ]+?\*?\s*\b(gemm_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_function():
    declared = _header_functions()
    assert len(declared) >= 9
    l = g.lib()
    for name in declared:
        assert hasattr(l, name), name
    assert sorted(declared) == sorted(g.EXPORTS)


def test_status_strings():
    for code in range(9):
        assert g.status_string(code)
    assert g.status_string(8) == "device wait timed out"
    assert g.status_string(99) == "unknown status"


def test_argument_errors_are_reported_before_any_device_use():
    l = g.lib()
    assert l.gemm_bf16(0, 0, 0, 0, 8, 8, 0) == g.GEMM_OK            # M == 0: nothing to do
    assert l.gemm_bf16(0, 0, 0, 8, 0, 8, 0) == g.GEMM_OK            # N == 0
    assert l.gemm_bf16(0, 0, 0, -1, 8, 8, 0) == g.GEMM_ERR_INVALID_ARG
    assert l.gemm_bf16(0, 0, 0, 8, 8, 8, 0) == g.GEMM_ERR_INVALID_ARG  # null pointers
    assert l.gemm_bf16(16, 16, 16, 8, 8, 12, 0) == g.GEMM_ERR_UNSUPPORTED_SHAPE  # K % 8
    assert l.gemm_bf16(16, 16, 16, 8, 12, 8, 0) == g.GEMM_ERR_UNSUPPORTED_SHAPE  # N % 8
    assert l.gemm_bf16(16, 24, 8, 8, 8, 8, 0) == g.GEMM_ERR_MISALIGNED
    assert l.gemm_nvfp4(16, 16, 16, 16, 16, 8, 8, 128, 0) == g.GEMM_ERR_UNSUPPORTED_SHAPE  # K % 256
    assert l.gemm_nvfp4(16, 16, 16, 0, 16, 8, 8, 256, 0) == g.GEMM_ERR_INVALID_ARG
    # sizes near INT_MAX: the row-block counts are far beyond what a launch can hold, and
    # their computation must not overflow into a negative count that passes the check
    big = 2**31 - 1
    assert l.gemm_nvfp4(16, 16, 16, 16, 16, big, 8, 256, 0) == g.GEMM_ERR_UNSUPPORTED_SHAPE
    assert l.gemm_nvfp4(16, 16, 16, 16, 16, 8, big - 7, 256, 0) == g.GEMM_ERR_UNSUPPORTED_SHAPE
    assert l.gemm_nvfp4_noalloc(16, 16, 16, 16, 16, big, 8, 256, 0) == g.GEMM_ERR_UNSUPPORTED_SHAPE
    o = g.options()
    o.clc = 3
    with pytest.raises(g.GemmError):
        g.gemm_bf16(16, 16, 16, 8, 8, 8, 0, o)
    with pytest.raises(g.GemmError):
        g.gemm_nvfp4(16, 16, 16, 16, 16, 8, 8, 256, 0, g.options(kernel=g.GEMM_KERNEL_BF16_1CTA))


def test_valid_call_without_gpu_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert g.lib().gemm_bf16(16, 16, 16, 8, 8, 8, 0) == g.GEMM_ERR_NO_DEVICE


def _order(num_m, num_n, group):
    return [g.tile_coord(num_m * 256, num_n * 256, 256, 256, group, t) for t in range(num_m * num_n)]


def test_tile_order_m_first_without_groups():
    # group = all of M: plain M-first walk ("NVFP4 GEMM on Blackwell", Kernel 5: the v4 order
    # (m0,n0), (m1,n0), ... (m0,n1), ...)
    assert _order(3, 2, 3) == [(0, 0), (1, 0), (2, 0), (0, 1), (1, 1), (2, 1)]


def test_tile_order_groups_match_supergroup_sequence_transposed():
    # The NVFP4 page's supergroup=4 walk visits (m0,n0), (m0,n1), (m0,n2), (m0,n3), (m1,n0), ...
    # Groups here run along M, so the same sequence appears with the roles of m and n exchanged.
    seq = _order(8, 3, 4)
    assert seq[:9] == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1), (1, 1), (2, 1), (3, 1), (0, 2)]
    assert seq[12:14] == [(4, 0), (5, 0)]


def test_tile_order_last_group_is_clamped():
    seq = _order(10, 2, 4)
    assert seq[16:] == [(8, 0), (9, 0), (8, 1), (9, 1)]


@pytest.mark.parametrize("num_m,num_n,group", [(1, 1, 1), (7, 5, 3), (16, 56, 9), (32, 32, 16), (5, 9, 8), (3, 4, 1)])
def test_tile_order_is_a_permutation(num_m, num_n, group):
    seq = _order(num_m, num_n, group)
    assert sorted(seq) == sorted(itertools.product(range(num_m), range(num_n)))


def test_tile_order_ragged_problem_sizes():
    # M = 4000 with 256-row tiles: 16 M-blocks, the last one holds rows 3840..3999
    assert g.tile_coord(4000, 14336, 256, 256, 16, 15) == (15, 0)
    with pytest.raises(g.GemmError):
        g.tile_coord(4000, 14336, 256, 256, 16, 16 * 56)


def test_group_choice():
    L2 = 126 * 2 ** 20
    # operands fit in L2: walk all of M
    assert g.choose_group_m(4096, 4096, 4096, 256, 256, 4, 74, L2) == 16
    # 8192^3 BF16, 76 co-resident pairs: two waves balanced at sqrt(2 * 76) ~ 12 M-blocks
    assert g.choose_group_m(8192, 8192, 8192, 256, 256, 4, 76, L2) == 12
    assert g.choose_group_m(6144, 6144, 6144, 256, 256, 4, 76, L2) == 12
    assert g.choose_group_m(4000, 14336, 4096, 256, 256, 4, 76, L2) == 12
    # NVFP4 (half a byte per element plus a scale byte per 16): operands that fit in L2 walk all
    # of M; larger ones balance two waves like BF16
    assert g.choose_group_m(8192, 8192, 8192, 256, 256, 1, 76, L2) == 32
    assert g.choose_group_m(16384, 16384, 16384, 256, 256, 1, 76, L2) == 12
    # beyond L2 (a very large K, or the 512 x 256 tile at 8192^3) the balanced group stays:
    # smaller groups only re-read B more often
    assert g.choose_group_m(8192, 8192, 65536, 256, 256, 4, 76, L2) == 12
    assert g.choose_group_m(12288, 12288, 12288, 256, 256, 4, 76, L2) == 12
    assert g.choose_group_m(8192, 8192, 8192, 512, 256, 4, 76, L2) == 9
    assert g.choose_group_m(8192, 8192, 8192, 256, 256, 1, 74, L2) >= 1


def test_mma_rate_argument_errors():
    import ctypes
    out = ctypes.c_double(0.0)
    assert g.lib().gemm_measure_mma_rate(8, ctypes.byref(out)) == g.GEMM_ERR_INVALID_ARG
    assert g.lib().gemm_measure_mma_rate(-1, ctypes.byref(out)) == g.GEMM_ERR_INVALID_ARG
    assert g.lib().gemm_measure_mma_rate(g.GEMM_MMA_BF16, None) == g.GEMM_ERR_INVALID_ARG


def test_bf16_plan_swaps_few_row_gemms():
    """C^T = B A^T for M <= 128 and N >= 256 on the default kernel, with or without a fused epilogue."""
    assert g.bf16_plan(16, 8192, 8192) == (1, 64)
    assert g.bf16_plan(1, 256, 64) == (1, 64)
    assert g.bf16_plan(64, 8192, 8192) == (1, 64)
    assert g.bf16_plan(65, 8192, 8192) == (1, 128)
    assert g.bf16_plan(128, 8192, 8192) == (1, 128)
    assert g.bf16_plan(129, 8192, 8192) == (0, 256)
    assert g.bf16_plan(16, 248, 8192) == (0, 256)          # N too small to fill the MMA rows
    assert g.bf16_plan(16, 8192, 8192, g.options(no_swap_ab=1)) == (0, 256)
    assert g.bf16_plan(16, 8192, 8192, g.options(kernel=g.GEMM_KERNEL_BF16_2CTA)) == (0, 256)
    assert g.bf16_plan(16, 8192, 8192, g.options(kernel=g.GEMM_KERNEL_BF16_1CTA)) == (0, 256)
    assert g.bf16_plan(16, 8192, 8192, epi=g.epilogue(activation=g.GEMM_ACT_RELU)) == (1, 64)  # fused, swapped
    assert g.bf16_plan(16, 8192, 8192, epi=g.epilogue()) == (1, 64)   # the identity epilogue is not fused
    with pytest.raises(g.GemmError):
        g.bf16_plan(-1, 8, 8)
    with pytest.raises(g.GemmError):
        g.bf16_plan(16, 8192, 8192, g.options(no_swap_ab=2))


def test_clc_rule_bands():
    """Static / dynamic scheduling: nothing to balance within one wave; beyond it the CLC order
    only for BF16 with K >= 16384 (where it measured faster on GB300, at any wave count)."""
    W = 76
    assert not g.clc_rule(1, W, 65536)
    assert not g.clc_rule(W, W, 65536)            # exactly one wave
    assert not g.clc_rule(W + 1, W, 16383)
    assert g.clc_rule(W + 1, W, 16384)
    assert not g.clc_rule(1024, W, 8192)          # 8192^3 BF16: 1024 tiles of 256 x 256, static
    assert not g.clc_rule(4096, W, 8192)          # 54 waves, K = 8192: static
    assert g.clc_rule(1024, W, 16384)
    assert g.clc_rule(4096, W, 16384)
    assert not g.clc_rule(256, W, 4096)
    # NVFP4 keeps the static order at every depth
    assert not g.clc_rule(1024, W, 16384, nvfp4=True)
    assert not g.clc_rule(4096, W, 65536, nvfp4=True)
    with pytest.raises(g.GemmError):
        g.clc_rule(10, 0, 8192)
    with pytest.raises(g.GemmError):
        g.clc_rule(-1, W, 8192)


def test_nvfp4_plan_pads_a_for_few_rows():
    """1 <= M < 32: the NVFP4 GEMM reads A from a 32-row copy, unless no_pad_a; otherwise A in place."""
    for M in (1, 2, 16, 31):
        assert g.nvfp4_plan(M, 8192, 8192) == 32
        assert g.nvfp4_plan(M, 8192, 8192, g.options(no_pad_a=1)) == M
    for M in (0, 32, 33, 256, 8192):
        assert g.nvfp4_plan(M, 8192, 8192) == M
    import ctypes
    out = ctypes.c_int()
    assert g.lib().gemm_nvfp4_plan(-1, 8, 256, None, ctypes.byref(out)) == g.GEMM_ERR_INVALID_ARG
    assert g.lib().gemm_nvfp4_plan(1, 8, 256, None, None) == g.GEMM_ERR_INVALID_ARG
    o = g.options()
    o.no_pad_a = 2
    assert g.lib().gemm_nvfp4_plan(1, 8, 256, ctypes.byref(o), ctypes.byref(out)) == g.GEMM_ERR_INVALID_ARG


def test_clock_probe_options_checked():
    """gemm_options_t.clock_probe: a negative CTA count, or a count without a buffer, is
    GEMM_ERR_INVALID_ARG (checked on the host before any launch)."""
    import ctypes
    out = ctypes.c_int()
    o = g.options()
    assert g.lib().gemm_nvfp4_plan(1, 8, 256, ctypes.byref(o), ctypes.byref(out)) == g.GEMM_OK
    o.clock_probe_ctas = -1
    assert g.lib().gemm_nvfp4_plan(1, 8, 256, ctypes.byref(o), ctypes.byref(out)) == g.GEMM_ERR_INVALID_ARG
    o.clock_probe_ctas = 4  # no buffer
    assert g.lib().gemm_nvfp4_plan(1, 8, 256, ctypes.byref(o), ctypes.byref(out)) == g.GEMM_ERR_INVALID_ARG
    o.clock_probe = 256  # any non-null address passes the host check (the kernel writes it)
    assert g.lib().gemm_nvfp4_plan(1, 8, 256, ctypes.byref(o), ctypes.byref(out)) == g.GEMM_OK


def test_bf16_wide_rule():
    """The 512 x 256 pair tile where its fewer, larger tiles still fill the 76 clusters."""
    assert g.bf16_wide_rule(8192, 8192, 8192)          # 512 wide tiles: 7 waves vs 13.8
    assert g.bf16_wide_rule(4000, 14336, 4096)         # 448: 6 waves vs 12
    assert g.bf16_wide_rule(6144, 6144, 6144)          # 288: 4 waves vs 8
    assert g.bf16_wide_rule(4096, 4096, 4096)          # 128: 2 waves = 3.77 vs 3.8 tile-times
    assert g.bf16_wide_rule(8192, 8192, 2048)          # 7 waves = 13.6 vs 13.8 (f = 1.03 at K = 2048)
    assert not g.bf16_wide_rule(8192, 8192, 1024)      # shallow K: the tile boundary costs too much
    assert not g.bf16_wide_rule(512, 512, 8192)        # 2 wide tiles vs 4 tiles, both as N-halves
    assert not g.bf16_wide_rule(2048, 2048, 8192)      # 32 wide tiles as N-halves: 1.51 vs 64 tiles: 1
    with pytest.raises(g.GemmError):
        g.bf16_wide_rule(8, 8, 8, 0)
    l = g.lib()
    assert l.gemm_bf16_wide_rule(-1, 8, 8, 76) == -g.GEMM_ERR_INVALID_ARG

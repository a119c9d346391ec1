"""Fused epilogue (C = act(alpha A B^T + beta C + bias)) through the C ABI against the oracle.

The oracle computes the product in FP64 (oracle.gemm_bf16 / gemm_nvfp4) and the epilogue
in FP64 (oracle.epilogue), then rounds once to BF16. The kernels evaluate the epilogue in
FP32 on the FP32 accumulator, so beside one BF16 ulp the tolerance allows the product's
FP32 accumulation error scaled by |alpha| and the FP32 rounding of the epilogue's terms.
"""
import math

import numpy as np
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import oracle
import synthetic_inputs as si
from dense_tensor_core_persistent_gb300 import build as gbuild
from parity import assert_nvfp4_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# name -> (alpha, beta, with bias, activation)
VARIANTS = {
    "scale_bias_relu": (0.75, 0.0, True, g.GEMM_ACT_RELU),
    "beta_only": (1.0, -0.5, False, g.GEMM_ACT_NONE),
    "all_gelu": (-1.25, 1.5, True, g.GEMM_ACT_GELU_TANH),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbuild.build()


def bias_bits(N, seed):
    """A bias vector: BF16 values uniform in [-2, 2] (bits)."""
    t = torch.empty(N).uniform_(-2, 2, generator=torch.Generator().manual_seed(seed))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_dev_bf16(bits_np):
    return torch.from_numpy(np.ascontiguousarray(bits_np).view(np.int16)).view(torch.bfloat16).to(DEV)


def prior_c(M, N, seed):
    """Prior contents of C: BF16 values uniform in [-2, 2] (bits)."""
    t = torch.empty(M, N).uniform_(-2, 2, generator=torch.Generator().manual_seed(seed))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def epilogue_args(variant, N, seed):
    alpha, beta, with_bias, act = VARIANTS[variant]
    b = bias_bits(N, seed) if with_bias else None
    return alpha, beta, b, act


def assert_fused_close(gpu_bits, acc, alpha, beta, c_old, bias, act, K, what):
    x = oracle.epilogue(acc, alpha, beta, c_old, bias, act)
    R = oracle.round_bf16(x)
    got = oracle.bf16_bits_to_f64(gpu_bits)
    mag = np.abs(alpha * acc)
    if beta != 0.0:
        mag = mag + np.abs(beta * oracle.bf16_bits_to_f64(c_old))
    if bias is not None:
        mag = mag + np.abs(oracle.bf16_bits_to_f64(bias))[None, :]
    slack = abs(alpha) * 1e-4 * math.sqrt(K) + 2.0 ** -22 * mag
    if act == g.GEMM_ACT_GELU_TANH:
        slack = slack * 1.2  # |gelu'| <= 1.13
    tol = oracle.ulp_bf16(R) + slack
    err = np.abs(got - oracle.bf16_bits_to_f64(R))
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance, max err {err.max():.3g}"


def run_bf16_fused(A, B, c_old, alpha, beta, bias, act, opts=None):
    M, N, K = A.shape[0], B.shape[0], A.shape[1]
    C = to_dev_bf16(c_old) if c_old is not None else torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bias_t = to_dev_bf16(bias) if bias is not None else None
    g.gemm_bf16_fused(A.to(DEV), B.to(DEV), C, M, N, K, g.epilogue(alpha, beta, bias_t, act), opts=opts)
    torch.cuda.synchronize()
    return bits(C)


# ---------------------------------------------------------------- BF16

@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("kernel", [g.GEMM_KERNEL_DEFAULT, g.GEMM_KERNEL_BF16_1CTA, g.GEMM_KERNEL_BF16_2CTA_WIDE])
def test_bf16_fused_ragged(variant, kernel):
    M, N, K = 300, 264, 320  # ragged M and N (264 = 4 * 64 + 8), K over several stages
    A, B = si.bf16_problem(31, M, N, K)
    alpha, beta, bias, act = epilogue_args(variant, N, 32)
    c_old = prior_c(M, N, 33)
    got = run_bf16_fused(A, B, c_old, alpha, beta, bias, act, opts=g.options(kernel=kernel))
    assert_fused_close(got, oracle.gemm_bf16(A, B), alpha, beta, c_old, bias, act, K, variant)


@pytest.mark.parametrize("kernel", [g.GEMM_KERNEL_DEFAULT, g.GEMM_KERNEL_BF16_2CTA_WIDE])
def test_bf16_fused_integer_inputs_bit_exact(kernel):
    """Integer operands, power-of-two alpha and beta, integer prior C and bias: every FP32
    step is exact, so the result must equal the oracle's rounding bit for bit."""
    M, N, K = 600, 264, 256  # the 512 x 256 tile: the second row block holds 88 rows (one CTA, wave 0)
    A, B = si.bf16_problem(0, M, N, K, kind="int")
    c_old = torch.randint(-8, 9, (M, N), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    c_old = c_old.view(torch.int16).numpy().view(np.uint16)
    bias = torch.randint(-16, 17, (N,), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    bias = bias.view(torch.int16).numpy().view(np.uint16)
    for alpha, beta, act in [(0.5, 2.0, g.GEMM_ACT_RELU), (-2.0, -0.25, g.GEMM_ACT_NONE)]:
        got = run_bf16_fused(A, B, c_old, alpha, beta, bias, act, opts=g.options(kernel=kernel))
        want = oracle.round_bf16(oracle.epilogue(oracle.gemm_bf16(A, B), alpha, beta, c_old, bias, act))
        assert np.array_equal(oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(want)), (alpha, beta, act)


def test_bf16_identity_epilogue_matches_unfused_bits():
    M, N, K = 300, 264, 320
    A, B = (t.to(DEV) for t in si.bf16_problem(34, M, N, K))
    C0 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    C1 = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    g.gemm_bf16(A, B, C0, M, N, K)
    g.gemm_bf16_fused(A, B, C1, M, N, K, g.epilogue())
    torch.cuda.synchronize()
    assert np.array_equal(bits(C0), bits(C1))


@pytest.mark.parametrize("max_clusters", [1, 3])
@pytest.mark.parametrize("kernel", [g.GEMM_KERNEL_DEFAULT, g.GEMM_KERNEL_BF16_2CTA_WIDE])
def test_bf16_fused_many_tiles_per_cluster(max_clusters, kernel):
    """Each epilogue warp loads the prior C of many chunks and tiles: its load barrier's
    phase alternates across tiles."""
    M, N, K = 1280, 1024, 256
    A, B = si.bf16_problem(35, M, N, K)
    c_old = prior_c(M, N, 36)
    bias = bias_bits(N, 37)
    got = run_bf16_fused(A, B, c_old, 1.5, -1.0, bias, g.GEMM_ACT_GELU_TANH,
                         opts=g.options(max_clusters=max_clusters, kernel=kernel))
    assert_fused_close(got, oracle.gemm_bf16(A, B), 1.5, -1.0, c_old, bias, g.GEMM_ACT_GELU_TANH, K, "many tiles")


def test_bf16_fused_default_wide_tile():
    """A fused call at a shape where the default takes the 512 x 256 tile (ragged in M, N
    and K), with alpha, beta, bias and GELU."""
    M, N, K = 2600, 3064, 4104
    assert g.bf16_wide_rule(M, N, K)
    A, B = si.bf16_problem(38, M, N, K)
    c_old = prior_c(M, N, 39)
    bias = bias_bits(N, 40)
    got = run_bf16_fused(A, B, c_old, -1.25, 1.5, bias, g.GEMM_ACT_GELU_TANH)
    assert_fused_close(got, oracle.gemm_bf16(A, B), -1.25, 1.5, c_old, bias, g.GEMM_ACT_GELU_TANH, K, "default wide")


# ---------------------------------------------------------------- NVFP4

def run_nvfp4_fused(a, sfa, b, sfb, c_old, alpha, beta, bias, act, path, opts=None):
    M, N, K = a.shape[0], b.shape[0], 2 * a.shape[1]
    C = to_dev_bf16(c_old)
    bias_t = to_dev_bf16(bias) if bias is not None else None
    ep = g.epilogue(alpha, beta, bias_t, act)
    a, sfa, b, sfb = (t.to(DEV) for t in (a, sfa, b, sfb))
    if path == "blocked_scales":
        g.gemm_nvfp4_blocked_fused(a, g.pack_scales(sfa), b, g.pack_scales(sfb), C, M, N, K, ep, opts=opts)
    else:
        g.gemm_nvfp4_fused(a, sfa, b, sfb, C, M, N, K, ep, opts=opts)
    torch.cuda.synchronize()
    return bits(C)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("path", ["rowmajor_scales", "blocked_scales"])
def test_nvfp4_fused_ragged(variant, path):
    M, N, K = 300, 264, 512  # the last 16-column store box of a row block is half outside N
    a, sfa, b, sfb = si.nvfp4_problem(41, M, N, K)
    alpha, beta, bias, act = epilogue_args(variant, N, 42)
    c_old = prior_c(M, N, 43)
    got = run_nvfp4_fused(a, sfa, b, sfb, c_old, alpha, beta, bias, act, path)
    ref = oracle.epilogue(oracle.gemm_nvfp4(a, sfa, b, sfb), alpha, beta, c_old, bias, act)
    assert_nvfp4_close(got, ref, variant)


@pytest.mark.parametrize("max_clusters", [1, 3])
def test_nvfp4_fused_many_tiles_per_cluster(max_clusters):
    M, N, K = 1280, 1024, 768
    a, sfa, b, sfb = si.nvfp4_problem(44, M, N, K)
    c_old = prior_c(M, N, 45)
    bias = bias_bits(N, 46)
    got = run_nvfp4_fused(a, sfa, b, sfb, c_old, 0.5, 2.0, bias, g.GEMM_ACT_RELU, "blocked_scales",
                          opts=g.options(max_clusters=max_clusters))
    ref = oracle.epilogue(oracle.gemm_nvfp4(a, sfa, b, sfb), 0.5, 2.0, c_old, bias, g.GEMM_ACT_RELU)
    assert_nvfp4_close(got, ref, "many tiles")


# ---------------------------------------------------------------- semantics and errors

@pytest.mark.parametrize("kind", ["bf16", "nvfp4"])
def test_beta_zero_does_not_read_c(kind):
    """With beta == 0 the prior C is not read: NaN there must not reach the result."""
    M, N = 300, 264
    nan_c = np.full((M, N), 0x7FC0, dtype=np.uint16)
    bias = bias_bits(N, 51)
    if kind == "bf16":
        K = 128
        A, B = si.bf16_problem(50, M, N, K)
        got = run_bf16_fused(A, B, nan_c, 2.0, 0.0, bias, g.GEMM_ACT_NONE)
        assert_fused_close(got, oracle.gemm_bf16(A, B), 2.0, 0.0, None, bias, g.GEMM_ACT_NONE, K, "beta 0")
    else:
        K = 256
        a, sfa, b, sfb = si.nvfp4_problem(52, M, N, K)
        got = run_nvfp4_fused(a, sfa, b, sfb, nan_c, 2.0, 0.0, bias, g.GEMM_ACT_NONE, "blocked_scales")
        assert_nvfp4_close(got, oracle.epilogue(oracle.gemm_nvfp4(a, sfa, b, sfb), 2.0, 0.0, None, bias), "beta 0")


@pytest.mark.parametrize("kind", ["bf16", "nvfp4", "nvfp4_blocked"])
def test_empty_sum_applies_the_epilogue(kind):
    """K == 0: the product is zero and C = act(beta * C + bias)."""
    M, N = 37, 72
    c_old = prior_c(M, N, 53)
    bias = bias_bits(N, 54)
    C = to_dev_bf16(c_old)
    ep = g.epilogue(3.0, -0.75, to_dev_bf16(bias), g.GEMM_ACT_GELU_TANH)
    empty = torch.empty(0, dtype=torch.uint8, device=DEV)
    if kind == "bf16":
        g.gemm_bf16_fused(empty, empty, C, M, N, 0, ep)
    elif kind == "nvfp4":
        g.gemm_nvfp4_fused(empty, empty, empty, empty, C, M, N, 0, ep)
    else:
        g.gemm_nvfp4_blocked_fused(empty, empty, empty, empty, C, M, N, 0, ep)
    torch.cuda.synchronize()
    assert_fused_close(bits(C), np.zeros((M, N)), 3.0, -0.75, c_old, bias, g.GEMM_ACT_GELU_TANH, 1, "K = 0")


def test_rejected_epilogues():
    M, N, K = 64, 64, 64
    A, B = (t.to(DEV) for t in si.bf16_problem(55, M, N, K))
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    bias = torch.zeros(N + 8, dtype=torch.bfloat16, device=DEV)
    l = g.lib()
    cases = [
        (g.gemm_epilogue_t(1.0, 0.0, None, 7, 0), g.GEMM_ERR_INVALID_ARG),                  # unknown activation
        (g.gemm_epilogue_t(1.0, 0.0, None, 0, 1), g.GEMM_ERR_INVALID_ARG),                  # reserved set
        (g.gemm_epilogue_t(1.0, 0.0, bias.data_ptr() + 2, 0, 0), g.GEMM_ERR_MISALIGNED),  # bias not 16-byte aligned
    ]
    for ep, want in cases:
        import ctypes
        st = l.gemm_bf16_fused(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, None, ctypes.byref(ep), None)
        assert st == want, (ep.activation, ep.reserved, st)
        st = l.gemm_nvfp4_blocked_fused(A.data_ptr(), A.data_ptr(), B.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, 256,
                                        None, ctypes.byref(ep), None)
        assert st == want, ("nvfp4", ep.activation, ep.reserved, st)


@pytest.mark.parametrize("kind", ["bf16", "nvfp4"])
@pytest.mark.parametrize("no_pdl", [0, 1])
def test_beta_reads_the_previous_result_on_one_stream(kind, no_pdl):
    """Call 1 writes C; call 2 on the same stream reads it as its prior C (beta = 1). With
    programmatic dependent launch the second kernel starts early, so its prior-C loads must
    still wait for the first kernel's stores. The expected prior C is call 1's own result
    (computed once more beforehand: identical launches give identical bits), which may
    differ from the oracle's rounding by one ulp."""
    M, N = 512, 1024
    opts = g.options(no_pdl=no_pdl)
    s = torch.cuda.Stream()
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    first_c = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    if kind == "bf16":
        K = 512
        A1, B1 = (t.to(DEV) for t in si.bf16_problem(61, M, N, K))
        A2, B2 = si.bf16_problem(62, M, N, K)
        g.gemm_bf16(A1, B1, first_c, M, N, K, opts=opts)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.gemm_bf16(A1, B1, C, M, N, K, stream=s, opts=opts)
            g.gemm_bf16_fused(A2.to(DEV), B2.to(DEV), C, M, N, K, g.epilogue(1.0, 1.0), stream=s, opts=opts)
        s.synchronize()
        assert_fused_close(bits(C), oracle.gemm_bf16(A2, B2), 1.0, 1.0, bits(first_c), None, g.GEMM_ACT_NONE, K,
                           "chained")
    else:
        K = 1024
        p1 = [t.to(DEV) for t in si.nvfp4_problem(63, M, N, K)]
        p2 = [t.to(DEV) for t in si.nvfp4_problem(64, M, N, K)]
        g.gemm_nvfp4(*p1, first_c, M, N, K, opts=opts)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.gemm_nvfp4(*p1, C, M, N, K, stream=s, opts=opts)
            g.gemm_nvfp4_fused(*p2, C, M, N, K, g.epilogue(1.0, 1.0), stream=s, opts=opts)
        s.synchronize()
        ref = oracle.epilogue(oracle.gemm_nvfp4(*[t.cpu() for t in p2]), 1.0, 1.0, bits(first_c), None)
        assert_nvfp4_close(bits(C), ref, "chained")


# ---------------------------------------------------------------- few rows: swapped (C^T = B A^T)

FEW_ROW_SHAPES = [
    (1, 1024, 512),      # tile N 64
    (16, 2056, 1024),    # ragged N
    (64, 520, 1024),     # ragged last block of the long dimension
    (100, 776, 136),     # tile N 128, partial K stage
    (16, 1024, 4096),    # K split 8 ways: the reduction kernel applies the epilogue
    (4, 8192, 6144),     # two splits: one cluster of two pairs, the first applies the epilogue
]


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("shape", FEW_ROW_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bf16_fused_few_rows_swapped(variant, shape):
    M, N, K = shape
    assert g.bf16_plan(M, N, K, epi=g.epilogue(activation=g.GEMM_ACT_RELU))[0] == 1
    A, B = si.bf16_problem(M + N + K, M, N, K)
    alpha, beta, bias, act = epilogue_args(variant, N, 40)
    c_old = prior_c(M, N, 41)
    got = run_bf16_fused(A, B, c_old, alpha, beta, bias, act)
    assert_fused_close(got, oracle.gemm_bf16(A, B), alpha, beta, c_old, bias, act, K, f"{variant} {shape}")
    # the same call without swap-AB agrees within the same tolerance
    got2 = run_bf16_fused(A, B, c_old, alpha, beta, bias, act, opts=g.options(no_swap_ab=1))
    assert_fused_close(got2, oracle.gemm_bf16(A, B), alpha, beta, c_old, bias, act, K, f"{variant} {shape} no swap")


def test_bf16_fused_few_rows_integer_inputs_bit_exact():
    # integer operands, power-of-two alpha and beta, integer bias: every step exact in FP32
    M, N, K = 48, 2048, 256
    A, B = si.bf16_problem(42, M, N, K, kind="int")
    bias = np.arange(N, dtype=np.float32) % 7 - 3
    bias = torch.from_numpy(bias).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    c_old = prior_c(M, N, 43)
    c_old_int = torch.from_numpy(np.round(oracle.bf16_bits_to_f64(c_old) * 4)).to(torch.bfloat16)
    c_old = c_old_int.view(torch.int16).numpy().view(np.uint16)
    got = run_bf16_fused(A, B, c_old, 2.0, 0.5, bias, g.GEMM_ACT_RELU)
    want = oracle.round_bf16(oracle.epilogue(oracle.gemm_bf16(A, B), 2.0, 0.5, c_old, bias, g.GEMM_ACT_RELU))
    assert np.array_equal(oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(want))


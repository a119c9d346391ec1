"""Pins for the CPU oracle (no GPU needed).

Each test checks the oracle against something other than itself: values the
pages print, closed forms, exact rational brute force, or an independent
library routine (torch's BF16 / FP8 conversions, torch's FP64 matmul).
"""
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.strip() for l in f if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------- decoders

def test_e2m1_matches_printed_code_points():
    """All 16 E2M1 codes decode to the 16 values printed on the NVFP4 page."""
    printed = sorted(float(v) for v in _golden_lines("e2m1_values.txt"))
    decoded = [oracle.dec_e2m1(c) for c in range(16)]
    assert sorted(decoded) == printed
    # sign bit is bit 3: codes 0..7 non-negative and strictly increasing with the
    # magnitude bits (exponent above mantissa), codes 8..15 their negatives
    pos = decoded[:8]
    assert all(np.signbit(v) == False for v in pos)  # noqa: E712
    assert all(pos[i] < pos[i + 1] for i in range(7))
    for c in range(8):
        assert decoded[c | 8] == -decoded[c]
        assert np.signbit(decoded[c | 8])


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.dec_e4m3(c) for c in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # spot values of the scale range used by the NVFP4 workload
    assert oracle.dec_e4m3(0x18) == 2.0 ** -4
    assert oracle.dec_e4m3(0x38) == 1.0
    assert oracle.dec_e4m3(0x58) == 16.0
    assert oracle.dec_e4m3(0x7E) == 448.0


def test_bf16_decode_all_codes_match_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.dec_bf16(b) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# ---------------------------------------------------------------- rounding

def _torch_f32_to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(f32.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_on_float32_values():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # every tie case: low 16 bits exactly half an ulp
    ties = (rng.integers(0, 2 ** 16, size=50_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    allbits = np.concatenate([bits, ties])
    f32 = allbits.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    got = oracle.round_bf16(f32.astype(np.float64))
    ref = _torch_f32_to_bf16_bits(f32)
    assert np.array_equal(got, ref)


def _all_finite_bf16_sorted():
    b = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite, increasing
    return b, (b << 16).view(np.float32).astype(np.float64)


def test_bf16_rne_brute_force_on_doubles():
    """Doubles with more precision than FP32, rounded by exhaustive nearest search."""
    bits, vals = _all_finite_bf16_sorted()
    rng = random.Random(11)
    for _ in range(3000):
        i = rng.randrange(1, len(vals) - 1)
        lo, hi = Fraction(vals[i]), Fraction(vals[i + 1])
        mid = (lo + hi) / 2
        choice = rng.randrange(4)
        if choice == 0:
            x = float(mid)                                   # exact tie
        elif choice == 1:
            x = float(mid + (hi - lo) * Fraction(1, 2 ** 40))  # just above the tie
        elif choice == 2:
            x = float(mid - (hi - lo) * Fraction(1, 2 ** 40))  # just below
        else:
            x = float(lo + (hi - lo) * Fraction(rng.random()))
        fx = Fraction(x)
        j = int(np.searchsorted(vals, x, side="right")) - 1
        dlo, dhi = fx - Fraction(vals[j]), Fraction(vals[j + 1]) - fx
        if dlo < dhi:
            want = bits[j]
        elif dhi < dlo:
            want = bits[j + 1]
        else:
            want = bits[j] if bits[j] % 2 == 0 else bits[j + 1]
        sign = rng.randrange(2)
        got = oracle.bf16_rne(-x if sign else x)
        assert got == (int(want) | (0x8000 if sign else 0)), (x, hex(got), hex(int(want)))


def test_bf16_rne_integer_ties_round_to_even():
    # in [256, 512) the BF16 step is 2: odd integers are ties
    assert [oracle.bf16_rne(v) for v in (257, 259, 261, 263)] == [
        oracle.bf16_rne(256), oracle.bf16_rne(260), oracle.bf16_rne(260), oracle.bf16_rne(264)]
    assert oracle.dec_bf16(oracle.bf16_rne(257.0)) == 256.0
    assert oracle.dec_bf16(oracle.bf16_rne(259.0)) == 260.0
    assert oracle.dec_bf16(oracle.bf16_rne(257.0000001)) == 258.0
    assert oracle.bf16_rne(0.0) == 0 and oracle.bf16_rne(-0.0) == 0x8000
    assert oracle.bf16_rne(1e39) == 0x7F80 and oracle.bf16_rne(-1e39) == 0xFF80
    assert oracle.bf16_rne(2.0 ** -133) == 0x0001          # smallest subnormal
    assert oracle.bf16_rne(2.0 ** -134) == 0x0000          # tie to even (zero)
    assert oracle.bf16_rne(3 * 2.0 ** -134) == 0x0002      # tie 1.5 ulp -> 2


def test_ulp_bf16():
    r = oracle.round_bf16(np.array([1.0, 1.5, 255.0, 256.0, -3.0, 0.0, 2.0 ** -130]))
    assert list(oracle.ulp_bf16(r)) == [2.0 ** -7, 2.0 ** -7, 2.0 ** 0, 2.0 ** 1, 2.0 ** -6, 2.0 ** -133, 2.0 ** -133]


# ---------------------------------------------------------------- BF16 GEMM

def _frac_gemm(Ad, Bd):
    M, K = Ad.shape
    N = Bd.shape[0]
    return [[sum((Fraction(Ad[i, k]) * Fraction(Bd[j, k]) for k in range(K)), Fraction(0))
             for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (2, 3, 7), (3, 2, 16), (7, 5, 33), (16, 16, 3)])
def test_bf16_gemm_brute_force_exact(m, n, k):
    A, B = si.bf16_problem(100 + m * n * k, m, n, k)
    C = oracle.gemm_bf16(A, B)
    exact = _frac_gemm(A.double().numpy(), B.double().numpy())
    absum = (A.double().abs() @ B.double().abs().T).numpy()
    for i in range(m):
        for j in range(n):
            assert abs(Fraction(C[i, j]) - exact[i][j]) <= Fraction(absum[i, j]) * k * Fraction(1, 2 ** 52)


@pytest.mark.parametrize("m,n,k", [(5, 9, 64), (33, 17, 40)])
def test_bf16_gemm_integer_inputs_exact(m, n, k):
    A, B = si.bf16_problem(5, m, n, k, kind="int")
    C = oracle.gemm_bf16(A, B)
    exact = _frac_gemm(A.double().numpy(), B.double().numpy())
    assert all(C[i, j] == exact[i][j] for i in range(m) for j in range(n))


def test_bf16_gemm_identity_gives_b_transposed():
    K, N = 24, 11
    A = torch.eye(K, dtype=torch.bfloat16)
    _, B = si.bf16_problem(3, 1, N, K)
    C = oracle.gemm_bf16(A, B)
    assert np.array_equal(C, B.double().numpy().T)


def test_bf16_gemm_all_ones_gives_k():
    for K in (1, 8, 256, 4096):
        A = torch.ones(3, K, dtype=torch.bfloat16)
        B = torch.ones(5, K, dtype=torch.bfloat16)
        assert np.all(oracle.gemm_bf16(A, B) == K)


def test_bf16_gemm_matches_torch_fp64_matmul():
    for (m, n, k) in [(64, 48, 80), (130, 70, 264)]:
        A, B = si.bf16_problem(9, m, n, k)
        C = oracle.gemm_bf16(A, B)
        ref = (A.double() @ B.double().T).numpy()
        bound = (A.double().abs() @ B.double().abs().T).numpy() * k * 2.0 ** -52
        assert np.all(np.abs(C - ref) <= bound)


def test_bf16_gemm_row_range_and_sampled_agree_with_full():
    A, B = si.bf16_problem(4, 37, 29, 72)
    full = oracle.gemm_bf16(A, B)
    assert np.array_equal(oracle.gemm_bf16(A, B, 10, 21), full[10:21])
    rng = np.random.default_rng(1)
    rows, cols = rng.integers(0, 37, 100), rng.integers(0, 29, 100)
    assert np.array_equal(oracle.gemm_bf16_at(A, B, rows, cols), full[rows, cols])


# ---------------------------------------------------------------- NVFP4 GEMM

def _e2m1_table():
    """code -> value from the printed value set, assigned by sign bit 3 and magnitude order."""
    vals = sorted({abs(float(v)) for v in _golden_lines("e2m1_values.txt")})  # 0,0.5,...,6
    return [vals[c] for c in range(8)] + [-vals[c] for c in range(8)]


def _unpack(packed: torch.Tensor) -> np.ndarray:
    p = packed.numpy()
    codes = np.empty((p.shape[0], 2 * p.shape[1]), dtype=np.uint8)
    codes[:, 0::2] = p & 0xF
    codes[:, 1::2] = p >> 4
    return codes


def _nvfp4_decode_lib(packed, sf):
    """Decode with the printed E2M1 table and torch's E4M3 conversion (not the oracle's)."""
    table = np.array(_e2m1_table())
    vals = table[_unpack(packed)]
    scales = sf.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(scales, 16, axis=1)


def test_nvfp4_code_points_through_the_gemm():
    """Row of A = the 16 codes (scale 1), B one-hot: C[0, j] is code j's printed value."""
    K = 16
    codes = torch.arange(16, dtype=torch.uint8).view(1, 16)
    A = si.pack_e2m1(codes)
    SFA = torch.full((1, 1), 0x38, dtype=torch.uint8)  # E4M3 1.0
    onehot = torch.zeros(16, K, dtype=torch.uint8)
    onehot[torch.arange(16), torch.arange(16)] = 0x2     # E2M1 1.0
    B = si.pack_e2m1(onehot)
    SFB = torch.full((16, 1), 0x38, dtype=torch.uint8)
    C = oracle.gemm_nvfp4(A, SFA, B, SFB)
    assert list(C[0]) == _e2m1_table()


def test_nvfp4_low_nibble_is_even_k():
    K = 32
    A = torch.zeros(1, K // 2, dtype=torch.uint8)
    A[0, 3] = 0x0C | (0x07 << 4)       # element 6 = code 0xC (-2), element 7 = code 0x7 (6)
    SFA = torch.full((1, 2), 0x38, dtype=torch.uint8)
    e6 = torch.zeros(1, K, dtype=torch.uint8); e6[0, 6] = 0x2
    e7 = torch.zeros(1, K, dtype=torch.uint8); e7[0, 7] = 0x2
    B = torch.cat([si.pack_e2m1(e6), si.pack_e2m1(e7)])
    SFB = torch.full((2, 2), 0x38, dtype=torch.uint8)
    C = oracle.gemm_nvfp4(A, SFA, B, SFB)
    assert list(C[0]) == [-2.0, 6.0]


def test_nvfp4_nibble_order_is_invisible_in_c():
    """Swapping the nibbles of every byte of BOTH operands permutes K the same way
    in A and B, inside one scale block, so C cannot change: the packing reading
    (even K in the low nibble) is a storage convention, not part of the result."""
    A, SFA, B, SFB = si.nvfp4_problem(12, 9, 7, 64)
    swap = lambda p: ((p & 0xF) << 4) | (p >> 4)
    assert np.array_equal(oracle.gemm_nvfp4(A, SFA, B, SFB),
                          oracle.gemm_nvfp4(swap(A), SFA, swap(B), SFB))


@pytest.mark.parametrize("m,n,k", [(1, 1, 16), (3, 2, 32), (4, 5, 48)])
def test_nvfp4_gemm_brute_force_exact(m, n, k):
    A, SFA, B, SFB = si.nvfp4_problem(200 + k, m, n, k)
    C = oracle.gemm_nvfp4(A, SFA, B, SFB)
    Ad = _nvfp4_decode_lib(A, SFA)
    Bd = _nvfp4_decode_lib(B, SFB)
    exact = _frac_gemm(Ad, Bd)
    assert all(Fraction(C[i, j]) == exact[i][j] for i in range(m) for j in range(n))


def test_nvfp4_gemm_matches_torch_fp64_matmul():
    m, n, k = 40, 24, 256
    A, SFA, B, SFB = si.nvfp4_problem(4, m, n, k)
    C = oracle.gemm_nvfp4(A, SFA, B, SFB)
    ref = _nvfp4_decode_lib(A, SFA) @ _nvfp4_decode_lib(B, SFB).T
    assert np.array_equal(C, ref)  # all partial sums exact at this size


def test_nvfp4_scale_linearity():
    """Doubling one SFA entry (E4M3 exponent + 1) doubles exactly that block's contribution."""
    m, n, k = 2, 3, 64
    A, SFA, B, SFB = si.nvfp4_problem(8, m, n, k)
    C0 = oracle.gemm_nvfp4(A, SFA, B, SFB)
    SFA2 = SFA.clone()
    SFA2[1, 2] += 8                     # exponent field + 1 -> value x 2
    C1 = oracle.gemm_nvfp4(A, SFA2, B, SFB)
    Ad = _nvfp4_decode_lib(A, SFA)
    Bd = _nvfp4_decode_lib(B, SFB)
    block = Ad[1, 32:48] @ Bd[:, 32:48].T
    assert np.array_equal(C1[0], C0[0])
    assert np.array_equal(C1[1] - C0[1], block)


def test_nvfp4_all_ones_gives_k():
    for K in (16, 256, 8192):
        codes = torch.full((2, K), 0x2, dtype=torch.uint8)
        A = si.pack_e2m1(codes)
        SF = torch.full((2, K // 16), 0x38, dtype=torch.uint8)
        assert np.all(oracle.gemm_nvfp4(A, SF, A, SF) == K)


def test_nvfp4_sampled_and_row_range_agree_with_full():
    A, SFA, B, SFB = si.nvfp4_problem(6, 19, 23, 96)
    full = oracle.gemm_nvfp4(A, SFA, B, SFB)
    assert np.array_equal(oracle.gemm_nvfp4(A, SFA, B, SFB, 4, 11), full[4:11])
    rng = np.random.default_rng(2)
    rows, cols = rng.integers(0, 19, 60), rng.integers(0, 23, 60)
    assert np.array_equal(oracle.gemm_nvfp4_at(A, SFA, B, SFB, rows, cols), full[rows, cols])


# ---------------------------------------------------------------- fused epilogue
# Pins for oracle.epilogue: closed forms computed here element by element (BF16 decoded by
# torch, not by the oracle), the order of the operations, and GELU against an independent
# formula and against the exact (erf) GELU it approximates.

def _bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits):
    t = torch.from_numpy(np.array([bits], dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return float(t.float().item())


def test_epilogue_identity():
    acc = np.random.default_rng(1).standard_normal((4, 6)) * 100
    assert np.array_equal(oracle.epilogue(acc), acc)


def test_epilogue_alpha_beta_bias_closed_form():
    rng = np.random.default_rng(2)
    M, N = 3, 5                          # not square: a bias indexed by row would not broadcast
    acc = rng.standard_normal((M, N)) * 10
    c_old = _bf16_bits(rng.uniform(-4, 4, (M, N)))
    bias = _bf16_bits([0.5, -1.0, 2.0, -3.5, 8.0])
    got = oracle.epilogue(acc, alpha=0.75, beta=-1.5, c_old=c_old, bias=bias)
    for i in range(M):
        for j in range(N):
            want = 0.75 * acc[i, j] + (-1.5) * _bf16_value(c_old[i, j]) + _bf16_value(bias[j])
            assert got[i, j] == pytest.approx(want, rel=1e-15, abs=1e-15)


def test_epilogue_order_of_operations():
    acc = np.array([[1.0, -1.0]])
    bias = _bf16_bits([1.0, 2.0])
    # alpha scales the product only: 2 * 1 + 1 = 3 (not 2 * (1 + 1))
    assert oracle.epilogue(acc, alpha=2.0, bias=bias)[0, 0] == 3.0
    # the activation follows the bias: relu(-1 + 2) = 1 (not relu(-1) + 2)
    assert oracle.epilogue(acc, bias=bias, activation=oracle.ACT_RELU)[0, 1] == 1.0


def test_epilogue_beta_zero_does_not_read_c():
    acc = np.array([[1.0, 2.0]])
    nan_bits = np.array([[0x7FC0, 0xFFC0]], dtype=np.uint16)
    assert np.array_equal(oracle.epilogue(acc, alpha=1.0, beta=0.0, c_old=nan_bits), acc)


def test_epilogue_relu():
    acc = np.array([[-3.0, -0.0, 0.0, 2.5]])
    got = oracle.epilogue(acc, activation=oracle.ACT_RELU)
    assert list(got[0]) == [0.0, 0.0, 0.0, 2.5]


def test_gelu_tanh_against_independent_forms():
    xs = np.linspace(-8.0, 8.0, 1601)
    got = oracle.gelu_tanh(xs)
    # 0.5 (1 + tanh z) = 1 / (1 + exp(-2z)): the same function through a sigmoid
    import math
    k = math.sqrt(2.0 / math.pi)
    for x, g in zip(xs, got):
        z = k * (x + 0.044715 * x ** 3)
        assert g == pytest.approx(x / (1.0 + math.exp(-2.0 * z)), rel=1e-12, abs=1e-12)
        # the exact GELU x Phi(x), which the tanh form approximates to within 1e-3
        assert abs(g - 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))) < 1e-3
        # gelu(x) - gelu(-x) = x, since tanh is odd
    assert np.allclose(oracle.gelu_tanh(xs) - oracle.gelu_tanh(-xs), xs, rtol=0, atol=1e-12)
    assert oracle.gelu_tanh([0.0])[0] == 0.0


def test_epilogue_gelu_dispatch():
    acc = np.array([[1.0, -2.0]])
    assert np.array_equal(oracle.epilogue(acc, activation=oracle.ACT_GELU_TANH), oracle.gelu_tanh(acc))
    with pytest.raises(ValueError):
        oracle.epilogue(acc, activation=9)

"""BF16 GEMM on the GPU (through the C ABI) against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import oracle
import synthetic_inputs as si
from dense_tensor_core_persistent_gb300 import build as gbuild
from parity import assert_bf16_close, assert_bf16_exact, bits, sample_coords

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


VARIANTS = {
    "pair_persistent": dict(),
    "pair_tile_per_cluster": dict(persistent=0),
    "single_cta": dict(kernel=g.GEMM_KERNEL_BF16_1CTA, persistent=0),
    "single_cta_persistent": dict(kernel=g.GEMM_KERNEL_BF16_1CTA),
    "pair_k64_persistent": dict(kernel=g.GEMM_KERNEL_BF16_2CTA_K64),
    "pair_k64_tile_per_cluster": dict(kernel=g.GEMM_KERNEL_BF16_2CTA_K64, persistent=0),
    "pair_wide_persistent": dict(kernel=g.GEMM_KERNEL_BF16_2CTA_WIDE),
    "pair_wide_tile_per_cluster": dict(kernel=g.GEMM_KERNEL_BF16_2CTA_WIDE, persistent=0),
}


def run(A, B, **opt):
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = g.matmul_bf16(Ad, Bd, opts=g.options(**opt) if opt else None)
    torch.cuda.synchronize()
    return bits(C)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_c1_uniform_256(variant):
    """256^3, entries uniform in [-1, 1] from seed 0."""
    A, B = si.bf16_problem(0, 256, 256, 256)
    assert_bf16_close(run(A, B, **VARIANTS[variant]), oracle.gemm_bf16(A, B), 256, variant)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_c1_integer_twin_bit_exact(variant):
    """256^3 with integers in [-4, 4]: every FP32 partial sum is exact, so the output is too."""
    A, B = si.bf16_problem(0, 256, 256, 256, kind="int")
    assert_bf16_exact(run(A, B, **VARIANTS[variant]), oracle.gemm_bf16(A, B), variant)


SHAPES = [
    (300, 264, 200),     # ragged M, N and a partial K stage
    (513, 520, 136),
    (1000, 776, 1032),
    (129, 8, 8),         # tiny N, single K stage with zero fill
    (1, 8, 64),
    (257, 1024, 520),
    (2048, 264, 64),
]


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes(variant, shape):
    M, N, K = shape
    A, B = si.bf16_problem(M + N + K, M, N, K)
    assert_bf16_close(run(A, B, **VARIANTS[variant]), oracle.gemm_bf16(A, B), K, f"{variant} {shape}")


@pytest.mark.parametrize("max_clusters,group_m", [(1, 0), (3, 1), (3, 2), (5, 3), (7, 16)])
@pytest.mark.parametrize("kernel", [g.GEMM_KERNEL_BF16_2CTA, g.GEMM_KERNEL_BF16_1CTA, g.GEMM_KERNEL_BF16_2CTA_K64,
                                    g.GEMM_KERNEL_BF16_2CTA_WIDE])
def test_many_tiles_per_cluster(kernel, max_clusters, group_m):
    """Few clusters, many tiles each: the stage ring and the two TMEM slots cycle across tiles."""
    M, N, K = 1280, 1024, 456   # 5 x 4 tiles of 256 x 256, 8 K stages (last one partial)
    A, B = si.bf16_problem(77, M, N, K)
    C = run(A, B, kernel=kernel, max_clusters=max_clusters, group_m=group_m)
    assert_bf16_close(C, oracle.gemm_bf16(A, B), K, f"kernel {kernel} clusters {max_clusters} group {group_m}")


@pytest.mark.parametrize("max_clusters", [16, 9, 19])
@pytest.mark.parametrize("kernel", [g.GEMM_KERNEL_BF16_2CTA, g.GEMM_KERNEL_BF16_1CTA, g.GEMM_KERNEL_BF16_2CTA_K64,
                                    g.GEMM_KERNEL_BF16_2CTA_WIDE])
def test_tail_wave_split_into_halves(kernel, max_clusters):
    """A last wave at most half full is computed as N-halves of its tiles (N = 128 MMAs)."""
    M, N, K = 1280, 1000, 328     # 5 x 4 tiles (2-CTA) with a ragged last column block
    A, B = si.bf16_problem(31, M, N, K)
    ref = oracle.gemm_bf16(A, B)
    split = run(A, B, kernel=kernel, max_clusters=max_clusters)
    assert_bf16_close(split, ref, K, f"split, clusters {max_clusters}")
    whole = run(A, B, kernel=kernel, max_clusters=max_clusters, no_tail_split=1)
    assert_bf16_close(whole, ref, K, f"no split, clusters {max_clusters}")


@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 136, 64), (512, 512, 1024)], ids=lambda s: "x".join(map(str, s)))
def test_small_problems_split_across_clusters(shape):
    """Fewer tiles than half the co-resident clusters: every tile runs as two N-halves."""
    M, N, K = shape
    A, B = si.bf16_problem(0, M, N, K, kind="int")
    assert_bf16_exact(run(A, B), oracle.gemm_bf16(A, B), f"{shape}")


def test_integer_inputs_many_tiles_bit_exact():
    M, N, K = 1536, 1280, 1024
    A, B = si.bf16_problem(9, M, N, K, kind="int")
    assert_bf16_exact(run(A, B, max_clusters=4), oracle.gemm_bf16(A, B), "int many tiles")


def test_output_guard_band_untouched():
    """Nothing outside the M x N output is written (ragged edges are clipped by the TMA store)."""
    M, N, K = 300, 264, 128
    A, B = si.bf16_problem(5, M, N, K)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.bfloat16, device=DEV)
    sentinel = bits(buf[:pad]).copy()
    C = buf[pad:pad + M * N].view(M, N)
    g.gemm_bf16(A.to(DEV), B.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(bits(buf[:pad]), sentinel)
    assert np.array_equal(bits(buf[pad + M * N:]), sentinel)
    assert_bf16_close(bits(C), oracle.gemm_bf16(A, B), K, "guard band")


def test_empty_and_degenerate_sizes():
    C = torch.full((16, 16), 7.0, dtype=torch.bfloat16, device=DEV)
    A = torch.ones(16, 8, dtype=torch.bfloat16, device=DEV)
    g.gemm_bf16(A, A, C, 0, 16, 8)        # M = 0: nothing written
    g.gemm_bf16(A, A, C, 16, 0, 8)        # N = 0
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)
    g.gemm_bf16(A, A, C, 16, 16, 0)       # K = 0: empty sum
    torch.cuda.synchronize()
    assert torch.all(C == 0.0)


def test_rejected_arguments():
    A = torch.ones(64, 64, dtype=torch.bfloat16, device=DEV)
    C = torch.empty(64, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16(A, A, C, 64, 64, 60)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16(A.data_ptr() + 2, A, C, 64, 64, 64)
    assert e.value.status == g.GEMM_ERR_MISALIGNED


def test_all_ones_full_8192_every_element_exact():
    """Property at the full headline size: all-ones operands give C = K = 8192 everywhere."""
    M = N = K = 8192
    A = torch.ones(M, K, dtype=torch.bfloat16, device=DEV)
    C = g.matmul_bf16(A, A)
    torch.cuda.synchronize()
    assert torch.all(C == float(K)).item()


def _full_size_sampled(seed, M, N, K, kind="uniform", n=4096, exact=False):
    A, B = si.bf16_problem(seed, M, N, K, kind=kind, device=DEV)
    C = g.matmul_bf16(A, B)   # default launch: the one the benchmark times
    torch.cuda.synchronize()
    rows, cols = sample_coords(M, N, n, seed)
    got = bits(C)[rows, cols]
    ref = oracle.gemm_bf16_at(A.cpu(), B.cpu(), rows, cols)
    if exact:
        assert_bf16_exact(got, ref, f"{M}x{N}x{K} {kind}")
    else:
        assert_bf16_close(got, ref, K, f"{M}x{N}x{K}")


def _full_size_every_element(seed, M, N, K, kind="uniform", exact=False, block=2048):
    """A configuration at its full size, in the launch the benchmark times, compared with the
    oracle on every output (the oracle runs on blocks of `block` rows)."""
    A, B = si.bf16_problem(seed, M, N, K, kind=kind, device=DEV)
    C = g.matmul_bf16(A, B)
    torch.cuda.synchronize()
    got = bits(C)
    Ah, Bh = A.cpu(), B.cpu()
    for r0 in range(0, M, block):
        r1 = min(M, r0 + block)
        ref = oracle.gemm_bf16(Ah, Bh, r0, r1)
        if exact:
            assert_bf16_exact(got[r0:r1], ref, f"{M}x{N}x{K} {kind} rows {r0}..")
        else:
            assert_bf16_close(got[r0:r1], ref, K, f"{M}x{N}x{K} rows {r0}..")


def test_c2_4096_cubed_every_element():
    """4096^3 from seed 1: all 16.8M outputs (about 3 s of oracle time)."""
    _full_size_every_element(1, 4096, 4096, 4096)


def test_c3_8192_cubed_sampled():
    _full_size_sampled(2, 8192, 8192, 8192)


def test_c4_ragged_4000x14336x4096_every_element():
    """4000 x 14336 x 4096 from seed 3: all 57.3M outputs, including the last row block, whose
    second CTA holds rows 3968..3999 and reads zeros (TMA out-of-bounds fill) past row 3999.
    Blocks of 1000 rows put a block boundary inside that last 256-row tile."""
    _full_size_every_element(3, 4000, 14336, 4096, block=1000)


@pytest.mark.parametrize("shape", [(64, 28672, 8192), (1, 8192, 8192), (128, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_few_rows_full_size_sampled(shape):
    # the swapped path at full depth: a 64-row product over a 28672-wide weight (tile N 64,
    # 448 tiles), a matrix-vector product (K split over several clusters) and 128 rows
    M, N, K = shape
    assert g.bf16_plan(M, N, K)[0] == 1
    _full_size_sampled(11, M, N, K, n=min(4096, M * N))


@pytest.mark.slow
def test_c3_shape_integer_inputs_every_element_bit_exact():
    """The 8192^3 shape with integers in [-4, 4] from seed 2: |partial sums| <= 16 * 8192 <
    2^24, so every FP32 sum is exact and all 67M outputs must equal the oracle's rounding."""
    _full_size_every_element(2, 8192, 8192, 8192, kind="int", exact=True)


# ---------------------------------------------------------------- the 512 x 256 pair tile (two M-waves per CTA)

WIDE = g.GEMM_KERNEL_BF16_2CTA_WIDE


@pytest.mark.parametrize("shape", [(4000, 1000, 520), (1536, 512, 64), (513, 264, 1032), (1, 8, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_wide_tile_integer_inputs_bit_exact(shape):
    """Integer operands keep every FP32 partial sum exact, so both M-waves of each CTA (rows
    256r + 128w + lane of a 512-row tile) must reproduce the oracle bit for bit; ragged M
    cuts the last tile inside a wave, ragged N inside a 32-column store box."""
    M, N, K = shape
    A, B = si.bf16_problem(M + 2 * N + K, M, N, K, kind="int")
    assert_bf16_exact(run(A, B, kernel=WIDE), oracle.gemm_bf16(A, B), f"wide {shape}")


@pytest.mark.slow
def test_wide_tile_c4_every_element():
    """4000 x 14336 x 4096 from seed 3 on the 512 x 256 tile: all 57.3M outputs. The last
    row block (rows 3584..4095) holds 416 valid rows: its second CTA's second wave holds
    rows 3968..3999 and reads zeros past row 3999."""
    M, N, K = 4000, 14336, 4096
    A, B = si.bf16_problem(3, M, N, K, device=DEV)
    C = g.matmul_bf16(A, B, opts=g.options(kernel=WIDE))
    torch.cuda.synchronize()
    got = bits(C)
    Ah, Bh = A.cpu(), B.cpu()
    for r0 in range(0, M, 1000):
        assert_bf16_close(got[r0:r0 + 1000], oracle.gemm_bf16(Ah, Bh, r0, r0 + 1000), K, f"wide C4 rows {r0}..")


def test_default_takes_wide_tile_on_ragged_shape():
    """The default kernel choice at a ragged shape the wide-tile rule selects (72 tiles of
    512 x 256 in one wave, the last row and column blocks cut), against the oracle."""
    M, N, K = 2600, 3064, 4104
    assert g.bf16_wide_rule(M, N, K)
    A, B = si.bf16_problem(17, M, N, K)
    assert_bf16_close(run(A, B), oracle.gemm_bf16(A, B), K, "default, wide tile")


def test_wide_tile_rejects_clc():
    A = torch.ones(512, 64, dtype=torch.bfloat16, device=DEV)
    C = torch.empty(512, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16(A, A, C, 512, 512, 64, opts=g.options(kernel=WIDE, clc=g.GEMM_CLC_ON))
    assert e.value.status == g.GEMM_ERR_INVALID_ARG


def test_generator_same_values_on_gpu_and_cpu():
    a_cpu = si.uniform_bf16(3, 0, 257, 129)
    a_gpu = si.uniform_bf16(3, 0, 257, 129, device=DEV)
    assert torch.equal(a_cpu, a_gpu.cpu())
    s_cpu = si.e4m3_scales(4, 2, 64, 32)
    assert torch.equal(s_cpu, si.e4m3_scales(4, 2, 64, 32, device=DEV).cpu())


def test_one_launch_per_call():
    A, B = si.bf16_problem(0, 512, 512, 512, device=DEV)
    before = g.launch_count()
    g.matmul_bf16(A, B)
    torch.cuda.synchronize()
    assert g.launch_count() == before + 1


@pytest.mark.parametrize("kernel", [g.GEMM_KERNEL_BF16_2CTA, g.GEMM_KERNEL_BF16_1CTA, g.GEMM_KERNEL_BF16_2CTA_K64,
                                    g.GEMM_KERNEL_BF16_2CTA_WIDE])
def test_bounded_wait_reports_timeout_and_context_survives(kernel):
    """debug flag 1: the MMA issuer waits on a barrier nothing arrives on. The bounded wait
    expires (100 ms), the kernel records GEMM_ERR_TIMEOUT and exits; the context stays usable."""
    g.get_device_status()  # clear
    A, B = si.bf16_problem(0, 512, 512, 256, device=DEV)
    g.matmul_bf16(A, B, opts=g.options(kernel=kernel, wait_limit_us=100_000, debug_flags=1))
    st, detail = g.get_device_status()
    assert st == g.GEMM_ERR_TIMEOUT
    assert (detail >> 8) & 0xFF in (1, 2, 3)   # the role whose wait ran out first
    # the next GEMM on the same context is correct
    A2, B2 = si.bf16_problem(1, 256, 256, 256)
    assert_bf16_close(run(A2, B2, kernel=kernel), oracle.gemm_bf16(A2, B2), 256, "after timeout")
    assert g.get_device_status()[0] == g.GEMM_OK


def test_mma_instruction_rates():
    """The two MMA kinds the kernels issue, measured on this GPU (FLOP per SM clock). BF16:
    the documented 8192 (M=256 N=256 K=16 in 128 cycles per SM pair). The FP4 block-scaled
    kind is a multiple of it; the kernels' roofline notes depend on that ratio."""
    bf16 = g.measure_mma_rate(g.GEMM_MMA_BF16)
    fp4 = g.measure_mma_rate(g.GEMM_MMA_NVFP4)
    assert 0.9 * 8192 <= bf16 <= 1.02 * 8192, bf16
    assert 3.5 <= fp4 / bf16 <= 6.5, (bf16, fp4)
    assert g.get_device_status()[0] == g.GEMM_OK


FP4_FORMS = ["GEMM_MMA_NVFP4", "GEMM_MMA_NVFP4_1CTA_N128", "GEMM_MMA_NVFP4_1CTA_N192", "GEMM_MMA_NVFP4_1CTA_N256",
             "GEMM_MMA_NVFP4_PAIR_N128", "GEMM_MMA_NVFP4_PAIR_N128_2ACC", "GEMM_MMA_MXF4_PAIR_N256"]


def test_fp4_instruction_forms(record_property):
    """Every block-scaled FP4 form a kernel could be built from, measured back to back: each
    must run (no timeout) at a rate within the nominal FP4 range (4x to 6x of BF16 per
    clock at most). The figures are printed for the record."""
    rates = {name: g.measure_mma_rate(getattr(g, name)) for name in FP4_FORMS}
    for name, r in rates.items():
        record_property(name, r)
        print(f"{name}: {r:.0f} FLOP/clk/SM")
        assert 1000 <= r <= 6.2 * 8192, (name, r)
    assert g.get_device_status()[0] == g.GEMM_OK


@pytest.mark.parametrize("no_pdl", [0, 1])
def test_dependent_launches_on_one_stream(no_pdl):
    """Back-to-back GEMMs where each reads what the previous one wrote (read after write)
    and writes what the previous one read (write after read). With programmatic dependent
    launch the next kernel starts early, so its global accesses must still wait."""
    M = N = K = 512
    opts = g.options(no_pdl=no_pdl)
    A, B = si.bf16_problem(90, M, N, K, kind="int", device=DEV)
    _, D = si.bf16_problem(91, M, N, K, kind="int", device=DEV)
    s = torch.cuda.Stream(device=DEV)
    X = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    A2 = A.clone()
    with torch.cuda.stream(s):
        for _ in range(3):
            g.gemm_bf16(A, B, X, M, N, K, stream=s, opts=opts)       # X = A B^T
            g.gemm_bf16(X, D, Y, M, N, K, stream=s, opts=opts)       # reads X
            g.gemm_bf16(D, B, A2, M, N, K, stream=s, opts=opts)      # overwrites A2 ...
            g.gemm_bf16(A2, B, X, M, N, K, stream=s, opts=opts)      # ... then reads it, writes X
    s.synchronize()
    X_ref = oracle.gemm_bf16(A.cpu(), B.cpu())
    # the intermediate results enter the next GEMM as BF16 bit patterns (one rounding of the
    # exact FP32 sums: integer inputs keep every partial sum exact)
    Y_ref = oracle.gemm_bf16(oracle.round_bf16(X_ref), D.cpu())
    A2_ref = oracle.gemm_bf16(D.cpu(), B.cpu())
    X2_ref = oracle.gemm_bf16(oracle.round_bf16(A2_ref), B.cpu())
    assert_bf16_close(bits(Y), Y_ref, K, "Y = (A B^T) D^T")
    assert_bf16_close(bits(A2), A2_ref, K, "A2 = D B^T")
    assert_bf16_close(bits(X), X2_ref, K, "X = A2 B^T")


# ---------------------------------------------------------------- few-row GEMMs (C^T = B A^T)

SWAP_SHAPES = [
    (1, 256, 64),        # a matrix-vector product
    (7, 264, 200),       # ragged N, partial K stage
    (16, 1024, 320),
    (64, 520, 1024),     # tile N 64, ragged last 256-row block of the long dimension
    (65, 776, 136),      # tile N 128
    (128, 4104, 256),
]


@pytest.mark.parametrize("shape", SWAP_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_few_rows_swapped_against_oracle(shape):
    M, N, K = shape
    swap, tile_n = g.bf16_plan(M, N, K)
    assert swap == 1 and tile_n == (64 if M <= 64 else 128)
    A, B = si.bf16_problem(M * 7 + N + K, M, N, K)
    ref = oracle.gemm_bf16(A, B)
    assert_bf16_close(run(A, B), ref, K, f"swapped {shape}")
    assert_bf16_close(run(A, B, no_swap_ab=1), ref, K, f"not swapped {shape}")


def test_few_rows_swapped_integer_inputs_bit_exact():
    M, N, K = 48, 2048, 256
    A, B = si.bf16_problem(3, M, N, K, kind="int")
    assert_bf16_exact(run(A, B), oracle.gemm_bf16(A, B), "swapped integer")


@pytest.mark.parametrize("max_clusters", [1, 3])
def test_few_rows_swapped_many_tiles_per_cluster(max_clusters):
    M, N, K = 32, 8192, 256   # 32 tiles of the long dimension on 1 or 3 clusters
    A, B = si.bf16_problem(4, M, N, K)
    assert_bf16_close(run(A, B, max_clusters=max_clusters), oracle.gemm_bf16(A, B), K, f"clusters {max_clusters}")


def test_few_rows_swapped_guard_band_untouched():
    """The transposed stores write nothing outside C."""
    M, N, K = 40, 520, 128
    A, B = si.bf16_problem(6, M, N, K)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.bfloat16, device=DEV)
    sentinel = bits(buf[:pad]).copy()
    C = buf[pad:pad + M * N].view(M, N)
    g.gemm_bf16(A.to(DEV), B.to(DEV), C, M, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(bits(buf[:pad]), sentinel)
    assert np.array_equal(bits(buf[pad + M * N:]), sentinel)
    assert_bf16_close(bits(C), oracle.gemm_bf16(A, B), K, "guard band")


# K splits of the swapped GEMM (FP32 partials in a workspace, summed by a second kernel)
SPLIT_SHAPES = [
    # (M, N, K, launches): 3 to 8 splits add their partials in a second kernel; 2 splits run
    # as one cluster of two CTA pairs per tile, whose first pair adds the other's partials
    (16, 1024, 4096, 2),    # 4 tiles, 32 stages: 8 splits
    (100, 2048, 2048, 2),   # tile N 128, 8 tiles, 16 stages: 4 splits
    (5, 512, 2056, 2),      # 2 tiles, 17 stages (the last one ragged): 4 splits of 5, 5, 5 and 2
    (4, 8192, 6144, 1),     # tile N 64, 32 tiles, 48 stages: 2 splits (2 pairs per cluster)
    (8, 5120, 2048, 2),     # 20 tiles, 16 stages: 3 splits
]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda s: "x".join(map(str, s[:3])))
def test_few_rows_split_k_against_oracle(shape):
    M, N, K, launches = shape
    A, B = si.bf16_problem(M * 5 + N + K, M, N, K)
    ref = oracle.gemm_bf16(A, B)
    before = g.launch_count()
    got = run(A, B)
    assert g.launch_count() == before + launches
    assert_bf16_close(got, ref, K, f"split {shape}")
    assert_bf16_close(run(A, B, no_split_k=1), ref, K, f"swapped, not split {shape}")
    assert_bf16_close(run(A, B, no_swap_ab=1), ref, K, f"not swapped {shape}")
    # the same splits through the workspace and the reduction kernel (CLC requested)
    assert_bf16_close(run(A, B, clc=g.GEMM_CLC_ON), ref, K, f"split, reduction kernel {shape}")


def test_few_rows_split_k_integer_inputs_bit_exact():
    M, N, K = 32, 1024, 2048   # |partial sums| <= 16 * 2048: exact in FP32, whatever the split
    A, B = si.bf16_problem(8, M, N, K, kind="int")
    assert_bf16_exact(run(A, B), oracle.gemm_bf16(A, B), "split integer")


def test_few_rows_split_k_with_capped_clusters():
    M, N, K = 16, 512, 4096    # 2 tiles on 7 clusters: 3 splits of 11, 11 and 10 stages
    A, B = si.bf16_problem(9, M, N, K)
    assert_bf16_close(run(A, B, max_clusters=7), oracle.gemm_bf16(A, B), K, "split, 7 clusters")


@pytest.mark.parametrize("shape", [(16, 1024, 320), (100, 2056, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_few_rows_swapped_tile_per_cluster(shape):
    """persistent = 0: one cluster per tile, no K splits."""
    M, N, K = shape
    A, B = si.bf16_problem(M + N, M, N, K)
    before = g.launch_count()
    got = run(A, B, persistent=0)
    assert g.launch_count() == before + 1
    assert_bf16_close(got, oracle.gemm_bf16(A, B), K, f"tile per cluster {shape}")


@pytest.mark.slow
def test_c3_8192_cubed_every_element():
    """The headline configuration in the launch the benchmark times, compared with the
    oracle on all 67M outputs (the oracle runs in 2048-row blocks, about 25 s of host work)."""
    M = N = K = 8192
    A, B = si.bf16_problem(2, M, N, K, device=DEV)
    C = g.matmul_bf16(A, B)
    torch.cuda.synchronize()
    got = bits(C)
    Ah, Bh = A.cpu(), B.cpu()
    for r0 in range(0, M, 2048):
        assert_bf16_close(got[r0:r0 + 2048], oracle.gemm_bf16(Ah, Bh, r0, r0 + 2048), K, f"C3 rows {r0}..")


def test_split_k_calls_back_to_back_on_one_stream():
    """Split-K calls take their workspace from a stream-ordered pool and add it with a second
    launch: several in a row on one stream, each into its own output."""
    M, N, K = 16, 1024, 4096
    probs = [si.bf16_problem(70 + i, M, N, K) for i in range(3)]
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for (A, B), C in zip(probs, outs):
            g.gemm_bf16(A.to(DEV), B.to(DEV), C, M, N, K, stream=s)
    s.synchronize()
    for (A, B), C in zip(probs, outs):
        assert_bf16_close(bits(C), oracle.gemm_bf16(A, B), K, "back to back")

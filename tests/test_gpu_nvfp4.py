"""NVFP4 block-scaled GEMM on the GPU (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import oracle
import synthetic_inputs as si
from dense_tensor_core_persistent_gb300 import build as gbuild
from parity import assert_bf16_exact, assert_nvfp4_close, bits, sample_coords

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
E4M3_ONE = 0x38


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


PATHS = ["rowmajor_scales", "blocked_scales"]


def run(a, sfa, b, sfb, path="rowmajor_scales", **opt):
    """GEMM through the C ABI; the blocked path packs the scales on the GPU first."""
    opts = g.options(**opt) if opt else None
    a, sfa, b, sfb = (t.to(DEV) for t in (a, sfa, b, sfb))
    if path == "blocked_scales":
        C = g.matmul_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfb), opts=opts)
    else:
        C = g.matmul_nvfp4(a, sfa, b, sfb, opts=opts)
    torch.cuda.synchronize()
    return bits(C)


def blocked_layout_reference(sf: np.ndarray, K: int) -> np.ndarray:
    """The blocked scale layout written out from its definition in include/gemm.h."""
    rows = sf.shape[0]
    rb_count, ksteps = -(-rows // 128), K // 64
    out = np.zeros(rb_count * 128 * (K // 16), dtype=np.uint8)
    for rb in range(rb_count):
        for j in range(ksteps):
            base = (rb * ksteps + j) * 512
            for l in range(32):
                for q in range(4):
                    r = rb * 128 + l + 32 * q
                    if r < rows:
                        out[base + 16 * l + 4 * q: base + 16 * l + 4 * q + 4] = sf[r, 4 * j: 4 * j + 4]
    return out


@pytest.mark.parametrize("rows,K", [(128, 64), (300, 512), (1, 1088), (256, 4096)])
def test_pack_scales_layout(rows, K):
    sf = si.e4m3_scales(7, si.TENSOR_SFA, rows, K // 16)
    packed = g.pack_scales(sf.to(DEV))
    torch.cuda.synchronize()
    assert packed.numel() == g.nvfp4_blocked_scale_bytes(rows, K)
    assert np.array_equal(packed.cpu().numpy(), blocked_layout_reference(sf.numpy(), K))


@pytest.mark.parametrize("path", PATHS)
def test_code_points_through_the_tensor_cores(path):
    """Row 0 of A holds the 16 E2M1 codes (unit scales); B row j is one-hot at element j:
    C[0, j] must be code j's value, so the hardware's E2M1 decode matches the oracle's."""
    M, N, K = 256, 256, 256
    codes = torch.zeros(M, K, dtype=torch.uint8)
    codes[0, :16] = torch.arange(16, dtype=torch.uint8)
    onehot = torch.zeros(N, K, dtype=torch.uint8)
    onehot[torch.arange(16), torch.arange(16)] = 0x2           # 1.0
    sf = torch.full((M, K // 16), E4M3_ONE, dtype=torch.uint8)
    a, b = si.pack_e2m1(codes), si.pack_e2m1(onehot)
    got = oracle.bf16_bits_to_f64(run(a, sf, b, sf, path))
    ref = oracle.gemm_nvfp4(a, sf, b, sf)
    assert list(got[0, :16]) == list(ref[0, :16])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("path", PATHS)
def test_scale_placement_per_row_and_block(path):
    """Distinct power-of-two scales per (row, 16-block) on all-ones codes: C[i, j] is the exact
    dot product of the two scale rows, so a scale routed to the wrong row or block shows."""
    M, N, K = 256, 256, 512
    ones = torch.full((M, K), 0x2, dtype=torch.uint8)
    a = si.pack_e2m1(ones)
    rng = np.random.default_rng(3)
    sfa = torch.from_numpy(rng.choice([0x30, 0x38, 0x40, 0x48], size=(M, K // 16)).astype(np.uint8))
    sfb = torch.from_numpy(rng.choice([0x28, 0x38, 0x40], size=(N, K // 16)).astype(np.uint8))
    assert_bf16_exact(run(a, sfa, a, sfb, path), oracle.gemm_nvfp4(a, sfa, a, sfb), "scale placement")


@pytest.mark.parametrize("shape", [(256, 256, 256), (512, 512, 1024), (300, 264, 512), (1, 8, 256), (640, 768, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", PATHS)
def test_unit_scales_bit_exact(shape, path):
    """All scales 1.0: products are multiples of 1/4 and |sums| <= 36 K, exact in FP32."""
    M, N, K = shape
    a, _, b, _ = si.nvfp4_problem(11, M, N, K)
    sfa = torch.full((M, K // 16), E4M3_ONE, dtype=torch.uint8)
    sfb = torch.full((N, K // 16), E4M3_ONE, dtype=torch.uint8)
    assert_bf16_exact(run(a, sfa, b, sfb, path), oracle.gemm_nvfp4(a, sfa, b, sfb), f"{shape} {path}")


@pytest.mark.parametrize("shape", [(256, 256, 256), (512, 512, 1024), (300, 264, 512), (1000, 776, 2304)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("path", PATHS)
def test_random_scales(shape, path):
    """Codes uniform over the 16 code points, scales uniform over E4M3 values in [2^-4, 2^4]."""
    M, N, K = shape
    a, sfa, b, sfb = si.nvfp4_problem(4, M, N, K)
    assert_nvfp4_close(run(a, sfa, b, sfb, path), oracle.gemm_nvfp4(a, sfa, b, sfb), f"{shape} {path}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("max_clusters,group_m,K", [(1, 0, 1536), (3, 2, 1536), (5, 1, 1536), (1, 0, 1792), (3, 1, 2304)])
def test_many_tiles_per_cluster(max_clusters, group_m, K, path):
    # 5 x 4 tiles, 6, 7 or 9 K stages per tile: with tiles following one another on a cluster,
    # the A/B ring (6 slots) and the two scale rings (4 and 5 slots) start each tile at
    # different positions, and an odd stage count ends each tile with a single stage
    M, N = 1280, 1024
    a, sfa, b, sfb = si.nvfp4_problem(21, M, N, K)
    assert_nvfp4_close(run(a, sfa, b, sfb, path, max_clusters=max_clusters, group_m=group_m),
                       oracle.gemm_nvfp4(a, sfa, b, sfb), f"clusters {max_clusters}, K {K}")


@pytest.mark.parametrize("path", PATHS)
def test_output_guard_band_untouched(path):
    """Nothing outside the M x N output is written: the last 16-column store box of each row
    block is half outside N (264 = 16 * 16 + 8) and the last row block is cut at M."""
    M, N, K = 300, 264, 512
    a, sfa, b, sfb = (t.to(DEV) for t in si.nvfp4_problem(23, M, N, K))
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.bfloat16, device=DEV)
    sentinel = bits(buf[:pad]).copy()
    C = buf[pad:pad + M * N].view(M, N)
    if path == "blocked_scales":
        g.gemm_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfb), C, M, N, K)
    else:
        g.gemm_nvfp4(a, sfa, b, sfb, C, M, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(bits(buf[:pad]), sentinel)
    assert np.array_equal(bits(buf[pad + M * N:]), sentinel)
    assert_nvfp4_close(bits(C), oracle.gemm_nvfp4(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu()), "guard band")


@pytest.mark.parametrize("path", PATHS)
def test_c5_8192_cubed_sampled(path):
    M = N = K = 8192
    a, sfa, b, sfb = si.nvfp4_problem(4, M, N, K, device=DEV)
    if path == "blocked_scales":
        C = g.matmul_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfb))
    else:
        C = g.matmul_nvfp4(a, sfa, b, sfb)
    torch.cuda.synchronize()
    rows, cols = sample_coords(M, N, 4096, 4)
    ref = oracle.gemm_nvfp4_at(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu(), rows, cols)
    got = bits(C)[rows, cols]
    assert_nvfp4_close(got, ref, "C5 sampled")


def test_c5_shape_unit_scales_sampled_bit_exact():
    M = N = K = 8192
    a, _, b, _ = si.nvfp4_problem(4, M, N, K, device=DEV)
    sfa = torch.full((M, K // 16), E4M3_ONE, dtype=torch.uint8, device=DEV)
    C = g.matmul_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfa))
    torch.cuda.synchronize()
    rows, cols = sample_coords(M, N, 8192, 5)
    ref = oracle.gemm_nvfp4_at(a.cpu(), sfa.cpu(), b.cpu(), sfa.cpu(), rows, cols)
    assert_bf16_exact(bits(C)[rows, cols], ref, "C5 unit scales")


def test_empty_and_rejected():
    C = torch.full((16, 16), 3.0, dtype=torch.bfloat16, device=DEV)
    a = torch.zeros(16, 128, dtype=torch.uint8, device=DEV)
    sf = torch.full((16, 16), E4M3_ONE, dtype=torch.uint8, device=DEV)
    g.gemm_nvfp4(a, sf, a, sf, C, 16, 16, 0)
    torch.cuda.synchronize()
    assert torch.all(C == 0.0)
    with pytest.raises(g.GemmError) as e:
        g.gemm_nvfp4(a, sf, a, sf, C, 16, 16, 128)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("path", PATHS)
def test_bounded_wait_reports_timeout_and_context_survives(path):
    g.get_device_status()
    a, sfa, b, sfb = si.nvfp4_problem(4, 512, 512, 512, device=DEV)
    opts = g.options(wait_limit_us=100_000, debug_flags=1)
    if path == "blocked_scales":
        g.matmul_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfb), opts=opts)
    else:
        g.matmul_nvfp4(a, sfa, b, sfb, opts=opts)
    st, _ = g.get_device_status()
    assert st == g.GEMM_ERR_TIMEOUT
    a, sfa, b, sfb = si.nvfp4_problem(5, 256, 256, 256)
    assert_nvfp4_close(run(a, sfa, b, sfb, path), oracle.gemm_nvfp4(a, sfa, b, sfb), "after timeout")
    assert g.get_device_status()[0] == g.GEMM_OK


def test_concurrent_calls_on_two_streams_use_separate_workspaces():
    """gemm_nvfp4 (row-major scales) takes its scale workspace from a stream-ordered pool:
    two calls in flight on different streams must not share it."""
    M, N, K = 512, 512, 2048
    probs = [si.nvfp4_problem(40 + i, M, N, K, device=DEV) for i in range(2)]
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(3):
        for (a, sfa, b, sfb), out, s in zip(probs, outs, streams):
            g.gemm_nvfp4(a, sfa, b, sfb, out, M, N, K, stream=s)
    torch.cuda.synchronize()
    for (a, sfa, b, sfb), out in zip(probs, outs):
        ref = oracle.gemm_nvfp4(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu())
        assert_nvfp4_close(bits(out), ref, "two streams")


def test_launches_per_call():
    """gemm_nvfp4: one packing kernel for both scale matrices, then the GEMM kernel;
    gemm_nvfp4_blocked: the GEMM kernel alone."""
    M, N, K = 384, 264, 512
    a, sfa, b, sfb = si.nvfp4_problem(6, M, N, K, device=DEV)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    before = g.launch_count()
    g.gemm_nvfp4(a, sfa, b, sfb, C, M, N, K)
    torch.cuda.synchronize()
    assert g.launch_count() == before + 2
    pa, pb = g.pack_scales(sfa), g.pack_scales(sfb)
    torch.cuda.synchronize()
    before = g.launch_count()
    g.gemm_nvfp4_blocked(a, pa, b, pb, C, M, N, K)
    torch.cuda.synchronize()
    assert g.launch_count() == before + 1


# ---------------------------------------------------------------- few rows: A from a padded copy

FEW_ROW_SHAPES = [(1, 264, 512), (7, 1024, 2048), (16, 520, 256), (31, 4104, 1024)]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("shape", FEW_ROW_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_few_rows_read_a_from_padded_copy(shape, path):
    """1 <= M < 32: the GEMM reads A from a 32-row copy (rows M..31 unset). The result must
    match the oracle, and be bit-identical to reading A in place (no_pad_a = 1): the same
    rows enter the same MMAs."""
    M, N, K = shape
    assert g.nvfp4_plan(M, N, K) == 32 and g.nvfp4_plan(M, N, K, g.options(no_pad_a=1)) == M
    a, sfa, b, sfb = si.nvfp4_problem(M * 3 + N, M, N, K)
    padded = run(a, sfa, b, sfb, path)
    assert_nvfp4_close(padded, oracle.gemm_nvfp4(a, sfa, b, sfb), f"padded {shape} {path}")
    assert np.array_equal(padded, run(a, sfa, b, sfb, path, no_pad_a=1))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("shape", [(1, 28672, 8192), (16, 28672, 8192)], ids=lambda s: "x".join(map(str, s)))
def test_few_rows_full_size_every_element(shape, path):
    """A decode-sized NVFP4 GEMM (one or 16 rows against a 28672 x 8192 weight): every output
    against the oracle, through the padded copy of A (the default)."""
    M, N, K = shape
    a, sfa, b, sfb = si.nvfp4_problem(M + 7, M, N, K)
    assert_nvfp4_close(run(a, sfa, b, sfb, path), oracle.gemm_nvfp4(a, sfa, b, sfb), f"{shape} {path}")


def test_few_rows_launches_per_call():
    """Fewer than 32 rows: gemm_nvfp4's packing launch also copies A (2 launches in all);
    gemm_nvfp4_blocked launches a copy kernel before the GEMM (2); with no_pad_a, 2 and 1."""
    M, N, K = 12, 264, 512
    a, sfa, b, sfb = si.nvfp4_problem(7, M, N, K, device=DEV)
    pa, pb = g.pack_scales(sfa), g.pack_scales(sfb)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    for no_pad, want_row, want_blk in ((0, 2, 2), (1, 2, 1)):
        opts = g.options(no_pad_a=no_pad)
        before = g.launch_count()
        g.gemm_nvfp4(a, sfa, b, sfb, C, M, N, K, opts=opts)
        assert g.launch_count() == before + want_row
        before = g.launch_count()
        g.gemm_nvfp4_blocked(a, pa, b, pb, C, M, N, K, opts=opts)
        assert g.launch_count() == before + want_blk
    torch.cuda.synchronize()


@pytest.mark.parametrize("path", PATHS)
def test_few_rows_unit_scales_bit_exact(path):
    M, N, K = 5, 776, 1024
    a, _, b, _ = si.nvfp4_problem(12, M, N, K)
    sfa = torch.full((M, K // 16), E4M3_ONE, dtype=torch.uint8)
    sfb = torch.full((N, K // 16), E4M3_ONE, dtype=torch.uint8)
    assert_bf16_exact(run(a, sfa, b, sfb, path), oracle.gemm_nvfp4(a, sfa, b, sfb), f"few rows unit scales {path}")


@pytest.mark.parametrize("path", PATHS)
def test_few_rows_guard_band_untouched(path):
    """The padded rows' products (C rows M..31 of the kernel's view) are never stored."""
    M, N, K = 3, 264, 512
    a, sfa, b, sfb = (t.to(DEV) for t in si.nvfp4_problem(24, M, N, K))
    pad = 40 * N   # more than the 29 rows the padded copy adds
    buf = torch.full((M * N + 2 * pad,), 12345.0, dtype=torch.bfloat16, device=DEV)
    sentinel = bits(buf[:pad]).copy()
    C = buf[pad:pad + M * N].view(M, N)
    if path == "blocked_scales":
        g.gemm_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfb), C, M, N, K)
    else:
        g.gemm_nvfp4(a, sfa, b, sfb, C, M, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(bits(buf[:pad]), sentinel)
    assert np.array_equal(bits(buf[pad + M * N:]), sentinel)
    assert_nvfp4_close(bits(C), oracle.gemm_nvfp4(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu()), "few-row guard band")


def test_few_rows_fused_epilogue_on_padded_copy():
    M, N, K = 9, 512, 1024
    a, sfa, b, sfb = (t.to(DEV) for t in si.nvfp4_problem(25, M, N, K))
    bias = torch.linspace(-1, 1, N).to(torch.bfloat16).to(DEV)
    C0 = (torch.arange(M * N, dtype=torch.float32).reshape(M, N) / (M * N) - 0.5).to(torch.bfloat16).to(DEV)
    out = {}
    for no_pad in (0, 1):
        C = C0.clone()
        g.gemm_nvfp4_fused(a, sfa, b, sfb, C, M, N, K, g.epilogue(0.5, 1.0, bias, g.GEMM_ACT_RELU),
                           opts=g.options(no_pad_a=no_pad))
        torch.cuda.synchronize()
        out[no_pad] = bits(C)
    assert np.array_equal(out[0], out[1])
    acc = oracle.gemm_nvfp4(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu())
    ref = oracle.epilogue(acc, 0.5, 1.0, bits(C0), bits(bias), oracle.ACT_RELU)
    assert_nvfp4_close(out[0], ref, "few rows fused")


@pytest.mark.parametrize("no_pdl", [0, 1])
def test_back_to_back_calls_on_one_stream(no_pdl):
    """Consecutive gemm_nvfp4 calls on one stream: each packs its scales into a pooled
    workspace that the previous call's GEMM may have just released, and with programmatic
    dependent launch each kernel starts before the previous one ends."""
    M, N, K = 384, 512, 1024
    probs = [si.nvfp4_problem(60 + i, M, N, K, device=DEV) for i in range(4)]
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    opts = g.options(no_pdl=no_pdl)
    s = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    for rep in range(2):
        for (a, sfa, b, sfb), out in zip(probs, outs):
            g.gemm_nvfp4(a, sfa, b, sfb, out, M, N, K, stream=s, opts=opts)
    s.synchronize()
    for (a, sfa, b, sfb), out in zip(probs, outs):
        ref = oracle.gemm_nvfp4(a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu())
        assert_nvfp4_close(bits(out), ref, "back to back")


@pytest.mark.slow
def test_c5_8192_cubed_every_element():
    """C5 in the launch the benchmark times (gemm_nvfp4 on row-major scales, packed inside
    the call), compared with the oracle on all 67M outputs, in 2048-row blocks. The same
    operands through gemm_nvfp4_blocked must give the identical bits (one GEMM kernel)."""
    M = N = K = 8192
    a, sfa, b, sfb = si.nvfp4_problem(4, M, N, K, device=DEV)
    C = g.matmul_nvfp4(a, sfa, b, sfb)
    Cb = g.matmul_nvfp4_blocked(a, g.pack_scales(sfa), b, g.pack_scales(sfb))
    torch.cuda.synchronize()
    got = bits(C)
    assert np.array_equal(got, bits(Cb))
    ah, sah, bh, sbh = a.cpu(), sfa.cpu(), b.cpu(), sfb.cpu()
    for r0 in range(0, M, 2048):
        assert_nvfp4_close(got[r0:r0 + 2048], oracle.gemm_nvfp4(ah, sah, bh, sbh, r0, r0 + 2048), f"C5 rows {r0}..")

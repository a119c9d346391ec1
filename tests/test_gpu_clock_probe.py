"""gemm_options_t.clock_probe on the GPU: every CTA of the GEMM launch records %globaltimer and
its SM's clock64 at the start and the end of its work, and the result is unchanged."""
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
    yield
    st, detail = g.get_device_status()
    assert st == g.GEMM_OK, f"a kernel reported status {st} ({detail:#x})"


def check_probe(probe, elapsed_ms, pairs=True):
    """The records are the grid's CTAs 0 .. n-1 (n even for CTA pairs), each with a start
    before its end, at a clock between the idle floor and the part's maximum (2070 MHz)."""
    v = probe.view(-1, 4).cpu()
    n = int((v[:, 0] > 0).sum())
    assert n > 0 and bool((v[:n, 0] > 0).all()) and bool((v[n:] == 0).all()), "records not CTAs 0 .. n-1"
    assert bool((v[:n, 2] > v[:n, 0]).all()) and bool((v[:n, 3] > v[:n, 1]).all())
    assert not pairs or n % 2 == 0
    r = g.clock_probe_mhz(probe)
    assert r["ctas"] == n
    assert 300 <= r["sm_mhz_min"] and r["sm_mhz_max"] <= 2300, r
    # the CTAs' span lies inside the launch as the stream's events time it
    assert r["span_us"] <= elapsed_ms * 1e3 * 1.05 + 5, (r, elapsed_ms)
    return r


def timed(fn):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


# K = 8192: every CTA works for tens of microseconds, long against the timer's granularity
@pytest.mark.parametrize("kernel,shape", [
    (g.GEMM_KERNEL_BF16_2CTA_WIDE, (2048, 2048, 8192)),  # 16 tiles of 512 x 256 (as N-halves)
    (g.GEMM_KERNEL_BF16_2CTA, (1024, 1024, 8192)),       # 16 tiles of 256 x 256 (as N-halves)
    (g.GEMM_KERNEL_BF16_1CTA, (512, 512, 8192)),         # 8 tiles of 128 x 256, one CTA each
], ids=["wide", "pair", "single_cta"])
def test_bf16_kernels_record_every_cta(kernel, shape):
    M, N, K = shape
    A, B = si.bf16_problem(70, M, N, K, kind="int", device=DEV)
    probe = torch.zeros(4 * 4096, dtype=torch.int64, device=DEV)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    g.gemm_bf16(A, B, C, M, N, K, opts=g.options(kernel=kernel))  # set-up outside the timed call
    torch.cuda.synchronize()
    C.zero_()
    ms = timed(lambda: g.gemm_bf16(A, B, C, M, N, K, opts=g.options(kernel=kernel, clock_probe=probe)))
    check_probe(probe, ms, pairs=kernel != g.GEMM_KERNEL_BF16_1CTA)
    assert_bf16_exact(bits(C), oracle.gemm_bf16(A.cpu(), B.cpu()), "with the probe")


def test_nvfp4_kernel_records_every_cta():
    M, N, K = 512, 1024, 8192  # 8 tiles of 256 x 256 (the scale-packing kernel records nothing)
    a, sfa, b, sfb = si.nvfp4_problem(71, M, N, K)
    probe = torch.zeros(4 * 4096, dtype=torch.int64, device=DEV)
    ins = [t.to(DEV) for t in (a, sfa, b, sfb)]
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    g.gemm_nvfp4(*ins, C, M, N, K)
    torch.cuda.synchronize()
    ms = timed(lambda: g.gemm_nvfp4(*ins, C, M, N, K, opts=g.options(clock_probe=probe)))
    check_probe(probe, ms)
    assert_nvfp4_close(bits(C), oracle.gemm_nvfp4(a, sfa, b, sfb), "with the probe")


def test_probe_capacity_limits_the_records():
    """CTAs at or beyond clock_probe_ctas store nothing (the buffer may be shorter than the grid)."""
    M, N, K = 2048, 2048, 1024
    A, B = si.bf16_problem(72, M, N, K, device=DEV)
    buf = torch.zeros(4 * 64, dtype=torch.int64, device=DEV)
    probe = buf[: 4 * 8]  # room for 8 CTAs of the grid's 128 (32 tiles as 64 N-halves)
    g.matmul_bf16(A, B, opts=g.options(kernel=g.GEMM_KERNEL_BF16_2CTA_WIDE, clock_probe=probe))
    torch.cuda.synchronize()
    v = buf.view(-1, 4).cpu()
    assert bool((v[:8, 0] > 0).all()) and bool((v[8:] == 0).all())

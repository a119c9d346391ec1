"""Library calls captured into a CUDA graph and replayed give the results of the same calls
made directly: BF16 (static and CLC schedules), the few-row path with its K-split workspace
and reduction kernel, NVFP4 with scales packed inside the call (a pooled workspace), and a
fused epilogue that reads the C an earlier captured call wrote."""
import pytest
import torch

import dense_tensor_core_persistent_gb300 as g
import synthetic_inputs as si
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


def captured(fn, stream):
    """Run fn(stream) once eagerly (so one-time set-up happens outside the capture), then
    capture it into a graph on `stream` and return the graph."""
    fn(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        fn(stream)
    return graph


@pytest.mark.parametrize("shape,clc", [((2304, 3072, 192), g.GEMM_CLC_OFF), ((2304, 3072, 192), g.GEMM_CLC_ON),
                                       ((16, 1024, 8192), g.GEMM_CLC_AUTO), ((300, 264, 320), g.GEMM_CLC_AUTO),
                                       ((8, 8192, 8192), g.GEMM_CLC_AUTO), ((2600, 3064, 4104), g.GEMM_CLC_AUTO)],
                         ids=["static", "clc", "few_rows_split_k", "ragged", "two_pairs_per_cluster", "wide_tile"])
def test_bf16_calls_replay_from_a_graph(shape, clc):
    M, N, K = shape
    A, B = si.bf16_problem(90, M, N, K, device=DEV)
    opts = g.options(clc=clc)
    if shape == (2600, 3064, 4104):
        assert g.bf16_wide_rule(M, N, K)  # the default takes the 512 x 256 tile here
    want = g.matmul_bf16(A, B, opts=opts)
    outs = [torch.zeros(M, N, dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    stream = torch.cuda.Stream(device=DEV)

    def calls(s):
        for C in outs:
            g.gemm_bf16(A, B, C, M, N, K, s, opts)

    graph = captured(calls, stream)
    for C in outs:
        C.zero_()
    before = g.launch_count()
    for _ in range(2):
        with torch.cuda.stream(stream):
            graph.replay()
    stream.synchronize()
    assert g.launch_count() == before  # replays launch nothing from the host
    for C in outs:
        assert torch.equal(C, want)


def test_nvfp4_with_pooled_scale_workspace_replays_from_a_graph():
    M, N, K = 1000, 1000, 1792
    a, sfa, b, sfb = (t.to(DEV) for t in si.nvfp4_problem(91, M, N, K))
    want = g.matmul_nvfp4(a, sfa, b, sfb)
    C = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    stream = torch.cuda.Stream(device=DEV)
    graph = captured(lambda s: g.gemm_nvfp4(a, sfa, b, sfb, C, M, N, K, s), stream)
    C.zero_()
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    assert torch.equal(C, want)


def test_fused_epilogue_reads_what_the_previous_captured_call_wrote():
    # C = A B^T, then C = A B^T + 1 * C; the replay must give the bits of the same two calls made directly
    M, N, K = 2304, 3072, 192
    A, B = si.bf16_problem(92, M, N, K, device=DEV)
    C = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    stream = torch.cuda.Stream(device=DEV)

    def calls(s):
        g.gemm_bf16(A, B, C, M, N, K, s)
        g.gemm_bf16_fused(A, B, C, M, N, K, g.epilogue(1.0, 1.0), s)

    calls(stream)
    stream.synchronize()
    want = C.clone()
    assert not torch.equal(want, g.matmul_bf16(A, B))  # the second call did read C
    graph = captured(calls, stream)
    C.fill_(7.0)
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    assert torch.equal(C, want)

"""Several host threads calling the library at once, each on its own stream: results equal
those of the same calls made one after another. This exercises the per-thread cache of
encoded tensor maps, the per-device workspace pool (row-major NVFP4 scales and few-row
K splits take workspace inside the call), the cached occupancy queries and the launch
counter. ctypes releases the interpreter lock during each foreign call."""
import threading

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


def test_four_host_threads_on_four_streams():
    bf = [si.bf16_problem(100 + i, M, N, K, device=DEV)
          for i, (M, N, K) in enumerate([(1000, 1000, 512), (16, 2048, 4096), (2304, 3072, 192)])]
    nv = si.nvfp4_problem(103, 1000, 1000, 1792, device=DEV)
    jobs = [
        ("bf16", bf[0], None),
        ("bf16", bf[1], None),                           # few rows: K split, pooled workspace
        ("bf16", bf[2], g.options(clc=g.GEMM_CLC_ON)),   # cluster launch control
        ("nvfp4", nv, None),                             # row-major scales: pooled workspace
    ]

    def one(job):
        kind, ins, opts = job
        if kind == "bf16":
            return g.matmul_bf16(ins[0], ins[1], opts=opts)
        return g.matmul_nvfp4(*ins)

    want = [one(j) for j in jobs]
    torch.cuda.synchronize()
    reps = 20
    got = [[None] * reps for _ in jobs]
    errors = []

    def worker(t):
        try:
            torch.cuda.set_device(DEV)
            stream = torch.cuda.Stream(device=DEV)
            with torch.cuda.stream(stream):
                for r in range(reps):
                    got[t][r] = one(jobs[t])
            stream.synchronize()
        except Exception as e:  # reported below, in the test's own thread
            errors.append(e)

    before = g.launch_count()
    threads = [threading.Thread(target=worker, args=(t,)) for t in range(len(jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for t in range(len(jobs)):
        for r in range(reps):
            assert torch.equal(got[t][r], want[t]), (jobs[t][0], t, r)
    # one launch per call, two for the K-split and the row-major-scale calls
    assert g.launch_count() - before == reps * (1 + 2 + 1 + 2)

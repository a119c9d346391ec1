"""Pins for the seeded input generator (no GPU needed)."""
import os

import numpy as np
import torch

import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_first_outputs():
    with open(os.path.join(GOLDEN, "splitmix64_state0.txt")) as f:
        want = [int(l, 16) for l in f if l.strip() and not l.startswith("#")]
    assert si.splitmix64_reference(0, len(want)) == want


def test_vector_form_equals_sequential_generator():
    for seed, tid in [(0, 0), (2, 1), (4, 3), (12345, 2)]:
        s0 = si.stream_state(seed, tid)
        ref = si.splitmix64_reference(s0, 257)
        got = si.draws(seed, tid, 0, 257).numpy().view(np.uint64)
        assert [int(v) for v in got] == ref
        # an offset window is the same stream
        got2 = si.draws(seed, tid, 100, 50).numpy().view(np.uint64)
        assert [int(v) for v in got2] == ref[100:150]


def test_streams_differ_by_seed_and_tensor():
    a = si.draws(1, 0, 0, 64)
    assert not torch.equal(a, si.draws(1, 1, 0, 64))
    assert not torch.equal(a, si.draws(2, 0, 0, 64))


def test_uniform_bf16_range_and_values():
    x = si.uniform_bf16(0, 0, 256, 256)
    assert x.dtype == torch.bfloat16 and x.shape == (256, 256)
    f = x.float()
    assert f.min() >= -1 and f.max() <= 1
    assert abs(f.mean().item()) < 0.01 and abs(f.var().item() - 1 / 3) < 0.01
    # first element from the documented encoding
    d = int(si.draws(0, 0, 0, 1).numpy().view(np.uint64)[0])
    v = (d >> 40) * 2.0 ** -23 - 1.0
    assert f[0, 0].item() == torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).item()


def test_integer_twin_values():
    x = si.int_bf16(0, 0, 64, 256).float()
    vals = torch.unique(x).tolist()
    assert vals == [float(v) for v in range(-4, 5)]


def test_e2m1_codes_and_packing():
    p = si.e2m1_codes_packed(4, 0, 8, 64)
    assert p.shape == (8, 32) and p.dtype == torch.uint8
    lo, hi = p & 0xF, p >> 4
    assert sorted(torch.unique(torch.cat([lo.flatten(), hi.flatten()])).tolist()) == list(range(16))
    d = si.draws(4, 0, 0, 2).numpy().view(np.uint64)
    assert int(p[0, 0]) == (int(d[0]) >> 60) | ((int(d[1]) >> 60) << 4)


def test_e4m3_scale_codes_cover_range():
    s = si.e4m3_scales(4, 2, 512, 64)
    u = torch.unique(s).tolist()
    assert u[0] == 0x18 and u[-1] == 0x58 and len(u) == 65
    vals = s.view(torch.float8_e4m3fn).float()
    assert vals.min() == 2.0 ** -4 and vals.max() == 16.0


def test_nvfp4_problem_shapes():
    a, sfa, b, sfb = si.nvfp4_problem(4, 10, 12, 256)
    assert a.shape == (10, 128) and b.shape == (12, 128)
    assert sfa.shape == (10, 16) and sfb.shape == (12, 16)

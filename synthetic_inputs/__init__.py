"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and lays them out as the operands the
GEMM consumes (BF16 matrices, packed E2M1 codes, E4M3 scale bytes). It holds
none of the GEMM's arithmetic: no decoding, no products, no sums, no output
rounding.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast Splittable Pseudorandom
Number Generators", OOPSLA 2014; the 64-bit finaliser with the constants
0xBF58476D1CE4E5B9 / 0x94D049BB133111EB). It is used in counter form: output
``i`` (0-based) of the stream that starts in state ``s0`` is
``mix(s0 + (i + 1) * 0x9E3779B97F4A7C15)``, which equals the ``i``-th value of
the sequential generator started in ``s0``.

Every tensor gets its own stream, selected by ``(seed, tensor_id)``::

    s0 = seed * 0x9E3779B97F4A7C15  XOR  (tensor_id + 1) * 0xD1B54A32D192ED03   (mod 2**64)

with tensor ids A=0, B=1, SFA=2, SFB=3. Values are drawn in row-major order of
the logical (unpacked) tensor. Encodings of one 64-bit draw ``x``:

* uniform[-1, 1] BF16: ``u = (x >> 40) * 2**-24`` then ``v = 2u - 1`` (exact in
  FP32), then round-to-nearest-even to BF16 (torch's conversion);
* integer twin: ``((x >> 32) * 9 >> 32) - 4``, uniform over {-4..4};
* E2M1 code: ``x >> 60``, uniform over the 16 code points; two codes per byte,
  the even K index in the low nibble;
* E4M3 scale: ``0x18 + ((x >> 32) * 65 >> 32)``, uniform over the 65 E4M3
  codes whose values lie in [2**-4, 2**4].

The implementation uses torch int64 tensors (two's-complement wrap-around for
the modular multiplies, masked shifts for logical right shifts), so the same
values come out on the CPU and on a GPU.
"""
from __future__ import annotations

import torch

GOLDEN_GAMMA = 0x9E3779B97F4A7C15
STREAM_MULT = 0xD1B54A32D192ED03
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

TENSOR_A, TENSOR_B, TENSOR_SFA, TENSOR_SFB = 0, 1, 2, 3

# E4M3 codes 0x18 (2**-4) .. 0x58 (2**4): 8 binades x 8 mantissas + 16.0
E4M3_SCALE_CODE_LO = 0x18
E4M3_SCALE_CODE_COUNT = 65

_CHUNK = 1 << 23


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit integer as a signed one (for torch int64)."""
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def stream_state(seed: int, tensor_id: int) -> int:
    """Initial SplitMix64 state of the stream for (seed, tensor_id), as an unsigned int."""
    return ((seed * GOLDEN_GAMMA) ^ ((tensor_id + 1) * STREAM_MULT)) & MASK64


def splitmix64_reference(state: int, count: int) -> list[int]:
    """Sequential SplitMix64 in plain Python integers (for cross-checking the vector form)."""
    out = []
    for _ in range(count):
        state = (state + GOLDEN_GAMMA) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * MIX1) & MASK64
        z = ((z ^ (z >> 27)) * MIX2) & MASK64
        out.append(z ^ (z >> 31))
    return out


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(MIX1)
    z = (z ^ _srl(z, 27)) * _s64(MIX2)
    return z ^ _srl(z, 31)


def draws(seed: int, tensor_id: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Draws ``start .. start+count-1`` of the (seed, tensor_id) stream, as int64 bit patterns."""
    s0 = _s64(stream_state(seed, tensor_id))
    i = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return _mix(i * _s64(GOLDEN_GAMMA) + s0)


def _fill(numel: int, seed: int, tensor_id: int, encode, out: torch.Tensor) -> torch.Tensor:
    flat = out.view(-1)
    for start in range(0, numel, _CHUNK):
        n = min(_CHUNK, numel - start)
        flat[start:start + n] = encode(draws(seed, tensor_id, start, n, out.device))
    return out


def _enc_uniform_pm1(x: torch.Tensor) -> torch.Tensor:
    u24 = _srl(x, 40).to(torch.float32)          # exact: < 2**24
    return (u24 * (2.0 ** -23) - 1.0).to(torch.bfloat16)


def _enc_int9(x: torch.Tensor) -> torch.Tensor:
    return ((_srl(x, 32) * 9) >> 32) - 4


def uniform_bf16(seed: int, tensor_id: int, rows: int, cols: int, device="cpu") -> torch.Tensor:
    """rows x cols BF16 matrix, entries i.i.d. uniform on [-1, 1] (rounded to BF16)."""
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=device)
    return _fill(rows * cols, seed, tensor_id, _enc_uniform_pm1, out)


def int_bf16(seed: int, tensor_id: int, rows: int, cols: int, device="cpu") -> torch.Tensor:
    """rows x cols BF16 matrix, entries i.i.d. uniform integers in [-4, 4] (exact in BF16)."""
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=device)
    return _fill(rows * cols, seed, tensor_id, lambda x: _enc_int9(x).to(torch.bfloat16), out)


def e2m1_codes_packed(seed: int, tensor_id: int, rows: int, k: int, device="cpu") -> torch.Tensor:
    """rows x k E2M1 codes, uniform over the 16 code points, packed to rows x k/2 bytes.

    Byte j of a row holds element 2j in bits 0-3 and element 2j+1 in bits 4-7.
    """
    if k % 2:
        raise ValueError("k must be even to pack two E2M1 codes per byte")
    codes = torch.empty(rows, k, dtype=torch.uint8, device=device)
    _fill(rows * k, seed, tensor_id, lambda x: _srl(x, 60).to(torch.uint8), codes)
    return pack_e2m1(codes)


def pack_e2m1(codes: torch.Tensor) -> torch.Tensor:
    """Pack a rows x k uint8 tensor of 4-bit codes two per byte (even index in the low nibble)."""
    c = codes.to(torch.uint8)
    return (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)


def e4m3_scales(seed: int, tensor_id: int, rows: int, kblocks: int, device="cpu") -> torch.Tensor:
    """rows x kblocks E4M3 scale bytes, uniform over the 65 codes valued in [2**-4, 2**4]."""
    out = torch.empty(rows, kblocks, dtype=torch.uint8, device=device)
    enc = lambda x: (E4M3_SCALE_CODE_LO + ((_srl(x, 32) * E4M3_SCALE_CODE_COUNT) >> 32)).to(torch.uint8)
    return _fill(rows * kblocks, seed, tensor_id, enc, out)


def bf16_problem(seed: int, m: int, n: int, k: int, kind: str = "uniform", device="cpu"):
    """(A, B) for a BF16 GEMM C = A B^T: A is m x k, B is n x k.

    kind = "uniform" (entries in [-1, 1]) or "int" (integers in [-4, 4]).
    """
    gen = uniform_bf16 if kind == "uniform" else int_bf16
    return gen(seed, TENSOR_A, m, k, device), gen(seed, TENSOR_B, n, k, device)


def nvfp4_problem(seed: int, m: int, n: int, k: int, device="cpu"):
    """(A, SFA, B, SFB) for an NVFP4 GEMM: packed codes m x k/2 and n x k/2, scales m x k/16 and n x k/16."""
    if k % 16:
        raise ValueError("k must be a multiple of 16 (one scale per 16 K-elements)")
    a = e2m1_codes_packed(seed, TENSOR_A, m, k, device)
    b = e2m1_codes_packed(seed, TENSOR_B, n, k, device)
    sfa = e4m3_scales(seed, TENSOR_SFA, m, k // 16, device)
    sfb = e4m3_scales(seed, TENSOR_SFB, n, k // 16, device)
    return a, sfa, b, sfb


def rotation_seed(seed: int, r: int) -> int:
    """Seed of rotation set r (r = 0 is the parity-checked set)."""
    return seed + 1000 * r

"""CPU oracle for C = A * B^T (BF16 and NVFP4 block-scaled), in FP64.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only users. The product path
(the CUDA library and its binding) never imports this package.

The arithmetic lives in ``oracle.c`` (plain C, OpenMP over output rows); this
module compiles it with gcc on first use and marshals numpy / torch CPU arrays.
See the header of ``oracle.c`` for the definitions followed and their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, OpenMP when available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB_OVERRIDE loads a deliberately broken copy (mutation tests only)
            l = ctypes.CDLL(os.environ.get("ORACLE_LIB_OVERRIDE") or build())
            l.oracle_dec_bf16.restype = ctypes.c_double
            l.oracle_dec_bf16.argtypes = [ctypes.c_uint16]
            l.oracle_dec_e2m1.restype = ctypes.c_double
            l.oracle_dec_e2m1.argtypes = [ctypes.c_uint8]
            l.oracle_dec_e4m3.restype = ctypes.c_double
            l.oracle_dec_e4m3.argtypes = [ctypes.c_uint8]
            l.oracle_bf16_rne.restype = ctypes.c_uint16
            l.oracle_bf16_rne.argtypes = [ctypes.c_double]
            l.oracle_round_bf16.restype = None
            l.oracle_round_bf16.argtypes = [_P, _I64, _P]
            l.oracle_gemm_bf16.restype = ctypes.c_int
            l.oracle_gemm_bf16.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _I64, _P]
            l.oracle_gemm_bf16_at.restype = None
            l.oracle_gemm_bf16_at.argtypes = [_P, _P, _I64, _P, _P, _I64, _P]
            l.oracle_gemm_nvfp4.restype = ctypes.c_int
            l.oracle_gemm_nvfp4.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P]
            l.oracle_gemm_nvfp4_at.restype = None
            l.oracle_gemm_nvfp4_at.argtypes = [_P, _P, _P, _P, _I64, _P, _P, _I64, _P]
            l.oracle_num_threads.restype = ctypes.c_int
            _lib = l
    return _lib


def _np(x, dtype) -> np.ndarray:
    """Contiguous numpy view/copy of a numpy array or CPU torch tensor, reinterpreted as dtype."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must live in host memory")
        x = x.contiguous()
        if x.dtype.itemsize != np.dtype(dtype).itemsize:
            raise ValueError(f"expected {np.dtype(dtype).itemsize}-byte elements, got {x.dtype}")
        x = x.view(torch_int_dtype(np.dtype(dtype).itemsize)).numpy()
    x = np.ascontiguousarray(x)
    return x.view(dtype)


def torch_int_dtype(itemsize: int):
    import torch
    return {1: torch.uint8, 2: torch.int16, 8: torch.int64}[itemsize]


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def dec_bf16(bits: int) -> float:
    return lib().oracle_dec_bf16(bits)


def dec_e2m1(code: int) -> float:
    return lib().oracle_dec_e2m1(code)


def dec_e4m3(code: int) -> float:
    return lib().oracle_dec_e4m3(code)


def bf16_rne(x: float) -> int:
    return lib().oracle_bf16_rne(float(x))


def round_bf16(x) -> np.ndarray:
    """Round an array of doubles to BF16 bit patterns (uint16), nearest-even, one step."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_round_bf16(_ptr(x), x.size, _ptr(out))
    return out


def gemm_bf16(A, B, row0: int = 0, row1: int | None = None) -> np.ndarray:
    """FP64 C = A * B^T (rows row0..row1-1). A: M x K, B: N x K BF16 (torch bf16 or uint16 bits)."""
    a = _np(A, np.uint16)
    b = _np(B, np.uint16)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("A and B must have the same K")
    row1 = M if row1 is None else row1
    C = np.empty((row1 - row0, N), dtype=np.float64)
    if lib().oracle_gemm_bf16(_ptr(a), _ptr(b), M, N, K, row0, row1, _ptr(C)) != 0:
        raise MemoryError("oracle_gemm_bf16: out of host memory")
    return C


def gemm_bf16_at(A, B, rows, cols) -> np.ndarray:
    """FP64 C[rows[t], cols[t]] for a list of output coordinates."""
    a = _np(A, np.uint16)
    b = _np(B, np.uint16)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= a.shape[0] or c.min() < 0 or c.max() >= b.shape[0]):
        raise IndexError("output coordinate out of range")
    out = np.empty(r.size, dtype=np.float64)
    lib().oracle_gemm_bf16_at(_ptr(a), _ptr(b), a.shape[1], _ptr(r), _ptr(c), r.size, _ptr(out))
    return out


def gemm_nvfp4(A, SFA, B, SFB, row0: int = 0, row1: int | None = None) -> np.ndarray:
    """FP64 C = A * B^T for packed E2M1 codes with per-16 E4M3 scales (rows row0..row1-1)."""
    a, sa, b, sb = (_np(t, np.uint8) for t in (A, SFA, B, SFB))
    M, Kh = a.shape
    N = b.shape[0]
    K = 2 * Kh
    if b.shape[1] != Kh or sa.shape != (M, K // 16) or sb.shape != (N, K // 16):
        raise ValueError("inconsistent NVFP4 operand shapes")
    row1 = M if row1 is None else row1
    C = np.empty((row1 - row0, N), dtype=np.float64)
    if lib().oracle_gemm_nvfp4(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K, row0, row1, _ptr(C)) != 0:
        raise MemoryError("oracle_gemm_nvfp4: out of host memory")
    return C


def gemm_nvfp4_at(A, SFA, B, SFB, rows, cols) -> np.ndarray:
    a, sa, b, sb = (_np(t, np.uint8) for t in (A, SFA, B, SFB))
    K = 2 * a.shape[1]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= a.shape[0] or c.min() < 0 or c.max() >= b.shape[0]):
        raise IndexError("output coordinate out of range")
    out = np.empty(r.size, dtype=np.float64)
    lib().oracle_gemm_nvfp4_at(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), K, _ptr(r), _ptr(c), r.size, _ptr(out))
    return out


def num_threads() -> int:
    return lib().oracle_num_threads()


def ulp_bf16(r_bits: np.ndarray) -> np.ndarray:
    """One BF16 ulp at each value R (given as BF16 bits): 2^(max(floor(log2|R|), -126) - 7); 2^-133 at zero."""
    bits = np.asarray(r_bits, dtype=np.uint16)
    exp_field = ((bits >> 7) & 0xFF).astype(np.int64)
    e = np.where(exp_field == 0, -126, exp_field - 127)
    return np.ldexp(1.0, (e - 7).astype(np.int32))


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- fused epilogue
# "NVFP4 GEMM on Blackwell", epilogue section: activation, bias and alpha/beta scaling are
# applied to the accumulator before it is stored. Reading taken here (the page names the
# operations, not their order): x = alpha * acc + beta * C_old + bias[col], then the
# activation, then one rounding to BF16.

ACT_NONE, ACT_RELU, ACT_GELU_TANH = 0, 1, 2


def gelu_tanh(x) -> np.ndarray:
    """GELU in its tanh form, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), in FP64."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x * x * x)))


def epilogue(acc, alpha=1.0, beta=0.0, c_old=None, bias=None, activation=ACT_NONE) -> np.ndarray:
    """FP64 value of act(alpha * acc + beta * C_old + bias[col]) before the rounding to BF16.

    acc: FP64 products, M x N. alpha, beta: taken at FP32 precision (the C ABI passes floats).
    c_old: BF16 bits of the prior C (M x N), read only when beta != 0. bias: BF16 bits, N
    values (one per column), or None."""
    alpha = float(np.float32(alpha))
    beta = float(np.float32(beta))
    x = alpha * np.asarray(acc, dtype=np.float64)
    if beta != 0.0:
        x = x + beta * bf16_bits_to_f64(c_old)
    if bias is not None:
        x = x + bf16_bits_to_f64(bias)[None, :]
    if activation == ACT_RELU:
        x = np.maximum(x, 0.0)
    elif activation == ACT_GELU_TANH:
        x = gelu_tanh(x)
    elif activation != ACT_NONE:
        raise ValueError("unknown activation")
    return x

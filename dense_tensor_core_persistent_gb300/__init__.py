"""Python binding of the GB300 (sm_103a) dense tensor-core GEMM library.

Argument marshalling only: every step of the GEMM runs in the CUDA kernels of
``_lib/libdtcp_gemm.so`` (built by ``build.py``), called through its C ABI
(``include/gemm.h``). There is no CPU or PyTorch fallback: if the library is
missing, importing the binding's functions raises.

Functions take raw device pointers (ints) or torch CUDA tensors; ``stream``
defaults to torch's current CUDA stream when torch is importable, else the
legacy default stream.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libdtcp_gemm.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED_SHAPE = 2
GEMM_ERR_MISALIGNED = 3
GEMM_ERR_NO_DEVICE = 4
GEMM_ERR_ARCH = 5
GEMM_ERR_DRIVER = 6
GEMM_ERR_LAUNCH = 7
GEMM_ERR_TIMEOUT = 8
GEMM_ERR_OUT_OF_MEMORY = 9
GEMM_ERR_SCRATCH_TOO_SMALL = 10
NVFP4_NOALLOC_SCRATCH_BYTES = 16 << 20

GEMM_KERNEL_DEFAULT = 0
GEMM_KERNEL_BF16_1CTA = 1
GEMM_KERNEL_BF16_2CTA = 2
GEMM_KERNEL_BF16_2CTA_K64 = 3
GEMM_KERNEL_BF16_2CTA_WIDE = 4

# Entry points declared in include/gemm.h (the CPU tests check the library exports all of them).
EXPORTS = (
    "gemm_bf16", "gemm_nvfp4", "gemm_status_string", "gemm_get_device_status", "gemm_bf16_ex",
    "gemm_nvfp4_ex", "gemm_tile_coord", "gemm_choose_group_m", "gemm_launch_count",
    "gemm_nvfp4_blocked_scale_bytes", "gemm_nvfp4_pack_scales", "gemm_nvfp4_blocked", "gemm_nvfp4_blocked_ex",
    "gemm_nvfp4_noalloc", "gemm_measure_mma_rate", "gemm_bf16_fused", "gemm_nvfp4_fused", "gemm_nvfp4_blocked_fused",
    "gemm_bf16_plan", "gemm_clc_rule", "gemm_nvfp4_plan", "gemm_bf16_wide_rule",
)

# gemm_activation_t
GEMM_ACT_NONE = 0
GEMM_ACT_RELU = 1
GEMM_ACT_GELU_TANH = 2


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class gemm_options_t(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int),
        ("persistent", ctypes.c_int),
        ("group_m", ctypes.c_int),
        ("max_clusters", ctypes.c_int),
        ("wait_limit_us", ctypes.c_uint32),
        ("debug_flags", ctypes.c_uint32),
        ("no_tail_split", ctypes.c_int),
        ("no_pdl", ctypes.c_int),
        ("no_swap_ab", ctypes.c_int),
        ("no_split_k", ctypes.c_int),
        ("clc", ctypes.c_int),
        ("no_pad_a", ctypes.c_int),
        ("clock_probe", ctypes.c_void_p),
        ("clock_probe_ctas", ctypes.c_int),
    ]


# gemm_options_t.clc
GEMM_CLC_AUTO = 0
GEMM_CLC_ON = 1
GEMM_CLC_OFF = 2


def options(kernel=GEMM_KERNEL_DEFAULT, persistent=1, group_m=0, max_clusters=0, wait_limit_us=0, debug_flags=0,
            no_tail_split=0, no_pdl=0, no_swap_ab=0, no_split_k=0, clc=GEMM_CLC_AUTO, no_pad_a=0, clock_probe=None):
    """`clock_probe`: None, or a CUDA int64 tensor of 4 values per CTA (see clock_probe_mhz)."""
    probe, probe_ctas = None, 0
    if clock_probe is not None:
        probe, probe_ctas = _ptr(clock_probe), clock_probe.numel() // 4
    return gemm_options_t(kernel, persistent, group_m, max_clusters, wait_limit_us, debug_flags, no_tail_split, no_pdl,
                          no_swap_ab, no_split_k, clc, no_pad_a, probe, probe_ctas)


def clock_probe_mhz(probe) -> dict:
    """Reads a clock probe after the launch completed (gemm_options_t.clock_probe): each CTA's
    SM clock over its work (clock64 difference / %globaltimer difference), the median and
    range over the CTAs that recorded, and the span from the first start to the last end."""
    v = probe.view(-1, 4).cpu().tolist()
    rec = [r for r in v if r[0] and r[2] > r[0]]
    if not rec:
        return {"ctas": 0}
    mhz = sorted((r[3] - r[1]) / (r[2] - r[0]) * 1e3 for r in rec)
    span_us = (max(r[2] for r in rec) - min(r[0] for r in rec)) / 1e3
    return {"ctas": len(rec), "sm_mhz": mhz[len(mhz) // 2], "sm_mhz_min": mhz[0], "sm_mhz_max": mhz[-1],
            "span_us": span_us}


class gemm_epilogue_t(ctypes.Structure):
    _fields_ = [
        ("alpha", ctypes.c_float),
        ("beta", ctypes.c_float),
        ("bias", ctypes.c_void_p),
        ("activation", ctypes.c_int),
        ("reserved", ctypes.c_int),
    ]


def epilogue(alpha=1.0, beta=0.0, bias=None, activation=GEMM_ACT_NONE) -> gemm_epilogue_t:
    """C = act(alpha * A B^T + beta * C + bias[col]); `bias` is a device tensor of N BF16 values or None."""
    return gemm_epilogue_t(alpha, beta, None if bias is None else _ptr(bias), activation, 0)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m dense_tensor_core_persistent_gb300.build` "
                "(the GEMM has no CPU fallback)")
        l = ctypes.CDLL(LIB_PATH)
        P, I = ctypes.c_void_p, ctypes.c_int
        l.gemm_bf16.argtypes = [P, P, P, I, I, I, P]
        l.gemm_bf16.restype = I
        l.gemm_bf16_ex.argtypes = [P, P, P, I, I, I, P, ctypes.POINTER(gemm_options_t)]
        l.gemm_bf16_ex.restype = I
        l.gemm_nvfp4.argtypes = [P, P, P, P, P, I, I, I, P]
        l.gemm_nvfp4.restype = I
        l.gemm_nvfp4_ex.argtypes = [P, P, P, P, P, I, I, I, P, ctypes.POINTER(gemm_options_t)]
        l.gemm_nvfp4_ex.restype = I
        l.gemm_status_string.argtypes = [I]
        l.gemm_status_string.restype = ctypes.c_char_p
        l.gemm_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        l.gemm_get_device_status.restype = I
        l.gemm_tile_coord.argtypes = [I, I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]
        l.gemm_tile_coord.restype = I
        l.gemm_choose_group_m.argtypes = [I, I, I, I, I, I, I, ctypes.c_longlong]
        l.gemm_choose_group_m.restype = I
        l.gemm_clc_rule.argtypes = [I, I, I, I]
        l.gemm_clc_rule.restype = I
        l.gemm_nvfp4_blocked_scale_bytes.argtypes = [I, I]
        l.gemm_nvfp4_blocked_scale_bytes.restype = ctypes.c_longlong
        l.gemm_nvfp4_pack_scales.argtypes = [P, P, I, I, P]
        l.gemm_nvfp4_pack_scales.restype = I
        l.gemm_nvfp4_blocked.argtypes = [P, P, P, P, P, I, I, I, P]
        l.gemm_nvfp4_blocked.restype = I
        l.gemm_nvfp4_blocked_ex.argtypes = [P, P, P, P, P, I, I, I, P, ctypes.POINTER(gemm_options_t)]
        l.gemm_nvfp4_blocked_ex.restype = I
        l.gemm_nvfp4_noalloc.argtypes = [P, P, P, P, P, I, I, I, P]
        l.gemm_nvfp4_noalloc.restype = I
        l.gemm_launch_count.argtypes = []
        l.gemm_launch_count.restype = ctypes.c_ulonglong
        l.gemm_measure_mma_rate.argtypes = [I, ctypes.POINTER(ctypes.c_double)]
        EP, OP = ctypes.POINTER(gemm_epilogue_t), ctypes.POINTER(gemm_options_t)
        l.gemm_bf16_fused.argtypes = [P, P, P, I, I, I, P, EP, OP]
        l.gemm_bf16_fused.restype = I
        l.gemm_nvfp4_fused.argtypes = [P, P, P, P, P, I, I, I, P, EP, OP]
        l.gemm_nvfp4_fused.restype = I
        l.gemm_nvfp4_blocked_fused.argtypes = [P, P, P, P, P, I, I, I, P, EP, OP]
        l.gemm_nvfp4_blocked_fused.restype = I
        l.gemm_bf16_plan.argtypes = [I, I, I, OP, EP, ctypes.POINTER(I), ctypes.POINTER(I)]
        l.gemm_bf16_plan.restype = I
        l.gemm_nvfp4_plan.argtypes = [I, I, I, OP, ctypes.POINTER(I)]
        l.gemm_nvfp4_plan.restype = I
        l.gemm_bf16_wide_rule.argtypes = [I, I, I, I]
        l.gemm_bf16_wide_rule.restype = I
        l.gemm_measure_mma_rate.restype = I
        _lib = l
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != GEMM_OK:
        raise GemmError(status, where)


def status_string(status: int) -> str:
    return lib().gemm_status_string(status).decode()


def gemm_bf16(A, B, C, M: int, N: int, K: int, stream=None, opts: gemm_options_t | None = None) -> None:
    """C[M,N] = A[M,K] @ B[N,K]^T in BF16 (FP32 accumulation); see include/gemm.h."""
    l = lib()
    if opts is None:
        st = l.gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(stream))
    else:
        st = l.gemm_bf16_ex(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(stream), ctypes.byref(opts))
    _check(st, "gemm_bf16")


def gemm_nvfp4(A, SFA, B, SFB, C, M: int, N: int, K: int, stream=None, opts: gemm_options_t | None = None) -> None:
    """C[M,N] = dequant(A, SFA) @ dequant(B, SFB)^T for packed E2M1 with per-16 E4M3 scales."""
    l = lib()
    if opts is None:
        st = l.gemm_nvfp4(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _stream(stream))
    else:
        st = l.gemm_nvfp4_ex(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _stream(stream),
                             ctypes.byref(opts))
    _check(st, "gemm_nvfp4")


def nvfp4_blocked_scale_bytes(rows: int, K: int) -> int:
    n = lib().gemm_nvfp4_blocked_scale_bytes(rows, K)
    if n < 0:
        raise GemmError(GEMM_ERR_UNSUPPORTED_SHAPE, "gemm_nvfp4_blocked_scale_bytes")
    return n


def gemm_nvfp4_pack_scales(SF, SF_blocked, rows: int, K: int, stream=None) -> None:
    """Row-major scales [rows][K/16] -> the blocked tensor-core layout (see include/gemm.h)."""
    _check(lib().gemm_nvfp4_pack_scales(_ptr(SF), _ptr(SF_blocked), rows, K, _stream(stream)),
           "gemm_nvfp4_pack_scales")


def gemm_nvfp4_blocked(A, SFA_blocked, B, SFB_blocked, C, M: int, N: int, K: int, stream=None,
                       opts: gemm_options_t | None = None) -> None:
    """gemm_nvfp4 with scales already in the blocked layout (the fast path)."""
    l = lib()
    if opts is None:
        st = l.gemm_nvfp4_blocked(_ptr(A), _ptr(SFA_blocked), _ptr(B), _ptr(SFB_blocked), _ptr(C), M, N, K,
                                  _stream(stream))
    else:
        st = l.gemm_nvfp4_blocked_ex(_ptr(A), _ptr(SFA_blocked), _ptr(B), _ptr(SFB_blocked), _ptr(C), M, N, K,
                                     _stream(stream), ctypes.byref(opts))
    _check(st, "gemm_nvfp4_blocked")


def _byref_or_null(x):
    return None if x is None else ctypes.byref(x)


def gemm_bf16_fused(A, B, C, M: int, N: int, K: int, epi: gemm_epilogue_t | None = None, stream=None,
                    opts: gemm_options_t | None = None) -> None:
    """gemm_bf16 with the fused epilogue C = act(alpha * A B^T + beta * C + bias)."""
    _check(lib().gemm_bf16_fused(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(stream), _byref_or_null(epi),
                                 _byref_or_null(opts)), "gemm_bf16_fused")


def gemm_nvfp4_fused(A, SFA, B, SFB, C, M: int, N: int, K: int, epi: gemm_epilogue_t | None = None, stream=None,
                     opts: gemm_options_t | None = None) -> None:
    """gemm_nvfp4 with the fused epilogue."""
    _check(lib().gemm_nvfp4_fused(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _stream(stream),
                                  _byref_or_null(epi), _byref_or_null(opts)), "gemm_nvfp4_fused")


def gemm_nvfp4_blocked_fused(A, SFA_blocked, B, SFB_blocked, C, M: int, N: int, K: int,
                             epi: gemm_epilogue_t | None = None, stream=None,
                             opts: gemm_options_t | None = None) -> None:
    """gemm_nvfp4_blocked with the fused epilogue."""
    _check(lib().gemm_nvfp4_blocked_fused(_ptr(A), _ptr(SFA_blocked), _ptr(B), _ptr(SFB_blocked), _ptr(C), M, N, K,
                                          _stream(stream), _byref_or_null(epi), _byref_or_null(opts)),
           "gemm_nvfp4_blocked_fused")


def bf16_plan(M: int, N: int, K: int, opts: gemm_options_t | None = None, epi: gemm_epilogue_t | None = None):
    """(swap_ab, tile_n) that gemm_bf16 uses for this problem (host only)."""
    swap, tile_n = ctypes.c_int(), ctypes.c_int()
    _check(lib().gemm_bf16_plan(M, N, K, _byref_or_null(opts), _byref_or_null(epi), ctypes.byref(swap),
                                ctypes.byref(tile_n)), "gemm_bf16_plan")
    return swap.value, tile_n.value


def bf16_wide_rule(M: int, N: int, K: int, wave: int = 76) -> bool:
    """Whether gemm_bf16's default kernel takes the 512 x 256 pair tile for this problem
    (static schedule, not swapped), with `wave` co-resident clusters."""
    r = lib().gemm_bf16_wide_rule(M, N, K, wave)
    if r < 0:
        raise GemmError(-r, "gemm_bf16_wide_rule")
    return r == 1


def nvfp4_plan(M: int, N: int, K: int, opts: gemm_options_t | None = None) -> int:
    """Rows of A the NVFP4 GEMM kernel reads for this problem: 32 when A is copied into a
    padded workspace first, else M (host only)."""
    a_rows = ctypes.c_int()
    _check(lib().gemm_nvfp4_plan(M, N, K, _byref_or_null(opts), ctypes.byref(a_rows)), "gemm_nvfp4_plan")
    return a_rows.value


def gemm_nvfp4_noalloc(A, SFA, B, SFB, C, M: int, N: int, K: int, stream=None) -> None:
    """gemm_nvfp4 without any device allocation: the rearranged scales live in a fixed
    16 MiB array inside the library (see include/gemm.h for the size limit and the
    rule that calls overlapping on the GPU must be ordered)."""
    _check(lib().gemm_nvfp4_noalloc(_ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), _ptr(C), M, N, K, _stream(stream)),
           "gemm_nvfp4_noalloc")


def get_device_status(stream=None) -> tuple[int, int]:
    """(status, detail word) reported by kernels since the last call; synchronises the stream."""
    detail = ctypes.c_uint32(0)
    st = lib().gemm_get_device_status(_stream(stream), ctypes.byref(detail))
    return st, detail.value


def tile_coord(M, N, tile_m, tile_n, group_m, t) -> tuple[int, int]:
    mb, nb = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().gemm_tile_coord(M, N, tile_m, tile_n, group_m, t, ctypes.byref(mb), ctypes.byref(nb)),
           "gemm_tile_coord")
    return mb.value, nb.value


def choose_group_m(M, N, K, tile_m, tile_n, elem_bytes_x2, concurrent_tiles, l2_bytes) -> int:
    g = lib().gemm_choose_group_m(M, N, K, tile_m, tile_n, elem_bytes_x2, concurrent_tiles, l2_bytes)
    if g < 0:
        raise GemmError(-g, "gemm_choose_group_m")
    return g


def clc_rule(items: int, wave: int, K: int, nvfp4: bool = False) -> bool:
    """Whether a persistent launch with the default options schedules its items with cluster launch control."""
    r = lib().gemm_clc_rule(items, wave, K, int(nvfp4))
    if r < 0:
        raise GemmError(-r, "gemm_clc_rule")
    return r == 1


def launch_count() -> int:
    return lib().gemm_launch_count()


GEMM_MMA_BF16 = 0
GEMM_MMA_NVFP4 = 1
GEMM_MMA_NVFP4_1CTA_N128 = 2
GEMM_MMA_NVFP4_1CTA_N192 = 3
GEMM_MMA_NVFP4_1CTA_N256 = 4
GEMM_MMA_NVFP4_PAIR_N128 = 5
GEMM_MMA_NVFP4_PAIR_N128_2ACC = 6
GEMM_MMA_MXF4_PAIR_N256 = 7


def measure_mma_rate(kind: int) -> float:
    """FLOP per SM clock of back-to-back M=256 N=256 MMAs of `kind` on the current device."""
    out = ctypes.c_double(0.0)
    _check(lib().gemm_measure_mma_rate(kind, ctypes.byref(out)), "gemm_measure_mma_rate")
    return out.value


# ---------------------------------------------------------------- torch-tensor conveniences

def matmul_bf16(A, B, out=None, stream=None, opts=None):
    """A (M x K) and B (N x K) BF16 CUDA tensors -> C = A @ B^T (M x N BF16)."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    gemm_bf16(A, B, out, M, N, K, stream, opts)
    return out


def pack_scales(SF, stream=None):
    """Row-major E4M3 scales (rows x K/16 uint8 CUDA tensor) -> blocked-layout uint8 tensor."""
    import torch
    rows, kb = SF.shape
    K = 16 * kb
    out = torch.empty(nvfp4_blocked_scale_bytes(rows, K), dtype=torch.uint8, device=SF.device)
    gemm_nvfp4_pack_scales(SF, out, rows, K, stream)
    return out


def matmul_nvfp4_blocked(A, SFA_blocked, B, SFB_blocked, out=None, stream=None, opts=None):
    """Like matmul_nvfp4, with scales from pack_scales."""
    import torch
    M = A.shape[0]
    N = B.shape[0]
    K = 2 * A.shape[1]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    gemm_nvfp4_blocked(A, SFA_blocked, B, SFB_blocked, out, M, N, K, stream, opts)
    return out


def matmul_nvfp4(A, SFA, B, SFB, out=None, stream=None, opts=None):
    """Packed E2M1 A (M x K/2), B (N x K/2) with E4M3 scales (M x K/16, N x K/16) -> BF16 C."""
    import torch
    M = A.shape[0]
    N = B.shape[0]
    K = 2 * A.shape[1]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    gemm_nvfp4(A, SFA, B, SFB, out, M, N, K, stream, opts)
    return out

"""Python binding of the GB300 FP8 fine-grained-scaled GEMM library (libdg.so).

Argument marshalling only: every function takes CUDA torch tensors, derives
the sizes, and calls the C entry point of the same name in ``include/dg.h`` on
the current torch stream.  All computation happens in the library's sm_103a
kernels; there is no fallback.  If ``libdg.so`` has not been built, importing
the native functions raises ``RuntimeError``.

Layouts (see ``include/dg.h``):
  A uint8 [M, K]; SFA fp32 [K/128, round_up(M, 4)]
  B uint8 [N, K] (or [G, N, K]); SFB fp32 [ceil(N/128), K/128] (or [G, ...])
  D bf16 [M, N]
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdg.so")
QBLOCK = 128

DG_OK = 0
DG_ERR_INVALID_ARG = 1
DG_ERR_UNSUPPORTED_SHAPE = 2
DG_ERR_MISALIGNED = 3
DG_ERR_UNSUPPORTED_DEVICE = 4
DG_ERR_CUDA = 5
DG_ERR_DEVICE_TIMEOUT = 6

DG_DTYPE_F32 = 0
DG_DTYPE_BF16 = 1

DG_LAYOUT_DENSE = 0
DG_LAYOUT_CONTIGUOUS = 1
DG_LAYOUT_MASKED = 2

DG_DEVFLAG_MASKED_M_CLAMPED = 0x1
DG_DEVFLAG_BAD_EXPERT = 0x2
DG_DEVFLAG_MIXED_BLOCK = 0x4
DG_DEVFLAG_TIMEOUT = 0x8

# every symbol include/dg.h declares
EXPORTED = (
    "dg_quant_act_1x128",
    "dg_quant_weight_128x128",
    "dg_fp8_gemm_nt",
    "dg_fp8_grouped_contiguous",
    "dg_fp8_grouped_masked",
    "dg_fp8_gemm_nt_q",
    "dg_fp8_grouped_contiguous_q",
    "dg_fp8_grouped_masked_q",
    "dg_query_plan",
    "dg_status_string",
    "dg_read_device_status",
)


class DgError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


class dg_plan_t(ctypes.Structure):
    _fields_ = [("block_m", ctypes.c_int), ("block_n", ctypes.c_int), ("stages", ctypes.c_int),
                ("num_tiles", ctypes.c_int), ("grid", ctypes.c_int), ("smem_bytes", ctypes.c_int)]


_lib = None


def build(force: bool = False) -> str:
    """Compile libdg.so in-tree with nvcc (sm_103a)."""
    from . import _build
    return _build.build(force=force)


def load() -> ctypes.CDLL:
    """Load libdg.so (raises RuntimeError if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with moe_grouped_gemm_x128_gb300.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    sig = {
        "dg_quant_act_1x128": [P, I, P, P, I, I, P],
        "dg_quant_weight_128x128": [P, P, P, I, I, I, P],
        "dg_fp8_gemm_nt": [P, P, P, P, P, I, I, I, P],
        "dg_fp8_grouped_contiguous": [P, P, P, P, P, P, I, I, I, I, P],
        "dg_fp8_grouped_masked": [P, P, P, P, P, P, I, I, I, I, I, P],
        "dg_fp8_gemm_nt_q": [P, P, P, P, P, P, I, I, I, P],
        "dg_fp8_grouped_contiguous_q": [P, P, P, P, P, P, P, I, I, I, I, P],
        "dg_fp8_grouped_masked_q": [P, P, P, P, P, P, P, I, I, I, I, I, P],
        "dg_query_plan": [I, I, I, I, I, I, ctypes.POINTER(dg_plan_t)],
        "dg_read_device_status": [ctypes.POINTER(ctypes.c_int), P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = I
    lib.dg_status_string.argtypes = [I]
    lib.dg_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().dg_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != DG_OK:
        raise DgError(fn, status, status_string(status))


_raw_stream = None


def _stream(stream) -> int | None:
    """The stream handle to launch on: `stream` if given, else the current
    torch stream of the current device (where the library launches)."""
    global _raw_stream
    if stream is not None:
        return int(stream)
    import torch
    if _raw_stream is None:
        # PyTorch's raw current-stream accessor costs a fraction of building
        # a Stream object (torch.cuda.current_stream()) on every call
        getter = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if getter is not None:
            _raw_stream = lambda: getter(torch._C._cuda_getDevice())
        else:
            _raw_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _raw_stream()


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


# ------------------------------------------------------------- quantisers --
def dg_quant_act_1x128(x, q=None, sfa=None, stream=None):
    """Per-token 1x128 quantiser.  x: CUDA fp32 or bf16 [M, K].
    Returns (q uint8 [M, K], sfa fp32 [K/128, round_up(M, 4)])."""
    import torch
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sfa is None:
        sfa = torch.zeros((K // QBLOCK, round_up(M, 4)), dtype=torch.float32, device=x.device)
    dt = {torch.float32: DG_DTYPE_F32, torch.bfloat16: DG_DTYPE_BF16}.get(x.dtype)
    if dt is None:
        raise TypeError(f"unsupported activation dtype {x.dtype}")
    assert x.is_contiguous() and q.is_contiguous() and sfa.is_contiguous()
    _check("dg_quant_act_1x128", load().dg_quant_act_1x128(_ptr(x), dt, _ptr(q), _ptr(sfa), M, K, _stream(stream)))
    return q, sfa


def dg_quant_weight_128x128(w, q=None, sfb=None, stream=None):
    """Per-block 128x128 quantiser.  w: CUDA fp32 [N, K] or [G, N, K].
    Returns (q uint8 like w, sfb fp32 [(G,) ceil(N/128), K/128])."""
    import torch
    squeeze = w.dim() == 2
    w3 = w.unsqueeze(0) if squeeze else w
    G, N, K = w3.shape
    if q is None:
        q = torch.empty(w3.shape, dtype=torch.uint8, device=w.device)
    if sfb is None:
        sfb = torch.empty((G, (N + QBLOCK - 1) // QBLOCK, K // QBLOCK), dtype=torch.float32, device=w.device)
    assert w3.is_contiguous() and w3.dtype == torch.float32
    _check("dg_quant_weight_128x128",
           load().dg_quant_weight_128x128(_ptr(w3), _ptr(q), _ptr(sfb), G, N, K, _stream(stream)))
    return (q[0], sfb[0]) if squeeze else (q, sfb)


# ------------------------------------------------------------------ GEMMs --
def dg_fp8_gemm_nt(a, sfa, b, sfb, d=None, stream=None):
    """Dense D = A . B^T (bf16 [M, N])."""
    import torch
    M, K = a.shape
    N = b.shape[0]
    if d is None:
        d = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _check("dg_fp8_gemm_nt", load().dg_fp8_gemm_nt(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), M, N, K,
                                                   _stream(stream)))
    return d


def dg_fp8_grouped_contiguous(a, sfa, b, sfb, m_indices, d=None, stream=None):
    """Contiguous MoE layout: a [sum_M, K], b [G, N, K], m_indices int32 [sum_M]."""
    import torch
    sum_M, K = a.shape
    G, N, _ = b.shape
    if d is None:
        d = torch.empty((sum_M, N), dtype=torch.bfloat16, device=a.device)
    _check("dg_fp8_grouped_contiguous",
           load().dg_fp8_grouped_contiguous(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(m_indices),
                                            sum_M, N, K, G, _stream(stream)))
    return d


def dg_fp8_grouped_masked(a, sfa, b, sfb, masked_m, d=None, expected_m: int = 0, stream=None):
    """Masked MoE layout: a [G, max_m, K], b [G, N, K], masked_m int32 [G] on
    the device; rows >= masked_m[g] of d are left untouched."""
    import torch
    G, max_m, K = a.shape
    N = b.shape[1]
    if d is None:
        d = torch.empty((G, max_m, N), dtype=torch.bfloat16, device=a.device)
    _check("dg_fp8_grouped_masked",
           load().dg_fp8_grouped_masked(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(masked_m), G, max_m,
                                        N, K, expected_m, _stream(stream)))
    return d


# --------------------------------------------- GEMMs, re-quantised output --
def _qout(shape, rows_ld: int, groups_shape, device, q, sfo):
    import torch
    if q is None:
        q = torch.empty(shape, dtype=torch.uint8, device=device)
    if sfo is None:
        sfo = torch.zeros((*groups_shape, rows_ld), dtype=torch.float32, device=device)
    assert q.is_contiguous() and sfo.is_contiguous()
    return q, sfo


def dg_fp8_gemm_nt_q(a, sfa, b, sfb, q=None, sfo=None, stream=None):
    """Dense D = A . B^T re-quantised: returns (q uint8 [M, N],
    sfo fp32 [N/128, round_up(M, 4)])."""
    M, K = a.shape
    N = b.shape[0]
    q, sfo = _qout((M, N), round_up(M, 4), (N // QBLOCK,), a.device, q, sfo)
    _check("dg_fp8_gemm_nt_q", load().dg_fp8_gemm_nt_q(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(q), _ptr(sfo),
                                                       M, N, K, _stream(stream)))
    return q, sfo


def dg_fp8_grouped_contiguous_q(a, sfa, b, sfb, m_indices, q=None, sfo=None, stream=None):
    """Contiguous MoE layout, re-quantised: returns (q uint8 [sum_M, N],
    sfo fp32 [N/128, sum_M]); rows with index -1 are left untouched."""
    sum_M, K = a.shape
    G, N, _ = b.shape
    q, sfo = _qout((sum_M, N), sum_M, (N // QBLOCK,), a.device, q, sfo)
    _check("dg_fp8_grouped_contiguous_q",
           load().dg_fp8_grouped_contiguous_q(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(q), _ptr(sfo),
                                              _ptr(m_indices), sum_M, N, K, G, _stream(stream)))
    return q, sfo


def dg_fp8_grouped_masked_q(a, sfa, b, sfb, masked_m, q=None, sfo=None, expected_m: int = 0, stream=None):
    """Masked MoE layout, re-quantised: returns (q uint8 [G, max_m, N],
    sfo fp32 [G, N/128, round_up(max_m, 4)]); rows >= masked_m[g] are left
    untouched."""
    G, max_m, K = a.shape
    N = b.shape[1]
    q, sfo = _qout((G, max_m, N), round_up(max_m, 4), (G, N // QBLOCK), a.device, q, sfo)
    _check("dg_fp8_grouped_masked_q",
           load().dg_fp8_grouped_masked_q(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(q), _ptr(sfo),
                                          _ptr(masked_m), G, max_m, N, K, expected_m, _stream(stream)))
    return q, sfo


def dg_query_plan(layout: int, M: int, N: int, K: int, G: int = 1, num_sms: int = 0) -> dict:
    """Tile plan for a problem (host-only when num_sms > 0)."""
    out = dg_plan_t()
    _check("dg_query_plan", load().dg_query_plan(layout, M, N, K, G, num_sms, ctypes.byref(out)))
    return {f: getattr(out, f) for f, _ in dg_plan_t._fields_}


def dg_read_device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device status word."""
    flags = ctypes.c_int(0)
    st = load().dg_read_device_status(ctypes.byref(flags), _stream(stream))
    if st not in (DG_OK, DG_ERR_DEVICE_TIMEOUT):
        _check("dg_read_device_status", st)
    return flags.value

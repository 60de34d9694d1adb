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
    "dg_selftest_wait_timeout",
    "dg_bf16_gemm_nt",
    "dg_quant_mx_1x32",
    "dg_mx_gemm_nt",
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
        "dg_query_plan": [I, I, I, I, I, I, I, ctypes.POINTER(dg_plan_t)],
        "dg_read_device_status": [ctypes.POINTER(ctypes.c_int), P],
        "dg_selftest_wait_timeout": [ctypes.c_longlong, P],
        "dg_bf16_gemm_nt": [P, P, P, I, I, I, P],
        "dg_quant_mx_1x32": [P, P, P, I, I, P],
        "dg_mx_gemm_nt": [P, P, P, P, P, I, I, I, P],
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


# Argument checks.  The C entry points take bare pointers, so a tensor of the
# wrong size, type, layout or device would make the kernels read or write
# outside it; every binding below checks each tensor against the sizes taken
# from its first operand before calling the library.
_dt = {}


def _dtypes():
    if not _dt:
        import torch
        _dt.update(fp8=(torch.uint8, torch.float8_e4m3fn), f32=(torch.float32,), bf16=(torch.bfloat16,),
                   i32=(torch.int32,), act=(torch.float32, torch.bfloat16))
    return _dt


def _dims(t, name: str, ndim: int):
    try:
        shape = t.shape
    except AttributeError:
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}") from None
    if len(shape) != ndim:
        raise ValueError(f"{name}: expected {ndim} dimensions, got shape {tuple(shape)}")
    return shape


def _want(t, name: str, shape: tuple, dtypes: tuple) -> None:
    try:
        ok = t.shape == shape and t.dtype in dtypes and t.is_contiguous()
    except AttributeError:
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}") from None
    if not ok:
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
        if t.dtype not in dtypes:
            raise TypeError(f"{name}: expected dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
        raise ValueError(f"{name}: must be contiguous")


def _on_device(*named) -> None:
    """Every tensor on the current CUDA device (where the library launches)."""
    dev = None
    for name, t in named:
        idx = t.get_device()
        if idx < 0:
            raise ValueError(f"{name}: a CUDA tensor is required (there is no CPU path), got one on {t.device}")
        if dev is None:
            import torch
            dev = torch._C._cuda_getDevice()
        if idx != dev:
            raise ValueError(f"{name}: on cuda:{idx}, but the current device is cuda:{dev}")


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


# ------------------------------------------------------------- quantisers --
def dg_quant_act_1x128(x, q=None, sfa=None, stream=None):
    """Per-token 1x128 quantiser.  x: CUDA fp32 or bf16 [M, K].
    Returns (q uint8 [M, K], sfa fp32 [K/128, round_up(M, 4)])."""
    import torch
    T = _dtypes()
    M, K = _dims(x, "x", 2)
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sfa is None:
        sfa = torch.zeros((K // QBLOCK, round_up(M, 4)), dtype=torch.float32, device=x.device)
    # one expression on the common path; the per-tensor checks name the culprit
    try:
        ok = (x.dtype in T["act"] and q.dtype in T["fp8"] and sfa.dtype in T["f32"] and q.shape == (M, K)
              and sfa.shape == (K // QBLOCK, round_up(M, 4)) and x.is_contiguous() and q.is_contiguous()
              and sfa.is_contiguous())
    except AttributeError:
        ok = False
    if not ok:
        _want(x, "x", (M, K), T["act"])
        _want(q, "q", (M, K), T["fp8"])
        _want(sfa, "sfa", (K // QBLOCK, round_up(M, 4)), T["f32"])
    _on_device(("x", x), ("q", q), ("sfa", sfa))
    dt = DG_DTYPE_F32 if x.dtype == torch.float32 else DG_DTYPE_BF16
    _check("dg_quant_act_1x128", load().dg_quant_act_1x128(_ptr(x), dt, _ptr(q), _ptr(sfa), M, K, _stream(stream)))
    return q, sfa


def dg_quant_weight_128x128(w, q=None, sfb=None, stream=None):
    """Per-block 128x128 quantiser.  w: CUDA fp32 [N, K] or [G, N, K].
    Returns (q uint8 like w, sfb fp32 [(G,) ceil(N/128), K/128])."""
    import torch
    T = _dtypes()
    if not isinstance(w, torch.Tensor) or w.dim() not in (2, 3):
        raise ValueError("w: expected a [N, K] or [G, N, K] torch.Tensor")
    squeeze = w.dim() == 2
    w3 = w.unsqueeze(0) if squeeze else w
    G, N, K = w3.shape
    _want(w3, "w", (G, N, K), T["f32"])
    if q is None:
        q = torch.empty(w3.shape, dtype=torch.uint8, device=w.device)
    elif squeeze:
        q = q.unsqueeze(0)
    if sfb is None:
        sfb = torch.empty((G, (N + QBLOCK - 1) // QBLOCK, K // QBLOCK), dtype=torch.float32, device=w.device)
    elif squeeze:
        sfb = sfb.unsqueeze(0)
    _want(q, "q", (G, N, K), T["fp8"])
    _want(sfb, "sfb", (G, (N + QBLOCK - 1) // QBLOCK, K // QBLOCK), T["f32"])
    _on_device(("w", w3), ("q", q), ("sfb", sfb))
    _check("dg_quant_weight_128x128",
           load().dg_quant_weight_128x128(_ptr(w3), _ptr(q), _ptr(sfb), G, N, K, _stream(stream)))
    return (q[0], sfb[0]) if squeeze else (q, sfb)


# ------------------------------------------------------------------ GEMMs --
def _grouped_operands(T, a, sfa, b, sfb, sfa_shape, G, N, K):
    _want(a, "a", tuple(a.shape), T["fp8"])
    _want(sfa, "sfa", sfa_shape, T["f32"])
    _want(b, "b", (G, N, K), T["fp8"])
    _want(sfb, "sfb", (G, -(-N // QBLOCK), K // QBLOCK), T["f32"])


def dg_fp8_gemm_nt(a, sfa, b, sfb, d=None, stream=None):
    """Dense D = A . B^T (bf16 [M, N])."""
    import torch
    T = _dtypes()
    M, K = _dims(a, "a", 2)
    N = _dims(b, "b", 2)[0]
    if d is None:
        d = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    fp8, f32 = T["fp8"], T["f32"]
    try:
        ok = (a.dtype in fp8 and b.dtype in fp8 and sfa.dtype in f32 and sfb.dtype in f32
              and d.dtype in T["bf16"] and b.shape == (N, K) and sfa.shape == (K // QBLOCK, round_up(M, 4))
              and sfb.shape == (-(-N // QBLOCK), K // QBLOCK) and d.shape == (M, N) and a.is_contiguous()
              and b.is_contiguous() and sfa.is_contiguous() and sfb.is_contiguous() and d.is_contiguous())
    except AttributeError:
        ok = False
    if not ok:
        _want(a, "a", (M, K), fp8)
        _want(sfa, "sfa", (K // QBLOCK, round_up(M, 4)), f32)
        _want(b, "b", (N, K), fp8)
        _want(sfb, "sfb", (-(-N // QBLOCK), K // QBLOCK), f32)
        _want(d, "d", (M, N), T["bf16"])
    _on_device(("a", a), ("sfa", sfa), ("b", b), ("sfb", sfb), ("d", d))
    _check("dg_fp8_gemm_nt", load().dg_fp8_gemm_nt(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), M, N, K,
                                                   _stream(stream)))
    return d


def dg_fp8_grouped_contiguous(a, sfa, b, sfb, m_indices, d=None, stream=None):
    """Contiguous MoE layout: a [sum_M, K], b [G, N, K], m_indices int32 [sum_M]."""
    import torch
    T = _dtypes()
    sum_M, K = _dims(a, "a", 2)
    G, N, _ = _dims(b, "b", 3)
    _grouped_operands(T, a, sfa, b, sfb, (K // QBLOCK, round_up(sum_M, 4)), G, N, K)
    _want(m_indices, "m_indices", (sum_M,), T["i32"])
    if d is None:
        d = torch.empty((sum_M, N), dtype=torch.bfloat16, device=a.device)
    _want(d, "d", (sum_M, N), T["bf16"])
    _on_device(("a", a), ("sfa", sfa), ("b", b), ("sfb", sfb), ("m_indices", m_indices), ("d", d))
    _check("dg_fp8_grouped_contiguous",
           load().dg_fp8_grouped_contiguous(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(m_indices),
                                            sum_M, N, K, G, _stream(stream)))
    return d


def dg_fp8_grouped_masked(a, sfa, b, sfb, masked_m, d=None, expected_m: int = 0, stream=None):
    """Masked MoE layout: a [G, max_m, K], b [G, N, K], masked_m int32 [G] on
    the device; rows >= masked_m[g] of d are left untouched."""
    import torch
    T = _dtypes()
    G, max_m, K = _dims(a, "a", 3)
    N = _dims(b, "b", 3)[1]
    _grouped_operands(T, a, sfa, b, sfb, (G, K // QBLOCK, round_up(max_m, 4)), G, N, K)
    _want(masked_m, "masked_m", (G,), T["i32"])
    if d is None:
        d = torch.empty((G, max_m, N), dtype=torch.bfloat16, device=a.device)
    _want(d, "d", (G, max_m, N), T["bf16"])
    _on_device(("a", a), ("sfa", sfa), ("b", b), ("sfb", sfb), ("masked_m", masked_m), ("d", d))
    _check("dg_fp8_grouped_masked",
           load().dg_fp8_grouped_masked(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(masked_m), G, max_m,
                                        N, K, expected_m, _stream(stream)))
    return d


# --------------------------------------------- GEMMs, re-quantised output --
def _qout(shape, rows_ld: int, groups_shape, device, q, sfo):
    import torch
    T = _dtypes()
    if q is None:
        q = torch.empty(shape, dtype=torch.uint8, device=device)
    if sfo is None:
        sfo = torch.zeros((*groups_shape, rows_ld), dtype=torch.float32, device=device)
    _want(q, "q", tuple(shape), T["fp8"])
    _want(sfo, "sfo", (*groups_shape, rows_ld), T["f32"])
    return q, sfo


def dg_fp8_gemm_nt_q(a, sfa, b, sfb, q=None, sfo=None, stream=None):
    """Dense D = A . B^T re-quantised: returns (q uint8 [M, N],
    sfo fp32 [N/128, round_up(M, 4)])."""
    T = _dtypes()
    M, K = _dims(a, "a", 2)
    N = _dims(b, "b", 2)[0]
    _want(a, "a", (M, K), T["fp8"])
    _want(sfa, "sfa", (K // QBLOCK, round_up(M, 4)), T["f32"])
    _want(b, "b", (N, K), T["fp8"])
    _want(sfb, "sfb", (-(-N // QBLOCK), K // QBLOCK), T["f32"])
    q, sfo = _qout((M, N), round_up(M, 4), (N // QBLOCK,), a.device, q, sfo)
    _on_device(("a", a), ("sfa", sfa), ("b", b), ("sfb", sfb), ("q", q), ("sfo", sfo))
    _check("dg_fp8_gemm_nt_q", load().dg_fp8_gemm_nt_q(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(q), _ptr(sfo),
                                                       M, N, K, _stream(stream)))
    return q, sfo


def dg_fp8_grouped_contiguous_q(a, sfa, b, sfb, m_indices, q=None, sfo=None, stream=None):
    """Contiguous MoE layout, re-quantised: returns (q uint8 [sum_M, N],
    sfo fp32 [N/128, sum_M]); rows with index -1 are left untouched."""
    T = _dtypes()
    sum_M, K = _dims(a, "a", 2)
    G, N, _ = _dims(b, "b", 3)
    _grouped_operands(T, a, sfa, b, sfb, (K // QBLOCK, round_up(sum_M, 4)), G, N, K)
    _want(m_indices, "m_indices", (sum_M,), T["i32"])
    q, sfo = _qout((sum_M, N), sum_M, (N // QBLOCK,), a.device, q, sfo)
    _on_device(("a", a), ("sfa", sfa), ("b", b), ("sfb", sfb), ("m_indices", m_indices), ("q", q), ("sfo", sfo))
    _check("dg_fp8_grouped_contiguous_q",
           load().dg_fp8_grouped_contiguous_q(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(q), _ptr(sfo),
                                              _ptr(m_indices), sum_M, N, K, G, _stream(stream)))
    return q, sfo


def dg_fp8_grouped_masked_q(a, sfa, b, sfb, masked_m, q=None, sfo=None, expected_m: int = 0, stream=None):
    """Masked MoE layout, re-quantised: returns (q uint8 [G, max_m, N],
    sfo fp32 [G, N/128, round_up(max_m, 4)]); rows >= masked_m[g] are left
    untouched."""
    T = _dtypes()
    G, max_m, K = _dims(a, "a", 3)
    N = _dims(b, "b", 3)[1]
    _grouped_operands(T, a, sfa, b, sfb, (G, K // QBLOCK, round_up(max_m, 4)), G, N, K)
    _want(masked_m, "masked_m", (G,), T["i32"])
    q, sfo = _qout((G, max_m, N), round_up(max_m, 4), (G, N // QBLOCK), a.device, q, sfo)
    _on_device(("a", a), ("sfa", sfa), ("b", b), ("sfb", sfb), ("masked_m", masked_m), ("q", q), ("sfo", sfo))
    _check("dg_fp8_grouped_masked_q",
           load().dg_fp8_grouped_masked_q(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(q), _ptr(sfo),
                                          _ptr(masked_m), G, max_m, N, K, expected_m, _stream(stream)))
    return q, sfo


def dg_query_plan(layout: int, M: int, N: int, K: int, G: int = 1, num_sms: int = 0, expected_m: int = 0) -> dict:
    """Tile plan for a problem (host-only when num_sms > 0); expected_m is the
    masked layout's hint."""
    out = dg_plan_t()
    _check("dg_query_plan", load().dg_query_plan(layout, M, N, K, G, expected_m, num_sms, ctypes.byref(out)))
    return {f: getattr(out, f) for f, _ in dg_plan_t._fields_}


def dg_read_device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device status word."""
    flags = ctypes.c_int(0)
    st = load().dg_read_device_status(ctypes.byref(flags), _stream(stream))
    if st not in (DG_OK, DG_ERR_DEVICE_TIMEOUT):
        _check("dg_read_device_status", st)
    return flags.value


def dg_selftest_wait_timeout(limit_cycles: int = 2_000_000, stream=None) -> None:
    """Enqueue the bounded-wait diagnostic: a kernel waits on a barrier that
    nothing arrives on and gives up after `limit_cycles` SM cycles, setting
    DG_DEVFLAG_TIMEOUT (read it with dg_read_device_status)."""
    _check("dg_selftest_wait_timeout", load().dg_selftest_wait_timeout(int(limit_cycles), _stream(stream)))


# ------------------------------------------------------ BF16 and MX GEMMs --
def dg_bf16_gemm_nt(a, b, d=None, stream=None):
    """D = A . B^T on bf16 operands: a bf16 [M, K], b bf16 [N, K] -> bf16 [M, N]."""
    import torch
    T = _dtypes()
    M, K = _dims(a, "a", 2)
    N = _dims(b, "b", 2)[0]
    if d is None:
        d = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _want(a, "a", (M, K), T["bf16"])
    _want(b, "b", (N, K), T["bf16"])
    _want(d, "d", (M, N), T["bf16"])
    _on_device(("a", a), ("b", b), ("d", d))
    _check("dg_bf16_gemm_nt", load().dg_bf16_gemm_nt(_ptr(a), _ptr(b), _ptr(d), M, N, K, _stream(stream)))
    return d


def dg_quant_mx_1x32(x, q=None, sx=None, stream=None):
    """MX quantiser: x fp32 [R, K] -> (q uint8 E4M3 [R, K], sx uint8 E8M0 [K/128, R, 4]).

    sx is chunk-major: sx[g, r, j] is the scale code of row r's 32-wide block
    4 g + j (the row-major [R, K/32] codes, permuted)."""
    import torch
    T = _dtypes()
    R, K = _dims(x, "x", 2)
    if q is None:
        q = torch.empty((R, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((K // 128, R, 4), dtype=torch.uint8, device=x.device)
    _want(x, "x", (R, K), T["f32"])
    _want(q, "q", (R, K), T["fp8"])
    _want(sx, "sx", (K // 128, R, 4), (torch.uint8,))
    _on_device(("x", x), ("q", q), ("sx", sx))
    _check("dg_quant_mx_1x32", load().dg_quant_mx_1x32(_ptr(x), _ptr(q), _ptr(sx), R, K, _stream(stream)))
    return q, sx


def dg_mx_gemm_nt(a, sa, b, sb, d=None, stream=None):
    """MX GEMM: a E4M3 [M, K], sa E8M0 [K/128, M, 4], b [N, K], sb [K/128, N, 4] -> bf16 [M, N]
    (scales in the chunk-major layout dg_quant_mx_1x32 writes)."""
    import torch
    T = _dtypes()
    M, K = _dims(a, "a", 2)
    N = _dims(b, "b", 2)[0]
    if d is None:
        d = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _want(a, "a", (M, K), T["fp8"])
    _want(sa, "sa", (K // 128, M, 4), (torch.uint8,))
    _want(b, "b", (N, K), T["fp8"])
    _want(sb, "sb", (K // 128, N, 4), (torch.uint8,))
    _want(d, "d", (M, N), T["bf16"])
    _on_device(("a", a), ("sa", sa), ("b", b), ("sb", sb), ("d", d))
    _check("dg_mx_gemm_nt", load().dg_mx_gemm_nt(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(d), M, N, K,
                                                 _stream(stream)))
    return d

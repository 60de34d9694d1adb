"""CPU oracle for the FP8 fine-grained-scaled GEMM (test infrastructure).

TEST INFRASTRUCTURE ONLY: the plain C definition in ``oracle.c`` wrapped for
numpy.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares nothing with the CUDA library
under ``moe_grouped_gemm_x128_gb300/``; neither imports the other.

Every function follows the pages "DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库"
(功能特色/细粒度缩放功能, 技术细节/两级累加技术, 功能特色/支持多种数据排列方式) and
the 2kiu.com DeepGEMM tutorial (4.4 精度控制与数值稳定性); the BF16 GEMM and the MX
functions follow the same tutorial (1, 2.2 and 7) and, for what MX means, the
OCP Microscaling Formats (MX) v1.0 specification.  The readings taken where the
pages are silent are stated in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
QBLOCK = 128

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (IEEE: no fast-math,
    no implicit FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode_bruteforce.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode_bruteforce.restype = ctypes.c_uint8
    lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_quant_act_1x128.argtypes = [P, I, I, P, P, I]
    lib.oracle_quant_act_1x128.restype = None
    lib.oracle_quant_act_1x128_bf16.argtypes = [P, I, I, P, P, I]
    lib.oracle_quant_act_1x128_bf16.restype = None
    lib.oracle_quant_weight_128x128.argtypes = [P, I, I, P, P]
    lib.oracle_quant_weight_128x128.restype = None
    lib.oracle_gemm_nt.argtypes = [P, P, I, P, P, P, P, I, I, I, P, I]
    lib.oracle_gemm_nt.restype = None
    lib.oracle_grouped_contiguous.argtypes = [P, P, I, P, P, P, P, I, I, I, I, P, I]
    lib.oracle_grouped_contiguous.restype = None
    lib.oracle_grouped_masked.argtypes = [P, P, I, P, P, P, P, I, I, I, I]
    lib.oracle_grouped_masked.restype = None
    lib.oracle_gemm_bf16_nt.argtypes = [P, P, P, I, I, I, P, I]
    lib.oracle_gemm_bf16_nt.restype = None
    lib.oracle_ue8m0_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_ue8m0_decode.restype = ctypes.c_double
    lib.oracle_quant_mx_1x32.argtypes = [P, I, I, P, P]
    lib.oracle_quant_mx_1x32.restype = None
    lib.oracle_gemm_mx_nt.argtypes = [P, P, P, P, P, I, I, I, P, I]
    lib.oracle_gemm_mx_nt.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def num_threads() -> int:
    return _load().oracle_num_threads()


# ------------------------------------------------------------------ scalars --
def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(code)


def e4m3_encode(x: float) -> int:
    return _load().oracle_e4m3_encode(x)


def e4m3_encode_bruteforce(x: float) -> int:
    return _load().oracle_e4m3_encode_bruteforce(x)


def bf16_rne(x: float) -> int:
    return _load().oracle_bf16_rne(x)


def e4m3_decode_table() -> np.ndarray:
    """float64[256] from the closed form (NaN at 0x7F and 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


# --------------------------------------------------------------- quantisers --
def quant_act_1x128(x: np.ndarray):
    """Per-token 1x128 quantiser.  x: fp32 [M,K] (or bf16 bits as uint16).
    Returns (q uint8 [M,K], sfa fp32 [K/128, round_up(M,4)]).  Padding
    columns of sfa (m >= M) are zero."""
    M, K = x.shape
    assert K % QBLOCK == 0
    ld = round_up(M, 4)
    q = np.empty((M, K), dtype=np.uint8)
    sfa = np.zeros((K // QBLOCK, ld), dtype=np.float32)
    if x.dtype == np.float32:
        x = np.ascontiguousarray(x)
        _load().oracle_quant_act_1x128(_ptr(x), M, K, _ptr(q), _ptr(sfa), ld)
    elif x.dtype == np.uint16:
        x = np.ascontiguousarray(x)
        _load().oracle_quant_act_1x128_bf16(_ptr(x), M, K, _ptr(q), _ptr(sfa), ld)
    else:
        raise TypeError(f"unsupported activation dtype {x.dtype}")
    return q, sfa


def quant_weight_128x128(w: np.ndarray):
    """Per-block 128x128 quantiser.  w: fp32 [N,K] or [G,N,K].
    Returns (q uint8, sfb fp32 [(G,) ceil(N/128), K/128])."""
    if w.ndim == 3:
        qs, ss = zip(*(quant_weight_128x128(w[g]) for g in range(w.shape[0])))
        return np.stack(qs), np.stack(ss)
    N, K = w.shape
    assert K % QBLOCK == 0 and w.dtype == np.float32
    w = np.ascontiguousarray(w)
    q = np.empty((N, K), dtype=np.uint8)
    sfb = np.empty(((N + QBLOCK - 1) // QBLOCK, K // QBLOCK), dtype=np.float32)
    _load().oracle_quant_weight_128x128(_ptr(w), N, K, _ptr(q), _ptr(sfb))
    return q, sfb


# ------------------------------------------------------------------- GEMMs --
def gemm_nt(a, sfa, b, sfb, rows=None, d=None, want_acc=False):
    """Dense D = A.B^T with fine-grained scales and per-128-K promotion.
    a uint8 [M,K]; sfa fp32 [K/128, ld>=M]; b uint8 [N,K]; sfb fp32
    [ceil(N/128), K/128].  Returns D as bf16 bits (uint16 [M,N]); with
    ``rows`` only those rows are computed (others keep ``d``'s contents, zero
    by default).  With want_acc also returns the fp32 accumulator."""
    M, K = a.shape
    N = b.shape[0]
    if d is None:
        d = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.float32) if want_acc else None
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    _load().oracle_gemm_nt(_ptr(np.ascontiguousarray(a)), _ptr(np.ascontiguousarray(sfa)),
                           sfa.shape[1], _ptr(np.ascontiguousarray(b)),
                           _ptr(np.ascontiguousarray(sfb)), _ptr(d), _ptr(acc), M, N, K,
                           _ptr(r), 0 if r is None else len(r))
    return (d, acc) if want_acc else d


def grouped_contiguous(a, sfa, b, sfb, m_indices, rows=None, d=None):
    """Contiguous MoE layout.  a uint8 [sum_M,K]; sfa [K/128, ld]; b uint8
    [G,N,K]; sfb [G, ceil(N/128), K/128]; m_indices int32 [sum_M] (-1 =
    padding).  Rows with a negative index keep ``d``'s contents."""
    sum_M, K = a.shape
    G, N, _ = b.shape
    if d is None:
        d = np.zeros((sum_M, N), dtype=np.uint16)
    mi = np.ascontiguousarray(m_indices, dtype=np.int32)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    _load().oracle_grouped_contiguous(
        _ptr(np.ascontiguousarray(a)), _ptr(np.ascontiguousarray(sfa)), sfa.shape[1],
        _ptr(np.ascontiguousarray(b)), _ptr(np.ascontiguousarray(sfb)), _ptr(d), _ptr(mi),
        sum_M, N, K, G, _ptr(r), 0 if r is None else len(r))
    return d


def grouped_masked(a, sfa, b, sfb, masked_m, d=None):
    """Masked MoE layout.  a uint8 [G,max_m,K]; sfa [G, K/128, ld]; b uint8
    [G,N,K]; sfb [G, ceil(N/128), K/128]; masked_m int32 [G].  Rows at or
    beyond masked_m[g] keep ``d``'s contents."""
    G, max_m, K = a.shape
    N = b.shape[1]
    if d is None:
        d = np.zeros((G, max_m, N), dtype=np.uint16)
    mm = np.ascontiguousarray(masked_m, dtype=np.int32)
    _load().oracle_grouped_masked(
        _ptr(np.ascontiguousarray(a)), _ptr(np.ascontiguousarray(sfa)), sfa.shape[2],
        _ptr(np.ascontiguousarray(b)), _ptr(np.ascontiguousarray(sfb)), _ptr(d), _ptr(mm),
        G, max_m, N, K)
    return d


# ------------------------------------------- GEMMs with re-quantised output --
# The fused output (the next step after the path: the pages' call to fuse the
# operations around a GEMM so that its result makes no extra round trip,
# 2kiu.com tutorial 7) is the GEMM's bf16 output re-quantised as the next
# GEMM's activation operand: E4M3 with one fp32 scale per 1x128 group of each
# output row.  It is the plain composition of two pinned functions,
# quant_act_1x128(bf16 D), so that it equals the unfused two-call pipeline.
def _requant_rows(d_bits: np.ndarray, rows: np.ndarray, q: np.ndarray, sfo: np.ndarray) -> None:
    """Quantise the listed rows of bf16 D (uint16 [M,N]) into q / sfo in place."""
    if len(rows) == 0:
        return
    qr, sr = quant_act_1x128(np.ascontiguousarray(d_bits[rows]))
    q[rows] = qr
    sfo[:, rows] = sr[:, :len(rows)]


def gemm_nt_quant(a, sfa, b, sfb, q=None, sfo=None):
    """Dense D = A.B^T as gemm_nt, re-quantised: returns (q uint8 [M,N],
    sfo fp32 [N/128, round_up(M,4)]).  N must be a multiple of 128."""
    M = a.shape[0]
    N = b.shape[0]
    assert N % QBLOCK == 0
    q = np.zeros((M, N), np.uint8) if q is None else q
    sfo = np.zeros((N // QBLOCK, round_up(M, 4)), np.float32) if sfo is None else sfo
    _requant_rows(gemm_nt(a, sfa, b, sfb), np.arange(M), q, sfo)
    return q, sfo


def grouped_contiguous_quant(a, sfa, b, sfb, m_indices, q=None, sfo=None):
    """Contiguous layout, re-quantised.  Rows with a negative expert index keep
    q's and sfo's contents."""
    sum_M = a.shape[0]
    N = b.shape[1]
    assert N % QBLOCK == 0
    q = np.zeros((sum_M, N), np.uint8) if q is None else q
    sfo = np.zeros((N // QBLOCK, round_up(sum_M, 4)), np.float32) if sfo is None else sfo
    d = grouped_contiguous(a, sfa, b, sfb, m_indices)
    _requant_rows(d, np.flatnonzero(np.asarray(m_indices) >= 0), q, sfo)
    return q, sfo


def grouped_masked_quant(a, sfa, b, sfb, masked_m, q=None, sfo=None):
    """Masked layout, re-quantised: q uint8 [G,max_m,N], sfo fp32
    [G, N/128, round_up(max_m,4)].  Rows at or beyond masked_m[g] keep q's and
    sfo's contents."""
    G, max_m, _ = a.shape
    N = b.shape[1]
    assert N % QBLOCK == 0
    q = np.zeros((G, max_m, N), np.uint8) if q is None else q
    sfo = np.zeros((G, N // QBLOCK, round_up(max_m, 4)), np.float32) if sfo is None else sfo
    d = grouped_masked(a, sfa, b, sfb, masked_m)
    for g in range(G):
        mm = int(min(max(int(masked_m[g]), 0), max_m))
        _requant_rows(d[g], np.arange(mm), q[g], sfo[g])
    return q, sfo


def bf16_bits_to_f32(d: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (d.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ BF16 GEMM ----
# A plain GEMM on bf16 operands, the second low-precision format the pages
# name beside FP8 (2kiu.com tutorial 1 and 2.2): the exact sum of products,
# rounded once to fp32 and then to bf16 (round to nearest even).
def gemm_bf16_nt(a_bits, b_bits, rows=None, d=None):
    """D = A.B^T on bf16 operands.  a_bits uint16 [M,K], b_bits uint16 [N,K]
    (bf16 bit patterns).  Returns bf16 bits uint16 [M,N]; with ``rows`` only
    those rows are computed (others keep ``d``'s contents, zero by default)."""
    M, K = a_bits.shape
    N = b_bits.shape[0]
    assert a_bits.dtype == np.uint16 and b_bits.dtype == np.uint16 and b_bits.shape[1] == K
    if d is None:
        d = np.zeros((M, N), dtype=np.uint16)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    _load().oracle_gemm_bf16_nt(_ptr(np.ascontiguousarray(a_bits)), _ptr(np.ascontiguousarray(b_bits)), _ptr(d),
                                M, N, K, _ptr(r), 0 if r is None else len(r))
    return d


# ------------------------------------------------------ MX (microscaling) --
# The MX formats the pages point to for finer scale granularity (2kiu.com
# tutorial 7), as the OCP Microscaling Formats (MX) v1.0 specification
# defines them: 32 consecutive values along K share one E8M0 scale 2^e.
MX_BLOCK = 32


def ue8m0_decode(code: int) -> float:
    return _load().oracle_ue8m0_decode(code)


def quant_mx_1x32(x: np.ndarray):
    """MX (E4M3 elements, E8M0 scales) quantiser of the rows of x fp32 [R,K].
    Returns (q uint8 [R,K], sx uint8 [R,K/32])."""
    R_, K = x.shape
    assert K % MX_BLOCK == 0 and x.dtype == np.float32
    x = np.ascontiguousarray(x)
    q = np.empty((R_, K), dtype=np.uint8)
    sx = np.empty((R_, K // MX_BLOCK), dtype=np.uint8)
    _load().oracle_quant_mx_1x32(_ptr(x), R_, K, _ptr(q), _ptr(sx))
    return q, sx


def gemm_mx_nt(a, sa, b, sb, rows=None, d=None):
    """MX GEMM D = A.B^T: a uint8 E4M3 [M,K], sa uint8 E8M0 [M,K/32], b [N,K],
    sb [N,K/32].  Returns bf16 bits uint16 [M,N] (``rows`` as gemm_bf16_nt)."""
    M, K = a.shape
    N = b.shape[0]
    assert K % MX_BLOCK == 0 and sa.shape == (M, K // MX_BLOCK) and sb.shape == (N, K // MX_BLOCK)
    if d is None:
        d = np.zeros((M, N), dtype=np.uint16)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    _load().oracle_gemm_mx_nt(_ptr(np.ascontiguousarray(a)), _ptr(np.ascontiguousarray(sa)),
                              _ptr(np.ascontiguousarray(b)), _ptr(np.ascontiguousarray(sb)), _ptr(d),
                              M, N, K, _ptr(r), 0 if r is None else len(r))
    return d

"""Shared helpers of the test suite (inputs, the tolerance rule, exact cases)."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as wl

QB = 128

# E4M3 codes of the small integers used by the exact-arithmetic cases
E4M3_OF_INT = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}


def int_codes(v: np.ndarray) -> np.ndarray:
    lut = np.zeros(5, dtype=np.uint8)
    for k, c in E4M3_OF_INT.items():
        lut[k + 2] = c
    return lut[v.astype(np.int64) + 2]


def exact_dense(M, N, K, seed):
    """E4M3 operands with values in {-2..2} and power-of-two scales 2^[-3,0]:
    every fp32 quantity of the path is exact, so the result is unique."""
    g = np.random.default_rng(seed)
    a = int_codes(wl.exact_operands(g, (M, K)))
    b = int_codes(wl.exact_operands(g, (N, K)))
    sfa = np.zeros((K // QB, oracle.round_up(M, 4)), dtype=np.float32)
    sfa[:, :M] = wl.exact_scales(g, (K // QB, M))
    sfb = wl.exact_scales(g, (-(-N // QB), K // QB))
    return a, sfa, b, sfb


def random_dense(M, N, K, seed, outliers=False):
    x, w = wl.dense_inputs(M, N, K, seed, outliers)
    a, sfa = oracle.quant_act_1x128(x)
    b, sfb = oracle.quant_weight_128x128(w)
    return a, sfa, b, sfb


def tolerance_check(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    """The stated bar for random inputs: ||gpu - ref||_F / ||ref||_F <= 1e-3 and
    per element |gpu - ref| <= 2^-7 |ref| + 1e-2 rms(ref).  `ref` is the
    oracle's bf16 output widened to fp32."""
    gpu = gpu.astype(np.float64)
    ref = ref.astype(np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    fro = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= 1e-3, f"{what}: relative Frobenius error {fro:.3e}"
    bad = np.abs(gpu - ref) > 2.0 ** -7 * np.abs(ref) + 1e-2 * rms
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the per-element bound"
    return fro


def bf16_bits_to_f32(d: np.ndarray) -> np.ndarray:
    return (d.astype(np.uint32) << 16).view(np.float32)


def mx_scales_chunk_major(s: np.ndarray) -> np.ndarray:
    """Row-major MX scale codes [R, K/32] in the library's chunk-major layout
    [K/128, R, 4] (a permutation: element [g, r, j] = s[r, 4 g + j])."""
    R, nb = s.shape
    return np.ascontiguousarray(s.reshape(R, nb // 4, 4).transpose(1, 0, 2))


def mx_scales_row_major(s: np.ndarray) -> np.ndarray:
    """The inverse of mx_scales_chunk_major: [K/128, R, 4] -> [R, K/32]."""
    G, R, _ = s.shape
    return np.ascontiguousarray(s.transpose(1, 0, 2).reshape(R, G * 4))

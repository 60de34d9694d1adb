"""Pins of the oracle's functions for the rows after the FP8 path: the BF16
GEMM and the MX (microscaling) quantiser and GEMM.

As for the FP8 functions, each is fixed by something other than itself:
closed forms, torch's float8_e4m3fn and bfloat16 conversions, numpy integer
and float64 matmul, and invariants, chosen so that a wrong exponent, a
transposed operand or a dropped block fails.  No GPU is needed."""
import math

import numpy as np
import torch

import oracle
from helpers import int_codes

MX = 32


def bf16_bits_of(x32: np.ndarray) -> np.ndarray:
    """torch's round-to-nearest-even fp32 -> bf16, as bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_bf16(g, shape, scale=1.0):
    return bf16_bits_of((g.standard_normal(shape) * scale).astype(np.float32))


# -------------------------------------------------------------- BF16 GEMM --
def test_bf16_gemm_integers_equal_int64_matmul():
    """Integer operands in [-8, 8]: every product and partial sum is exact, so
    D is the int64 matmul rounded to bf16 (an orientation or index mistake
    changes the non-square result)."""
    g = np.random.default_rng(1)
    for M, N, K in [(7, 5, 96), (33, 17, 1000), (1, 64, 4096)]:
        ai = g.integers(-8, 9, (M, K))
        bi = g.integers(-8, 9, (N, K))
        d = oracle.gemm_bf16_nt(bf16_bits_of(ai.astype(np.float32)), bf16_bits_of(bi.astype(np.float32)))
        ref = bf16_bits_of((ai @ bi.T).astype(np.float32))
        np.testing.assert_array_equal(d, ref)


def test_bf16_gemm_random_matches_float64_matmul():
    """Random bf16 operands: the result is the float64 matmul of the decoded
    values rounded to fp32 then bf16, up to the order of the double sums
    (which only matters on exact rounding ties)."""
    g = np.random.default_rng(2)
    M, N, K = 40, 56, 512
    a = random_bf16(g, (M, K))
    b = random_bf16(g, (N, K), scale=3.0)
    d = oracle.gemm_bf16_nt(a, b)
    ref = bf16_bits_of((bits_to_f64(a) @ bits_to_f64(b).T).astype(np.float32))
    same = d == ref
    assert same.mean() > 0.999
    ulp = np.abs(bits_to_f64(ref)) * 2.0 ** -7
    assert np.all(np.abs(bits_to_f64(d) - bits_to_f64(ref)) <= ulp + 1e-30)


def test_bf16_gemm_rows_subset_and_scaling():
    g = np.random.default_rng(3)
    a = random_bf16(g, (9, 128))
    b = random_bf16(g, (12, 128))
    full = oracle.gemm_bf16_nt(a, b)
    rows = np.array([0, 4, 8])
    part = oracle.gemm_bf16_nt(a, b, rows=rows, d=np.full((9, 12), 0x7FBF, np.uint16))
    np.testing.assert_array_equal(part[rows], full[rows])
    assert np.all(np.delete(part, rows, axis=0) == 0x7FBF)
    # scaling an operand by a power of two scales D exactly
    a2 = bf16_bits_of(bits_to_f64(a).astype(np.float32) * 4)
    np.testing.assert_array_equal(bits_to_f64(oracle.gemm_bf16_nt(a2, b)), 4 * bits_to_f64(full))


# -------------------------------------------------------------------- MX --
def test_ue8m0_decode_closed_form():
    assert oracle.ue8m0_decode(127) == 1.0
    assert oracle.ue8m0_decode(128) == 2.0
    assert oracle.ue8m0_decode(126) == 0.5
    assert oracle.ue8m0_decode(0) == 2.0 ** -127
    assert oracle.ue8m0_decode(254) == 2.0 ** 127
    assert math.isnan(oracle.ue8m0_decode(255))
    for c in range(255):
        assert oracle.ue8m0_decode(c) == math.ldexp(1.0, c - 127)


def mx_inputs():
    g = np.random.default_rng(4)
    x = g.standard_normal((6, 8 * MX)).astype(np.float32)
    x[0, 5] *= 30.0                       # an outlier in block 0
    x[1, :MX] = 0.0                       # an all-zero block
    x[1, MX:2 * MX] = 0.0
    x[1, MX + 7] = -3.0                   # a block with a single nonzero value
    x[2, :MX] *= 1e30                     # huge values
    x[2, MX:2 * MX] *= 1e-30              # tiny values
    x[3, 2 * MX:3 * MX] = -0.0
    x[4] = g.standard_normal(8 * MX).astype(np.float32) * 10.0 ** g.integers(-6, 6, 8 * MX)
    x[5, :MX] = 448.0 * 2.0 ** np.arange(-15, 17).astype(np.float32)
    return x


def test_mx_quantiser_equals_independent_computation():
    """numpy float64 for the shared exponent (frexp), torch's float8_e4m3fn
    cast (round to nearest even) for the elements after clamping to 448."""
    x = mx_inputs()
    q, sx = oracle.quant_mx_1x32(x)
    R, K = x.shape
    blocks = x.reshape(R, K // MX, MX).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, ex - 1 - 8, -127).clip(-127, 127)
    np.testing.assert_array_equal(sx, (e + 127).astype(np.uint8))
    scaled = np.ldexp(blocks, -e[:, :, None]).astype(np.float32).clip(-448, 448).reshape(R, K)
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # -0 inputs stay -0 in both; compare the bytes
    np.testing.assert_array_equal(q, ref)


def test_mx_quantiser_round_trip_and_block_maximum():
    x = mx_inputs()
    q, sx = oracle.quant_mx_1x32(x)
    dec = oracle.e4m3_decode_table()
    R, K = x.shape
    scale = np.ldexp(1.0, sx.astype(np.int64) - 127).repeat(MX, axis=1)
    back = dec[q] * scale
    xd = x.astype(np.float64)
    # below the top of the E4M3 range: half a step of the element grid
    inside = np.abs(xd) <= 448.0 * scale
    assert np.all((np.abs(xd - back) <= np.maximum(2.0 ** -4 * np.abs(xd), 2.0 ** -10 * scale))[inside])
    # above it (x / 2^e in (448, 512): the exponent comes from floor(log2 amax)),
    # the element saturates to +-448
    top = ~inside
    assert top.any()
    np.testing.assert_array_equal(np.abs(back[top]), 448.0 * scale[top])
    assert np.all(np.abs(xd[top]) < 512.0 * scale[top])
    assert np.all(np.sign(back[top]) == np.sign(xd[top]))
    # the largest element of every nonzero block codes to a magnitude in [256, 448]
    for r in range(R):
        for kb in range(K // MX):
            blk = xd[r, kb * MX:(kb + 1) * MX]
            if np.abs(blk).max() == 0:
                assert sx[r, kb] == 0 and np.all((q[r, kb * MX:(kb + 1) * MX] & 0x7F) == 0)
                continue
            i = int(np.abs(blk).argmax())
            mag = abs(dec[q[r, kb * MX + i]])
            if 0 < sx[r, kb] < 254:
                assert 256.0 <= mag <= 448.0, (r, kb, mag)


def exact_mx(g, M, N, K):
    a = int_codes(g.integers(-2, 3, (M, K)))
    b = int_codes(g.integers(-2, 3, (N, K)))
    sa = g.integers(124, 131, (M, K // MX)).astype(np.uint8)
    sb = g.integers(124, 131, (N, K // MX)).astype(np.uint8)
    return a, sa, b, sb


def test_mx_gemm_integer_codes_equal_blockwise_int64_matmul():
    """Codes of the integers -2..2 and power-of-two scales: each 32-block is an
    int64 matmul, scaled exactly in float64; the sum is exact, so D is its bf16
    rounding (a transposed operand, a swapped scale or a dropped block fails)."""
    g = np.random.default_rng(5)
    vals = {0x00: 0, 0x38: 1, 0x40: 2, 0xB8: -1, 0xC0: -2}
    for M, N, K in [(5, 7, 64), (33, 20, 320)]:
        a, sa, b, sb = exact_mx(g, M, N, K)
        ai = np.vectorize(vals.get)(a).astype(np.int64)
        bi = np.vectorize(vals.get)(b).astype(np.int64)
        ref = np.zeros((M, N))
        for kb in range(K // MX):
            blk = ai[:, kb * MX:(kb + 1) * MX] @ bi[:, kb * MX:(kb + 1) * MX].T
            ref += blk * np.ldexp(1.0, sa[:, kb].astype(np.int64) - 127)[:, None] \
                * np.ldexp(1.0, sb[:, kb].astype(np.int64) - 127)[None, :]
        np.testing.assert_array_equal(oracle.gemm_mx_nt(a, sa, b, sb), bf16_bits_of(ref.astype(np.float32)))


def test_mx_gemm_with_unit_scales_equals_fp8_gemm_with_unit_scales():
    """Cross-check of two oracle functions written separately: with every MX
    scale 2^0 and every FP8 scale 1.0, integer codes give exact sums in both,
    so the results are identical."""
    g = np.random.default_rng(6)
    M, N, K = 17, 24, 256
    a, _, b, _ = exact_mx(g, M, N, K)
    one_a = np.full((M, K // MX), 127, np.uint8)
    one_b = np.full((N, K // MX), 127, np.uint8)
    sfa = np.ones((K // 128, oracle.round_up(M, 4)), np.float32)
    sfb = np.ones((-(-N // 128), K // 128), np.float32)
    np.testing.assert_array_equal(oracle.gemm_mx_nt(a, one_a, b, one_b), oracle.gemm_nt(a, sfa, b, sfb))


def test_mx_gemm_scale_step_doubles_a_row():
    g = np.random.default_rng(7)
    a, sa, b, sb = exact_mx(g, 6, 9, 128)
    base = oracle.gemm_mx_nt(a, sa, b, sb)
    sa2 = sa.copy()
    sa2[2] += 1
    d2 = oracle.gemm_mx_nt(a, sa2, b, sb)
    np.testing.assert_array_equal(bits_to_f64(d2[2]), 2 * bits_to_f64(base[2]))
    np.testing.assert_array_equal(np.delete(d2, 2, axis=0), np.delete(base, 2, axis=0))


def test_mx_gemm_random_matches_float64_matmul():
    g = np.random.default_rng(8)
    M, N, K = 24, 40, 256
    qa, sa = oracle.quant_mx_1x32(g.standard_normal((M, K)).astype(np.float32))
    qb, sb = oracle.quant_mx_1x32(g.standard_normal((N, K)).astype(np.float32))
    dec = oracle.e4m3_decode_table()
    af = dec[qa] * np.ldexp(1.0, sa.astype(np.int64) - 127).repeat(MX, axis=1)
    bf = dec[qb] * np.ldexp(1.0, sb.astype(np.int64) - 127).repeat(MX, axis=1)
    ref = bf16_bits_of((af @ bf.T).astype(np.float32))
    d = oracle.gemm_mx_nt(qa, sa, qb, sb)
    assert (d == ref).mean() > 0.999
    assert np.all(np.abs(bits_to_f64(d) - bits_to_f64(ref)) <= np.abs(bits_to_f64(ref)) * 2.0 ** -7 + 1e-30)

"""Pins of the CPU oracle against things other than itself.

Each group below fixes one part of the oracle by closed forms, a library
routine that implements the same standard (torch's float8_e4m3fn and bfloat16
conversions, numpy float64 matmul), brute force on tiny inputs, or invariants,
so that a dropped term, a wrong sign or index, or a transposed operand fails at
least one of them.  No GPU is needed.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import random_dense

QB = 128


# ----------------------------------------------------------------- E4M3 ----
def test_decode_spot_values():
    # closed form: bias 7, 3 mantissa bits, subnormals m*2^-9, max 448, NaN 0x7F/0xFF
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x40) == 2.0
    assert oracle.e4m3_decode(0xB8) == -1.0
    z = oracle.e4m3_decode(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_decode_table_matches_torch_float8():
    ours = oracle.e4m3_decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.all(np.signbit(ours[~both_nan]) == np.signbit(ref[~both_nan]))


def test_decode_table_structure():
    t = oracle.e4m3_decode_table()
    assert np.isfinite(t).sum() == 254
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                     # strictly monotone 0x00..0x7E
    assert np.all(t[0x80:0xFF] == -t[:0x7F])            # sign symmetry


def _all_midpoints():
    t = oracle.e4m3_decode_table()[:0x7F]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)    # exact in fp32
    assert np.all(mids.astype(np.float64) == (t[:-1] + t[1:]) / 2)
    return t, mids


def test_encode_roundtrip_all_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_encode_ties_to_even_and_neighbours():
    t, mids = _all_midpoints()
    for i, m in enumerate(mids):
        lo, hi = i, i + 1
        even = lo if lo % 2 == 0 else hi
        assert oracle.e4m3_encode(float(m)) == even
        assert oracle.e4m3_encode(float(np.nextafter(m, np.float32(0)))) == lo
        assert oracle.e4m3_encode(float(np.nextafter(m, np.float32(1e9)))) == hi
        assert oracle.e4m3_encode(-float(m)) == 0x80 | even
    assert oracle.e4m3_encode(1.0625) == 0x38   # between 1 and 1.125 -> even 0x38
    assert oracle.e4m3_encode(1.1875) == 0x3A   # between 1.125 and 1.25 -> even 0x3A
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00


def test_encode_saturates():
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e30, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-1e-9) == 0x80 and oracle.e4m3_encode(-0.0) == 0x80


def test_encode_bisection_equals_bruteforce():
    t, mids = _all_midpoints()
    g = np.random.default_rng(5)
    xs = [mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
          t.astype(np.float32),
          g.standard_normal(3000).astype(np.float32) * np.float32(50),
          np.ldexp(g.random(2000), g.integers(-14, 10, 2000)).astype(np.float32)]
    for v in np.concatenate(xs):
        for s in (1.0, -1.0):
            x = float(np.float32(s * v))
            assert oracle.e4m3_encode(x) == oracle.e4m3_encode_bruteforce(x), x


def test_encode_matches_torch_below_448():
    g = np.random.default_rng(6)
    t, mids = _all_midpoints()
    x = np.concatenate([
        g.uniform(-447.9, 447.9, 20000).astype(np.float32),
        np.ldexp(g.uniform(-1, 1, 20000), g.integers(-16, 8, 20000)).astype(np.float32),
        mids[:-1], -mids[:-1], np.nextafter(mids, np.float32(0))[:-1]])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(ours, ref)


# ----------------------------------------------------------------- BF16 ----
def test_bf16_rne_matches_torch():
    g = np.random.default_rng(7)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(1000),
        # exact ties: low 16 bits == 0x8000
        ((g.integers(0, 0x7F00, 5000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -3.5, 65504.0, 3.4e38], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ----------------------------------------------------------- quantisers ----
def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _independent_act_quant(x: np.ndarray):
    """numpy amax + fp32 division, torch RNE cast (|x/s| <= 448 up to one ulp)."""
    M, K = x.shape
    xg = x.reshape(M, K // QB, QB)
    amax = np.abs(xg).max(axis=2)
    s = (np.maximum(amax, np.float32(1e-4)) / np.float32(448.0)).astype(np.float32)
    q = _torch_e4m3(xg / s[:, :, None]).reshape(M, K)
    return q, s.T


@pytest.mark.parametrize("M,K", [(1, 128), (5, 256), (129, 512), (64, 1024)])
def test_quant_act_matches_independent(M, K):
    g = np.random.default_rng(M * 1000 + K)
    x = wl.normal_matrix(g, (M, K), outliers=True)
    # distinct per-row and per-group magnitudes: a transposed sfa layout fails
    x *= np.ldexp(np.float32(1), g.integers(-6, 6, (M, 1))).astype(np.float32)
    x[:, :QB] *= np.float32(3.0)
    q, sfa = oracle.quant_act_1x128(x)
    q_ref, s_ref = _independent_act_quant(x)
    np.testing.assert_array_equal(q, q_ref)
    assert sfa.shape == (K // QB, oracle.round_up(M, 4))
    np.testing.assert_array_equal(sfa[:, :M], s_ref)
    assert np.all(sfa[:, M:] == 0)


def test_quant_act_roundtrip_bound_and_amax():
    g = np.random.default_rng(11)
    x = wl.normal_matrix(g, (33, 384), outliers=True)
    q, sfa = oracle.quant_act_1x128(x)
    dec = oracle.e4m3_decode_table()
    for kb in range(3):
        s = sfa[kb, :33].astype(np.float64)[:, None]
        xs = x[:, kb * QB:(kb + 1) * QB].astype(np.float64)
        back = dec[q[:, kb * QB:(kb + 1) * QB]] * s
        bound = (2.0 ** -4 + 2.0 ** -20) * np.abs(xs) + 2.0 ** -10 * s
        assert np.all(np.abs(xs - back) <= bound)
        # the element of largest magnitude lands on +-448 exactly
        idx = np.abs(xs).argmax(axis=1)
        codes = q[np.arange(33), kb * QB + idx]
        assert np.all((codes & 0x7F) == 0x7E)


def test_quant_act_zero_group_and_bf16_input():
    x = np.zeros((4, 256), dtype=np.float32)
    x[1, 200] = -3.0
    q, sfa = oracle.quant_act_1x128(x)
    s0 = np.float32(np.float32(1e-4) / np.float32(448.0))
    assert sfa[0, 0] == s0 and np.all(q[0] == 0)
    assert q[1, 200] == 0xFE and sfa[1, 1] == np.float32(3.0) / np.float32(448)
    # bf16 input: widened exactly, then the same rule
    g = np.random.default_rng(12)
    xf = g.standard_normal((7, 256)).astype(np.float32)
    xb = torch.from_numpy(xf).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    q1, s1 = oracle.quant_act_1x128(bits)
    q2, s2 = oracle.quant_act_1x128(xb.float().numpy())
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (192, 256), (2112 // 8, 256)])
def test_quant_weight_matches_independent(N, K):
    g = np.random.default_rng(N + K)
    w = wl.normal_matrix(g, (N, K))
    w *= np.ldexp(np.float32(1), g.integers(-4, 4, (N, 1))).astype(np.float32)
    q, sfb = oracle.quant_weight_128x128(w)
    NB, KB = -(-N // QB), K // QB
    assert sfb.shape == (NB, KB)
    for nb in range(NB):
        for kb in range(KB):
            blk = w[nb * QB:(nb + 1) * QB, kb * QB:(kb + 1) * QB]
            s = np.float32(max(np.abs(blk).max(), np.float32(1e-4)) / np.float32(448.0))
            assert sfb[nb, kb] == s
            np.testing.assert_array_equal(
                q[nb * QB:(nb + 1) * QB, kb * QB:(kb + 1) * QB], _torch_e4m3(blk / s))


# ------------------------------------------------------------------ GEMM ----
E4M3_OF_INT = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}


def _codes(v: np.ndarray) -> np.ndarray:
    lut = np.zeros(5, dtype=np.uint8)
    for k, c in E4M3_OF_INT.items():
        lut[k + 2] = c
    return lut[v.astype(np.int64) + 2]


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_case(M, N, K, seed):
    g = np.random.default_rng(seed)
    ai = wl.exact_operands(g, (M, K))
    bi = wl.exact_operands(g, (N, K))
    ld = oracle.round_up(M, 4)
    sfa = np.zeros((K // QB, ld), dtype=np.float32)
    sfa[:, :M] = wl.exact_scales(g, (K // QB, M))
    sfb = wl.exact_scales(g, (-(-N // QB), K // QB))
    return ai, bi, sfa, sfb


def exact_reference(ai, bi, sfa, sfb):
    """Integer block sums (int64 matmul) times the scales, summed in float64:
    exact for these inputs, so it equals every correct fp32 promotion."""
    M, K = ai.shape
    N = bi.shape[0]
    out = np.zeros((M, N), dtype=np.float64)
    nb_of_col = np.arange(N) // QB
    for kb in range(K // QB):
        p = ai[:, kb * QB:(kb + 1) * QB].astype(np.int64) @ bi[:, kb * QB:(kb + 1) * QB].astype(np.int64).T
        scale = sfa[kb, :M].astype(np.float64)[:, None] * sfb[nb_of_col, kb].astype(np.float64)[None, :]
        out += p * scale
    return out


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (1, 128, 128), (129, 192, 384), (37, 264, 256)])
def test_gemm_exact_against_integer_matmul(M, N, K):
    ai, bi, sfa, sfb = exact_case(M, N, K, seed=M + N + K)
    d, acc = oracle.gemm_nt(_codes(ai), sfa, _codes(bi), sfb, want_acc=True)
    ref = exact_reference(ai, bi, sfa, sfb)
    assert np.all(acc.astype(np.float64) == ref)
    np.testing.assert_array_equal(d, _bf16_bits(ref.astype(np.float32)))


def _dequant_reference(qa, sfa, qb, sfb):
    """Independent float64 path: dequantise both operands with their scales,
    then one numpy matmul A_deq . B_deq^T."""
    dec = oracle.e4m3_decode_table()
    M, K = qa.shape
    N = qb.shape[0]
    a = dec[qa] * np.repeat(sfa[:, :M].T.astype(np.float64), QB, axis=1)
    sb_full = np.repeat(np.repeat(sfb.astype(np.float64), QB, axis=0)[:N], QB, axis=1)
    b = dec[qb] * sb_full
    return a @ b.T


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (65, 200, 384), (3, 136, 1024)])
def test_gemm_random_against_dequantised_matmul(M, N, K):
    x, w = wl.dense_inputs(M, N, K, seed=M * 7 + N, outliers=True)
    qa, sfa = oracle.quant_act_1x128(x)
    qb, sfb = oracle.quant_weight_128x128(w)
    d, acc = oracle.gemm_nt(qa, sfa, qb, sfb, want_acc=True)
    ref = _dequant_reference(qa, sfa, qb, sfb)
    # differences: fp32 rounding of each block sum, of the scale product and of
    # each promotion step; bounded by ~ (3 + K/128) * 2^-24 * sum|terms|
    scale_ref = np.abs(ref).max()
    assert np.max(np.abs(acc - ref)) <= (3 + K // QB) * 2.0 ** -23 * scale_ref * 4
    # and the bf16 output is the RNE of the fp32 accumulator
    np.testing.assert_array_equal(d, _bf16_bits(acc))
    # the same product with B transposed in the reference would not match
    if N == M:
        pytest.skip("square")
    assert not np.allclose(acc[:min(M, N), :min(M, N)], ref.T[:min(M, N), :min(M, N)], rtol=1e-2)


def test_gemm_promotion_is_fp32_fma_in_block_order():
    # Two K blocks whose fp32 promotion rounds differently from a float64 sum:
    # acc = fma(p1, s1, fma(p0, s0, 0)) in fp32.
    K = 256
    a = np.zeros((1, K), dtype=np.uint8)
    b = np.zeros((1, K), dtype=np.uint8)
    a[0, 0] = 0x38          # 1.0 in block 0
    b[0, 0] = 0x38
    a[0, 128] = 0x38        # 1.0 in block 1
    b[0, 128] = 0x38
    sfa = np.zeros((2, 4), dtype=np.float32)
    sfa[0, 0] = np.float32(1.0)
    sfa[1, 0] = np.float32(2.0 ** -25)
    sfb = np.ones((1, 2), dtype=np.float32)
    d, acc = oracle.gemm_nt(a, sfa, b, sfb, want_acc=True)
    # 1 + 2^-25 rounds to 1 in fp32 (tie to even)
    assert acc[0, 0] == np.float32(1.0)
    sfa[1, 0] = np.float32(3 * 2.0 ** -25)
    d, acc = oracle.gemm_nt(a, sfa, b, sfb, want_acc=True)
    assert acc[0, 0] == np.float32(1.0 + 2.0 ** -23)


def test_gemm_invariants_zero_rows_and_scaling():
    ai, bi, sfa, sfb = exact_case(64, 256, 384, seed=3)
    qa, qb = _codes(ai), _codes(bi)
    d0, acc0 = oracle.gemm_nt(qa, sfa, qb, sfb, want_acc=True)
    qa2 = qa.copy()
    qa2[5] = 0
    sfa2 = sfa.copy()
    sfa2[:, 9] = 0
    sfa2[:, 17] *= 2
    d1, acc1 = oracle.gemm_nt(qa2, sfa2, qb, sfb, want_acc=True)
    assert np.all(acc1[5] == 0) and np.all(acc1[9] == 0)
    assert np.all(acc1[17] == 2 * acc0[17])
    keep = [r for r in range(64) if r not in (5, 9, 17)]
    assert np.all(acc1[keep] == acc0[keep])


def test_gemm_rows_subset_leaves_others():
    x, w = wl.dense_inputs(40, 128, 256, seed=9)
    qa, sfa = oracle.quant_act_1x128(x)
    qb, sfb = oracle.quant_weight_128x128(w)
    full = oracle.gemm_nt(qa, sfa, qb, sfb)
    rows = np.array([0, 7, 39], dtype=np.int32)
    d = np.full((40, 128), wl.SENTINEL_BF16, dtype=np.uint16)
    part = oracle.gemm_nt(qa, sfa, qb, sfb, rows=rows, d=d)
    np.testing.assert_array_equal(part[rows], full[rows])
    others = np.setdiff1d(np.arange(40), rows)
    assert np.all(part[others] == wl.SENTINEL_BF16)


# ---------------------------------------------------------- MoE layouts ----
def test_contiguous_equals_per_expert_dense():
    G, N, K = 3, 136, 256
    counts, m_indices, seg = wl.contiguous_routing(G, 300, seed=4)
    x = wl.normal_matrix(np.random.default_rng(1), (len(m_indices), K))
    w = wl.normal_matrix(np.random.default_rng(2), (G, N, K))
    qa, sfa = oracle.quant_act_1x128(x)
    qb, sfb = oracle.quant_weight_128x128(w)
    d = np.full((len(m_indices), N), wl.SENTINEL_BF16, dtype=np.uint16)
    out = oracle.grouped_contiguous(qa, sfa, qb, sfb, m_indices, d=d)
    for e in range(G):
        rows = np.arange(seg[e], seg[e] + counts[e])
        qx, sx = oracle.quant_act_1x128(x[rows])
        ref = oracle.gemm_nt(qx, sx, qb[e], sfb[e])
        np.testing.assert_array_equal(out[rows], ref)
    assert np.all(out[m_indices < 0] == wl.SENTINEL_BF16)


def test_masked_equals_per_expert_dense_and_leaves_tail():
    G, max_m, N, K = 4, 40, 128, 256
    g = np.random.default_rng(8)
    x = wl.normal_matrix(g, (G, max_m, K))
    w = wl.normal_matrix(g, (G, N, K))
    masked_m = np.array([0, 1, 40, 57], dtype=np.int32)  # 57 > max_m reads as 40
    qa = np.empty((G, max_m, K), dtype=np.uint8)
    sfa = np.zeros((G, K // QB, oracle.round_up(max_m, 4)), dtype=np.float32)
    for e in range(G):
        qa[e], sfa[e] = oracle.quant_act_1x128(x[e])
    qb, sfb = oracle.quant_weight_128x128(w)
    d = np.full((G, max_m, N), wl.SENTINEL_BF16, dtype=np.uint16)
    out = oracle.grouped_masked(qa, sfa, qb, sfb, masked_m, d=d)
    for e in range(G):
        valid = min(int(masked_m[e]), max_m)
        ref = oracle.gemm_nt(qa[e], sfa[e], qb[e], sfb[e])
        np.testing.assert_array_equal(out[e, :valid], ref[:valid])
        assert np.all(out[e, valid:] == wl.SENTINEL_BF16)


def test_masked_full_equals_batched_dense():
    G, max_m, N, K = 2, 16, 128, 128
    g = np.random.default_rng(9)
    ai = wl.exact_operands(g, (G, max_m, K))
    bi = wl.exact_operands(g, (G, N, K))
    sfa = np.zeros((G, 1, 16), dtype=np.float32)
    sfa[:] = wl.exact_scales(g, (G, 1, 16))
    sfb = wl.exact_scales(g, (G, 1, 1))
    out = oracle.grouped_masked(_codes(ai), sfa, _codes(bi), sfb, np.array([16, 16], np.int32))
    for e in range(G):
        ref = exact_reference(ai[e], bi[e], sfa[e], sfb[e])
        np.testing.assert_array_equal(out[e], _bf16_bits(ref.astype(np.float32)))


# ------------------------------------------------- re-quantised GEMM output --
def _check_requant(d_bits, q, sfo, rows):
    """Each listed row of q/sfo re-encodes the bf16 output d_bits: within the
    quantiser's round-trip bound, and each group's largest element on +-448."""
    dec = oracle.e4m3_decode_table()
    d = oracle.bf16_bits_to_f32(d_bits).astype(np.float64)
    for nb in range(d.shape[1] // QB):
        cols = slice(nb * QB, (nb + 1) * QB)
        s = sfo[nb, rows].astype(np.float64)[:, None]
        x = d[rows][:, cols]
        back = dec[q[rows][:, cols]] * s
        assert np.all(np.abs(x - back) <= (2.0 ** -4 + 2.0 ** -20) * np.abs(x) + 2.0 ** -10 * s)
        big = np.abs(x).max(axis=1) >= 1e-4
        idx = np.abs(x).argmax(axis=1)
        codes = q[rows][np.arange(len(rows)), nb * QB + idx]
        assert np.all((codes[big] & 0x7F) == 0x7E)


def test_gemm_quant_reencodes_the_bf16_output():
    a, sfa, b, sfb = random_dense(130, 384, 640, seed=41)
    q, sfo = oracle.gemm_nt_quant(a, sfa, b, sfb)
    assert q.shape == (130, 384) and sfo.shape == (3, 132)
    _check_requant(oracle.gemm_nt(a, sfa, b, sfb), q, sfo, np.arange(130))
    assert np.all(sfo[:, 130:] == 0)


def test_grouped_quant_leaves_uncomputed_rows():
    # masked: rows at or beyond masked_m keep their contents
    g = np.random.default_rng(5)
    G, max_m, N, K = 3, 70, 256, 256
    a = np.stack([random_dense(max_m, N, K, seed=50 + e)[0] for e in range(G)])
    sfa = np.stack([random_dense(max_m, N, K, seed=50 + e)[1] for e in range(G)])
    b = np.stack([random_dense(8, N, K, seed=60 + e)[2] for e in range(G)])
    sfb = np.stack([random_dense(8, N, K, seed=60 + e)[3] for e in range(G)])
    mm = np.array([70, 0, 33], np.int32)
    q0 = g.integers(0, 256, (G, max_m, N)).astype(np.uint8)
    s0 = g.random((G, N // QB, oracle.round_up(max_m, 4))).astype(np.float32)
    q, sfo = oracle.grouped_masked_quant(a, sfa, b, sfb, mm, q0.copy(), s0.copy())
    d = oracle.grouped_masked(a, sfa, b, sfb, mm)
    for e in range(G):
        _check_requant(d[e], q[e], sfo[e], np.arange(mm[e]))
        np.testing.assert_array_equal(q[e, mm[e]:], q0[e, mm[e]:])
        np.testing.assert_array_equal(sfo[e][:, mm[e]:], s0[e][:, mm[e]:])
    # contiguous: padding rows (index -1) keep their contents
    counts, mi, _ = wl.contiguous_routing(2, 200, seed=9)
    ac, sac = random_dense(len(mi), N, K, seed=70)[:2]
    q0 = g.integers(0, 256, (len(mi), N)).astype(np.uint8)
    s0 = g.random((N // QB, oracle.round_up(len(mi), 4))).astype(np.float32)
    q, sfo = oracle.grouped_contiguous_quant(ac, sac, b[:2], sfb[:2], mi, q0.copy(), s0.copy())
    pad = mi < 0
    np.testing.assert_array_equal(q[pad], q0[pad])
    np.testing.assert_array_equal(sfo[:, :len(mi)][:, pad], s0[:, :len(mi)][:, pad])
    _check_requant(oracle.grouped_contiguous(ac, sac, b[:2], sfb[:2], mi), q, sfo, np.flatnonzero(~pad))

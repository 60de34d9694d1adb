"""GPU parity of the two formats beside per-group-scaled FP8 (2kiu.com DeepGEMM
tutorial 1, 2.2 and 7): the BF16 GEMM and the MX (E4M3 elements, E8M0 scale
per 32 K values) quantiser and GEMM, through the C ABI, against the oracle.
Integer-valued cases are exact at every step, so they must match bit for bit;
random cases meet the stated tolerance."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg
import oracle
import workloads as wl
from helpers import bf16_bits_to_f32, int_codes, mx_scales_chunk_major, mx_scales_row_major, tolerance_check

pytestmark = pytest.mark.gpu

MX = 32


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    dg.load()
    dg.dg_read_device_status()
    yield
    assert not (dg.dg_read_device_status() & dg.DG_DEVFLAG_TIMEOUT)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_of(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (round to nearest even) of fp32 values."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def to_bf16_tensor(b: np.ndarray) -> torch.Tensor:
    return dev(b.view(np.int16)).view(torch.bfloat16)


# ------------------------------------------------------------------- BF16 --
BF16_SHAPES = [(128, 256, 64), (1, 8, 64), (300, 520, 640), (257, 200, 1152), (1000, 1288, 384), (129, 264, 4096)]


@pytest.fixture(params=["0", "1"], ids=["one_sm", "pair"])
def acc_pair(request, monkeypatch):
    """Both BF16 kernels: 128 x 256 tiles on one SM, 256 x 256 on a CTA pair."""
    monkeypatch.setenv("DG_FORCE_ACC_PAIR", request.param)
    return request.param


@pytest.mark.parametrize("M,N,K", BF16_SHAPES)
def test_bf16_integer_values_bit_identical(M, N, K, acc_pair):
    # integers in [-4, 4]: every product and every sum (|.| <= 16 K) is exact
    # in fp32, so the tensor core's order of summation cannot change a bit
    g = np.random.default_rng(M + N + K)
    a = bf16_of(g.integers(-4, 5, (M, K)).astype(np.float32))
    b = bf16_of(g.integers(-4, 5, (N, K)).astype(np.float32))
    d = dg.dg_bf16_gemm_nt(to_bf16_tensor(a), to_bf16_tensor(b))
    np.testing.assert_array_equal(bits(d), oracle.gemm_bf16_nt(a, b))


@pytest.mark.parametrize("M,N,K", [(300, 520, 640), (1000, 1288, 2048)])
def test_bf16_random_tolerance(M, N, K, acc_pair):
    g = np.random.default_rng(3 * M + K)
    a = bf16_of(g.standard_normal((M, K)).astype(np.float32))
    b = bf16_of(g.standard_normal((N, K)).astype(np.float32))
    d = dg.dg_bf16_gemm_nt(to_bf16_tensor(a), to_bf16_tensor(b))
    rows = wl.sample_rows(M, 64, 11, must=[0, M - 1, 127, 128])
    ref = oracle.gemm_bf16_nt(a, b, rows=rows)
    tolerance_check(bf16_bits_to_f32(bits(d)[rows]), bf16_bits_to_f32(ref[rows]), "bf16")


def test_bf16_full_size_exact_sampled():
    """The benchmark's BF16 shape (M=4096, N=7168, K=7168) in the plan the
    library picks (the CTA pair), integer operands: sampled rows bit for bit."""
    M, N, K = 4096, 7168, 7168
    g = np.random.default_rng(4242)
    a = bf16_of(g.integers(-2, 3, (M, K)).astype(np.float32))
    b = bf16_of(g.integers(-2, 3, (N, K)).astype(np.float32))
    d = dg.dg_bf16_gemm_nt(to_bf16_tensor(a), to_bf16_tensor(b))
    rows = wl.sample_rows(M, 16, 5, must=[0, 127, 128, 255, 256, M - 1])
    ref = oracle.gemm_bf16_nt(a, b, rows=rows)
    np.testing.assert_array_equal(bits(d)[rows], ref[rows])


# --------------------------------------------------------------------- MX --
@pytest.mark.parametrize("R,K", [(300, 1024), (1, 128), (129, 384)])
def test_mx_quantiser_bit_exact(R, K):
    g = np.random.default_rng(R + K)
    x = wl.normal_matrix(g, (R, K), outliers=True)
    x[0, :MX] = 0.0                                   # an all-zero block
    x[-1, MX:2 * MX] *= np.float32(1e-30)             # a block of tiny values
    if K >= 4 * MX:
        x[R // 2, 3 * MX:4 * MX] = np.float32(448.0)  # amax exactly a power-of-two boundary case
    q, sx = dg.dg_quant_mx_1x32(dev(x))
    q_ref, sx_ref = oracle.quant_mx_1x32(x)
    np.testing.assert_array_equal(mx_scales_row_major(sx.cpu().numpy()), sx_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


def exact_mx(g, M, N, K):
    """Codes of the integers -2..2 and scales 2^-3..2^3: every 32-block sum
    (|.| <= 128), its scaling (2^-6..2^6) and the running fp32 sum (multiples
    of 2^-6 below 2^18 for K <= 768) are exact, so the result is unique."""
    a = int_codes(g.integers(-2, 3, (M, K)))
    b = int_codes(g.integers(-2, 3, (N, K)))
    sa = g.integers(124, 131, (M, K // MX)).astype(np.uint8)
    sb = g.integers(124, 131, (N, K // MX)).astype(np.uint8)
    return a, sa, b, sb


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (129, 136, 128), (300, 264, 640), (1000, 520, 768), (1, 8, 384)])
def test_mx_gemm_exact_bit_identical(M, N, K, acc_pair):
    g = np.random.default_rng(7 * M + N + K)
    a, sa, b, sb = exact_mx(g, M, N, K)
    d = dg.dg_mx_gemm_nt(dev(a), dev(mx_scales_chunk_major(sa)), dev(b), dev(mx_scales_chunk_major(sb)))
    np.testing.assert_array_equal(bits(d), oracle.gemm_mx_nt(a, sa, b, sb))


def test_mx_gemm_each_block_scale_lands_on_its_block(acc_pair):
    """Rows of A and of B (in both 128-row halves of a tile) carry a distinct
    scale in every 32-wide block (so a scale applied to the wrong K block or
    the wrong row changes the result); exact inputs, bit for bit."""
    g = np.random.default_rng(99)
    M, N, K = 256, 256, 512
    a, sa, b, sb = exact_mx(g, M, N, K)
    sa[5] = 124 + (np.arange(K // MX) % 7)
    sa[100] = 125 + (np.arange(K // MX) % 5)
    sa[150] = 129 - (np.arange(K // MX) % 4)      # the second CTA's rows of a pair tile
    sb[17] = 130 - (np.arange(K // MX) % 7)
    sb[200] = 124 + (np.arange(K // MX) % 6)      # the second 128-row half of a 256-wide tile
    d = dg.dg_mx_gemm_nt(dev(a), dev(mx_scales_chunk_major(sa)), dev(b), dev(mx_scales_chunk_major(sb)))
    np.testing.assert_array_equal(bits(d), oracle.gemm_mx_nt(a, sa, b, sb))


@pytest.mark.parametrize("M,N,K", [(300, 520, 1024), (1000, 1288, 2048)])
def test_mx_quantise_then_gemm_tolerance(M, N, K, acc_pair):
    g = np.random.default_rng(M + 2 * N)
    x = wl.normal_matrix(g, (M, K), outliers=True)
    w = wl.normal_matrix(g, (N, K))
    qa, sa = dg.dg_quant_mx_1x32(dev(x))
    qb, sb = dg.dg_quant_mx_1x32(dev(w))
    d = dg.dg_mx_gemm_nt(qa, sa, qb, sb)
    qa_r, sa_r = oracle.quant_mx_1x32(x)
    qb_r, sb_r = oracle.quant_mx_1x32(w)
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_r)
    np.testing.assert_array_equal(mx_scales_row_major(sb.cpu().numpy()), sb_r)
    rows = wl.sample_rows(M, 64, 12, must=[0, M - 1, 127, 128])
    ref = oracle.gemm_mx_nt(qa_r, sa_r, qb_r, sb_r, rows=rows)
    tolerance_check(bf16_bits_to_f32(bits(d)[rows]), bf16_bits_to_f32(ref[rows]), "mx")


def test_mx_full_size_exact_sampled():
    """The benchmark's MX shape (M=4096, N=7168, K=7168) in the plan the
    library picks (the CTA pair), exact operands and power-of-two scales:
    sampled rows bit for bit."""
    M, N, K = 4096, 7168, 7168
    g = np.random.default_rng(4343)
    a, _, b, _ = exact_mx(g, M, N, K)
    # scales 2^-3..2^0: block sums (|.| <= 128) scaled by at most 1 and summed
    # over 224 blocks stay below 2^15 in multiples of 2^-6, exact in fp32
    sa = g.integers(124, 128, (M, K // MX)).astype(np.uint8)
    sb = g.integers(124, 128, (N, K // MX)).astype(np.uint8)
    d = dg.dg_mx_gemm_nt(dev(a), dev(mx_scales_chunk_major(sa)), dev(b), dev(mx_scales_chunk_major(sb)))
    rows = wl.sample_rows(M, 12, 6, must=[0, 127, 128, 255, 256, M - 1])
    ref = oracle.gemm_mx_nt(a, sa, b, sb, rows=rows)
    np.testing.assert_array_equal(bits(d)[rows], ref[rows])

"""GEMMs whose epilogue re-quantises the output (E4M3 codes + one fp32 scale
per 1x128 group of each row) against the oracle, through the C ABI.

The output is defined as the 1x128 quantiser applied to the GEMM's bf16
result, so: exact-arithmetic inputs match the oracle bit for bit; random
inputs match the GPU's own two-call pipeline (bf16 GEMM, then the quantiser)
bit for bit, and the oracle within the bounds a one-ulp bf16 difference
allows.  Rows the bf16 call would not write keep their bytes."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg
import oracle
import workloads as wl
from helpers import QB, bf16_bits_to_f32, exact_dense, random_dense

pytestmark = pytest.mark.gpu

Q_SENTINEL = 0x5A           # byte the untouched rows of q keep
SF_SENTINEL = -3.0          # value the untouched scales keep


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    dg.load()
    dg.dg_read_device_status()


@pytest.fixture(params=["128", "256"], ids=["bn128", "pair256"])
def qtile(request, monkeypatch):
    """Runs the test on the one-SM 128 x 128 tiles and on the CTA-pair 256 x
    256 tiles (DG_FORCE_BN; the masked layout keeps the one-SM tiles).  The
    two-call pipelines the random cases compare with use the same tiles, so
    that both sides see the tensor core's same summation."""
    monkeypatch.setenv("DG_FORCE_BN", request.param)
    return request.param


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def q_sf_buffers(q_shape, sf_shape):
    q = torch.full(q_shape, Q_SENTINEL, dtype=torch.uint8, device="cuda")
    sfo = torch.full(sf_shape, SF_SENTINEL, dtype=torch.float32, device="cuda")
    return q, sfo


def q_sf_sentinels(q_shape, sf_shape):
    return np.full(q_shape, Q_SENTINEL, np.uint8), np.full(sf_shape, SF_SENTINEL, np.float32)


def unfused_dense(a, sfa, b, sfb):
    """The GPU's two-call pipeline on the tiles DG_FORCE_BN names: bf16 D,
    then the 1x128 quantiser of D."""
    d = dg.dg_fp8_gemm_nt(dev(a), dev(sfa), dev(b), dev(sfb))
    q, sfo = dg.dg_quant_act_1x128(d)
    return host(d.view(torch.int16)).view(np.uint16), host(q), host(sfo)


def signed_steps(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes as signed step counts (magnitude codes are monotone; the
    two zeros coincide)."""
    mag = (codes & 0x7F).astype(np.int32)
    return np.where(codes & 0x80, -mag, mag)


def check_near_oracle(q, sfo, q_ref, sfo_ref, d_gpu, d_ref, what):
    """Random inputs: where the GPU's bf16 D equals the oracle's for a whole
    1x128 group the codes and the scale are identical; elsewhere the scale is
    within the relative change of the group's amax, and each code within one
    E4M3 step plus what the D difference moves it."""
    M, N = d_ref.shape
    groups = N // QB
    dg_ = d_gpu.reshape(M, groups, QB)
    dr_ = d_ref.reshape(M, groups, QB)
    same = np.all(dg_ == dr_, axis=2)                      # [M, groups]
    qg = q.reshape(M, groups, QB)
    qr = q_ref.reshape(M, groups, QB)
    np.testing.assert_array_equal(qg[same], qr[same], err_msg=f"{what}: codes of identical groups")
    np.testing.assert_array_equal(sfo.T[same], sfo_ref.T[same], err_msg=f"{what}: scales of identical groups")
    assert same.mean() > 0.5, f"{what}: only {same.mean():.2f} of the groups agree in bf16"
    # the rest: dequantised values within the E4M3 rounding of each side
    lut = oracle.e4m3_decode_table()
    deq = lut[q].reshape(M, groups, QB) * sfo.T[:, :, None]
    deq_ref = lut[q_ref].reshape(M, groups, QB) * sfo_ref.T[:, :, None]
    f_g = bf16_bits_to_f32(dg_).astype(np.float64)
    f_r = bf16_bits_to_f32(dr_).astype(np.float64)
    # half an E4M3 step of each side: 2^-4 relative, or half the subnormal step
    bound = (2.0 ** -4 * (np.abs(f_g) + np.abs(f_r)) + 2.0 ** -10 * (sfo.T + sfo_ref.T)[:, :, None]
             + np.abs(f_g - f_r))
    assert np.all(np.abs(deq - deq_ref) <= bound * (1 + 1e-6)), f"{what}: dequantised values apart"


# ------------------------------------------------------------------ dense --
DENSE_Q_SHAPES = [(128, 256, 512), (1, 128, 128), (129, 384, 384), (300, 640, 640), (513, 1024, 256),
                  (3, 128, 1152), (4224, 1280, 256)]


@pytest.mark.parametrize("M,N,K", DENSE_Q_SHAPES)
def test_dense_q_exact_bit_identical(M, N, K, qtile):
    a, sfa, b, sfb = exact_dense(M, N, K, seed=M * 7 + N + K)
    q, sfo = q_sf_buffers((M, N), (N // QB, oracle.round_up(M, 4)))
    dg.dg_fp8_gemm_nt_q(dev(a), dev(sfa), dev(b), dev(sfb), q, sfo)
    q_ref, sfo_ref = q_sf_sentinels((M, N), (N // QB, oracle.round_up(M, 4)))
    oracle.gemm_nt_quant(a, sfa, b, sfb, q_ref, sfo_ref)
    np.testing.assert_array_equal(host(q), q_ref)
    np.testing.assert_array_equal(host(sfo), sfo_ref)


@pytest.mark.parametrize("M,N,K", [(300, 640, 1024), (129, 256, 2048), (1024, 1536, 512)])
def test_dense_q_random_equals_two_call_pipeline(M, N, K, qtile):
    a, sfa, b, sfb = random_dense(M, N, K, seed=M + 3 * N + K, outliers=True)
    q, sfo = dg.dg_fp8_gemm_nt_q(dev(a), dev(sfa), dev(b), dev(sfb))
    d2, q2, sfo2 = unfused_dense(a, sfa, b, sfb)
    np.testing.assert_array_equal(host(q), q2)
    np.testing.assert_array_equal(host(sfo), sfo2)
    q_ref, sfo_ref = oracle.gemm_nt_quant(a, sfa, b, sfb)
    d_ref = oracle.gemm_nt(a, sfa, b, sfb)
    check_near_oracle(q2, sfo2[:, :M], q_ref, sfo_ref[:, :M], d2, d_ref, f"dense {M}x{N}x{K}")


def test_dense_q_repeatable():
    a, sfa, b, sfb = random_dense(256, 512, 1024, seed=41)
    first = [host(t) for t in dg.dg_fp8_gemm_nt_q(dev(a), dev(sfa), dev(b), dev(sfb))]
    for _ in range(3):
        again = [host(t) for t in dg.dg_fp8_gemm_nt_q(dev(a), dev(sfa), dev(b), dev(sfb))]
        np.testing.assert_array_equal(again[0], first[0])
        np.testing.assert_array_equal(again[1], first[1])


def test_dense_q_zero_groups_take_the_floor_scale():
    """A zero row group has amax 0: its scale is the floor 1e-4/448 and its
    codes are zero (the quantiser's rule for an all-zero group)."""
    M, N, K = 130, 256, 256
    a, sfa, b, sfb = exact_dense(M, N, K, seed=9)
    a[5] = 0
    b[128:] = 0
    q, sfo = dg.dg_fp8_gemm_nt_q(dev(a), dev(sfa), dev(b), dev(sfb))
    q, sfo = host(q), host(sfo)
    floor = np.float32(np.float32(1e-4) / np.float32(448.0))
    assert np.all(q[5] == 0) and np.all(sfo[:, 5] == floor)
    assert np.all(q[:, 128:] == 0) and np.all(sfo[1, :M] == floor)
    q_ref, sfo_ref = oracle.gemm_nt_quant(a, sfa, b, sfb)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sfo, sfo_ref)


# ------------------------------------------------------------- contiguous --
def contiguous_case(G, tokens, N, K, seed):
    counts, m_indices, seg = wl.contiguous_routing(G, tokens, seed)
    sum_M = len(m_indices)
    a, sfa, _, _ = exact_dense(sum_M, 8, K, seed)
    bs = [exact_dense(8, N, K, seed + 10 + e) for e in range(G)]
    return a, sfa, np.stack([x[2] for x in bs]), np.stack([x[3] for x in bs]), m_indices


@pytest.mark.parametrize("G,tokens,N,K", [(4, 700, 256, 512), (3, 129, 128, 128), (8, 1500, 384, 384)])
def test_contiguous_q_exact_bit_identical(G, tokens, N, K, qtile):
    a, sfa, b, sfb, mi = contiguous_case(G, tokens, N, K, seed=G * 5 + tokens)
    sum_M = a.shape[0]
    q, sfo = q_sf_buffers((sum_M, N), (N // QB, sum_M))
    dg.dg_fp8_grouped_contiguous_q(dev(a), dev(sfa), dev(b), dev(sfb), dev(mi), q, sfo)
    q_ref, sfo_ref = q_sf_sentinels((sum_M, N), (N // QB, sum_M))
    oracle.grouped_contiguous_quant(a, sfa, b, sfb, mi, q_ref, sfo_ref)
    q, sfo = host(q), host(sfo)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sfo, sfo_ref)
    pad = mi < 0
    assert pad.any() and np.all(q[pad] == Q_SENTINEL) and np.all(sfo[:, pad] == SF_SENTINEL)


def test_contiguous_q_random_equals_two_call_pipeline(qtile):
    G, tokens, N, K = 6, 900, 512, 1024
    counts, mi, seg = wl.contiguous_routing(G, tokens, seed=77)
    g = np.random.default_rng(78)
    a, sfa = oracle.quant_act_1x128(wl.normal_matrix(g, (len(mi), K), outliers=True))
    b, sfb = oracle.quant_weight_128x128(wl.normal_matrix(g, (G, N, K)))
    q, sfo = dg.dg_fp8_grouped_contiguous_q(dev(a), dev(sfa), dev(b), dev(sfb), dev(mi))
    d = dg.dg_fp8_grouped_contiguous(dev(a), dev(sfa), dev(b), dev(sfb), dev(mi))
    q2, sfo2 = dg.dg_quant_act_1x128(d)
    valid = mi >= 0
    q, sfo, q2, sfo2 = host(q), host(sfo), host(q2), host(sfo2)
    np.testing.assert_array_equal(q[valid], q2[valid])
    np.testing.assert_array_equal(sfo[:, valid], sfo2[:, valid])


# ----------------------------------------------------------------- masked --
def masked_case(G, max_m, N, K, seed):
    ld = oracle.round_up(max_m, 4)
    a = np.empty((G, max_m, K), np.uint8)
    sfa = np.zeros((G, K // QB, ld), np.float32)
    b = np.empty((G, N, K), np.uint8)
    sfb = np.empty((G, N // QB, K // QB), np.float32)
    for e in range(G):
        a[e], sfa[e], b[e], sfb[e] = exact_dense(max_m, N, K, seed + e)
    return a, sfa, b, sfb


@pytest.mark.parametrize("G,max_m,N,K,mm", [
    (4, 256, 256, 512, [0, 1, 255, 256]),
    (3, 200, 384, 384, [200, 129, 128]),
    (5, 130, 128, 640, [130, 0, 7, 129, 1]),
])
def test_masked_q_exact_bit_identical(G, max_m, N, K, mm):
    a, sfa, b, sfb = masked_case(G, max_m, N, K, seed=G * 13 + max_m)
    masked_m = np.asarray(mm, np.int32)
    ld = oracle.round_up(max_m, 4)
    q, sfo = q_sf_buffers((G, max_m, N), (G, N // QB, ld))
    dg.dg_fp8_grouped_masked_q(dev(a), dev(sfa), dev(b), dev(sfb), dev(masked_m), q, sfo)
    q_ref, sfo_ref = q_sf_sentinels((G, max_m, N), (G, N // QB, ld))
    oracle.grouped_masked_quant(a, sfa, b, sfb, masked_m, q_ref, sfo_ref)
    q, sfo = host(q), host(sfo)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sfo, sfo_ref)
    for e, v in enumerate(mm):
        assert np.all(q[e, v:] == Q_SENTINEL) and np.all(sfo[e, :, v:] == SF_SENTINEL)


def test_masked_q_cuda_graph_replay_follows_device_counts():
    G, max_m, N, K = 4, 256, 256, 512
    a, sfa, b, sfb = masked_case(G, max_m, N, K, seed=57)
    ta, tsa, tb, tsb = dev(a), dev(sfa), dev(b), dev(sfb)
    ld = oracle.round_up(max_m, 4)
    mm_dev = torch.zeros(G, dtype=torch.int32, device="cuda")
    q, sfo = q_sf_buffers((G, max_m, N), (G, N // QB, ld))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dg.dg_fp8_grouped_masked_q(ta, tsa, tb, tsb, mm_dev, q, sfo)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.dg_fp8_grouped_masked_q(ta, tsa, tb, tsb, mm_dev, q, sfo)
    for mm in ([5, 0, 256, 130], [256, 256, 1, 0]):
        masked_m = np.array(mm, np.int32)
        mm_dev.copy_(torch.from_numpy(masked_m))
        q.fill_(Q_SENTINEL)
        sfo.fill_(SF_SENTINEL)
        graph.replay()
        q_ref, sfo_ref = q_sf_sentinels((G, max_m, N), (G, N // QB, ld))
        oracle.grouped_masked_quant(a, sfa, b, sfb, masked_m, q_ref, sfo_ref)
        np.testing.assert_array_equal(host(q), q_ref)
        np.testing.assert_array_equal(host(sfo), sfo_ref)


def test_no_timeouts_were_flagged():
    assert not (dg.dg_read_device_status() & dg.DG_DEVFLAG_TIMEOUT)

"""GPU GEMMs (dense, contiguous, masked) against the oracle through the C ABI.

Exact-arithmetic inputs must match bit for bit; random inputs must meet the
stated tolerance.  Sizes span several tiles and a ragged tail in M and N."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg
import oracle
import workloads as wl
from helpers import QB, bf16_bits_to_f32, exact_dense, random_dense, tolerance_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    dg.load()
    dg.dg_read_device_status()


@pytest.fixture(params=[96, 128, 192, 256], ids=["bn96", "bn128", "bn192", "pair256"])
def tile_n(request, monkeypatch):
    """Runs the test with each compiled tile width (the plan's choice is
    pinned through DG_FORCE_BN): 96, 128 and 192 on one SM, and the 256 x 256
    tiles of the CTA-pair kernel (dense and contiguous layouts; the masked
    layout keeps the one-SM plan)."""
    monkeypatch.setenv("DG_FORCE_BN", str(request.param))
    return request.param


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_dense(a, sfa, b, sfb):
    d = torch.full((a.shape[0], b.shape[0]), float("nan"), dtype=torch.bfloat16, device="cuda")
    dg.dg_fp8_gemm_nt(dev(a), dev(sfa), dev(b), dev(sfb), d)
    return bits(d)


# ------------------------------------------------------------------ dense --
DENSE_SHAPES = [(128, 256, 512), (1, 128, 128), (129, 136, 384), (300, 392, 640), (513, 1024, 256),
                (256, 2112, 1024), (1100, 1288, 384), (4224, 1288, 256),
                # the narrowest N (one 16-byte row of D), N below one MMA width,
                # odd K-block counts against two-block stages, and a long K
                # whose fp32 accumulation is still exact on the exact inputs
                (3, 8, 256), (130, 24, 640), (257, 200, 1152), (65, 96, 18432)]


@pytest.mark.parametrize("M,N,K", DENSE_SHAPES)
def test_dense_exact_bit_identical(M, N, K, tile_n):
    a, sfa, b, sfb = exact_dense(M, N, K, seed=M * 3 + N + K)
    np.testing.assert_array_equal(gpu_dense(a, sfa, b, sfb), oracle.gemm_nt(a, sfa, b, sfb))


@pytest.mark.parametrize("M,N,K", DENSE_SHAPES)
def test_dense_random_tolerance(M, N, K, tile_n):
    a, sfa, b, sfb = random_dense(M, N, K, seed=M + 5 * N + K, outliers=True)
    ref = oracle.gemm_nt(a, sfa, b, sfb)
    tolerance_check(bf16_bits_to_f32(gpu_dense(a, sfa, b, sfb)), bf16_bits_to_f32(ref), f"dense {M}x{N}x{K}")


def test_dense_repeatable():
    a, sfa, b, sfb = random_dense(300, 512, 1024, seed=17)
    first = gpu_dense(a, sfa, b, sfb)
    for _ in range(3):
        np.testing.assert_array_equal(gpu_dense(a, sfa, b, sfb), first)


def test_dense_zero_rows_and_scale_doubling_exact():
    a, sfa, b, sfb = exact_dense(200, 256, 512, seed=5)
    base = gpu_dense(a, sfa, b, sfb)
    a2, sfa2 = a.copy(), sfa.copy()
    a2[3] = 0
    sfa2[:, 150] = 0
    sfa2[:, 151] *= 2
    out = gpu_dense(a2, sfa2, b, sfb)
    assert np.all(bf16_bits_to_f32(out[3]) == 0) and np.all(bf16_bits_to_f32(out[150]) == 0)
    np.testing.assert_array_equal(bf16_bits_to_f32(out[151]), 2 * bf16_bits_to_f32(base[151]))


def test_end_to_end_quantise_then_gemm():
    """fp32 activations -> GPU quantiser -> GPU GEMM, against the oracle's
    quantiser and GEMM on the same fp32 inputs."""
    x, w = wl.dense_inputs(256, 768, 1024, seed=21, outliers=True)
    b, sfb = oracle.quant_weight_128x128(w)
    qa, sfa_t = dg.dg_quant_act_1x128(dev(x))
    d = dg.dg_fp8_gemm_nt(qa, sfa_t, dev(b), dev(sfb))
    a_ref, sfa_ref = oracle.quant_act_1x128(x)
    np.testing.assert_array_equal(qa.cpu().numpy(), a_ref)
    tolerance_check(bf16_bits_to_f32(bits(d)), bf16_bits_to_f32(oracle.gemm_nt(a_ref, sfa_ref, b, sfb)), "e2e")


# ------------------------------------------------------------- contiguous --
def contiguous_case(G, tokens, N, K, seed, exact):
    counts, m_indices, seg = wl.contiguous_routing(G, tokens, seed)
    sum_M = len(m_indices)
    g = np.random.default_rng(seed + 1)
    if exact:
        a, sfa, _, _ = exact_dense(sum_M, 8, K, seed)
        bs = [exact_dense(8, N, K, seed + 10 + e) for e in range(G)]
        b = np.stack([x[2] for x in bs])
        sfb = np.stack([x[3] for x in bs])
    else:
        x = wl.normal_matrix(g, (sum_M, K), outliers=True)
        w = wl.normal_matrix(g, (G, N, K))
        a, sfa = oracle.quant_act_1x128(x)
        b, sfb = oracle.quant_weight_128x128(w)
    return a, sfa, b, sfb, m_indices


def gpu_contiguous(a, sfa, b, sfb, m_indices):
    d = sentinel_tensor((a.shape[0], b.shape[1]))
    dg.dg_fp8_grouped_contiguous(dev(a), dev(sfa), dev(b), dev(sfb), dev(m_indices), d.view(torch.bfloat16))
    return bits(d.view(torch.bfloat16))


@pytest.mark.parametrize("G,tokens,N,K", [(4, 700, 256, 512), (8, 1500, 392, 384), (3, 129, 128, 128), (2, 100, 8, 640)])
def test_contiguous_exact_bit_identical(G, tokens, N, K, tile_n):
    a, sfa, b, sfb, mi = contiguous_case(G, tokens, N, K, seed=G + tokens, exact=True)
    ref = np.full((a.shape[0], N), wl.SENTINEL_BF16, dtype=np.uint16)
    ref = oracle.grouped_contiguous(a, sfa, b, sfb, mi, d=ref)
    np.testing.assert_array_equal(gpu_contiguous(a, sfa, b, sfb, mi), ref)


@pytest.mark.parametrize("G,tokens,N,K", [(8, 2000, 512, 1024), (2, 300, 264, 256)])
def test_contiguous_random_tolerance(G, tokens, N, K, tile_n):
    a, sfa, b, sfb, mi = contiguous_case(G, tokens, N, K, seed=7 * G + tokens, exact=False)
    out = gpu_contiguous(a, sfa, b, sfb, mi)
    ref = oracle.grouped_contiguous(a, sfa, b, sfb, mi)
    valid = mi >= 0
    tolerance_check(bf16_bits_to_f32(out[valid]), bf16_bits_to_f32(ref[valid]), "contiguous")
    assert np.all(out[~valid] == wl.SENTINEL_BF16)


@pytest.mark.parametrize("force", ["", "256"], ids=["auto", "pair256"])
def test_contiguous_bad_expert_is_flagged(force, monkeypatch):
    monkeypatch.setenv("DG_FORCE_BN", force)
    a, sfa, b, sfb, mi = contiguous_case(2, 200, 128, 128, seed=3, exact=True)
    mi = mi.copy()
    mi[:128] = 5            # expert 5 does not exist (G = 2)
    out = gpu_contiguous(a, sfa, b, sfb, mi)
    flags = dg.dg_read_device_status()
    assert flags & dg.DG_DEVFLAG_BAD_EXPERT
    assert np.all(out[:128] == wl.SENTINEL_BF16)
    ref = oracle.grouped_contiguous(a, sfa, b, sfb, mi, d=np.full_like(out, wl.SENTINEL_BF16))
    np.testing.assert_array_equal(out, ref)


@pytest.mark.parametrize("force", ["", "256"], ids=["auto", "pair256"])
def test_contiguous_mixed_block_is_flagged_and_skipped(force, monkeypatch):
    """A 128-row block whose rows name two experts: rows that disagree with
    the block's first row are not written and the device flags the block."""
    monkeypatch.setenv("DG_FORCE_BN", force)
    a, sfa, b, sfb, mi = contiguous_case(3, 500, 256, 256, seed=8, exact=True)
    mi = mi.copy()
    first = int(np.flatnonzero(mi == 1)[0])
    mi[first + 5] = 2                        # one row of expert 2 inside expert 1's block
    out = gpu_contiguous(a, sfa, b, sfb, mi)
    assert dg.dg_read_device_status() & dg.DG_DEVFLAG_MIXED_BLOCK
    assert np.all(out[first + 5] == wl.SENTINEL_BF16)
    keep = mi.copy()
    keep[first + 5] = -1                     # the oracle's view: that row is left alone
    ref = oracle.grouped_contiguous(a, sfa, b, sfb, keep, d=np.full_like(out, wl.SENTINEL_BF16))
    np.testing.assert_array_equal(out, ref)


@pytest.mark.parametrize("G,tokens,N,K", [(5, 1700, 264, 384), (1, 300, 512, 256), (6, 2600, 520, 128)])
def test_contiguous_pair_rows_odd_blocks_and_padding(G, tokens, N, K, monkeypatch):
    """CTA-pair tiles on experts with odd numbers of 128-row blocks (the last
    block of such an expert is computed alone), N not a multiple of 256 and
    an odd number of K blocks: exact inputs, bit for bit."""
    monkeypatch.setenv("DG_FORCE_BN", "256")
    a, sfa, b, sfb, mi = contiguous_case(G, tokens, N, K, seed=G * 7 + N, exact=True)
    ref = np.full((a.shape[0], N), wl.SENTINEL_BF16, dtype=np.uint16)
    ref = oracle.grouped_contiguous(a, sfa, b, sfb, mi, d=ref)
    np.testing.assert_array_equal(gpu_contiguous(a, sfa, b, sfb, mi), ref)


# ----------------------------------------------------------------- masked --
def masked_case(G, max_m, N, K, masked_m, seed, exact):
    g = np.random.default_rng(seed)
    ld = oracle.round_up(max_m, 4)
    a = np.empty((G, max_m, K), np.uint8)
    sfa = np.zeros((G, K // QB, ld), np.float32)
    b = np.empty((G, N, K), np.uint8)
    sfb = np.empty((G, -(-N // QB), K // QB), np.float32)
    for e in range(G):
        if exact:
            a[e], sfa[e], b[e], sfb[e] = exact_dense(max_m, N, K, seed + e)
        else:
            x = wl.normal_matrix(g, (max_m, K), outliers=True)
            w = wl.normal_matrix(g, (N, K))
            a[e], sfa[e] = oracle.quant_act_1x128(x)
            b[e], sfb[e] = oracle.quant_weight_128x128(w)
    return a, sfa, b, sfb, np.asarray(masked_m, np.int32)


def sentinel_tensor(shape):
    v = wl.SENTINEL_BF16 if wl.SENTINEL_BF16 < 32768 else wl.SENTINEL_BF16 - 65536
    return torch.full(shape, v, dtype=torch.int16, device="cuda")


def gpu_masked(a, sfa, b, sfb, masked_m):
    d = sentinel_tensor((a.shape[0], a.shape[1], b.shape[1]))
    dg.dg_fp8_grouped_masked(dev(a), dev(sfa), dev(b), dev(sfb), dev(masked_m), d.view(torch.bfloat16))
    return bits(d.view(torch.bfloat16))


@pytest.mark.parametrize("G,max_m,N,K,mm", [
    (4, 256, 256, 512, [0, 1, 255, 256]),
    (3, 200, 392, 384, [200, 129, 128]),
    (2, 64, 128, 128, [64, 3]),
    (5, 130, 8, 640, [130, 0, 7, 129, 1]),
])
def test_masked_exact_bit_identical(G, max_m, N, K, mm, tile_n):
    a, sfa, b, sfb, masked_m = masked_case(G, max_m, N, K, mm, seed=G * 11 + max_m, exact=True)
    ref = oracle.grouped_masked(a, sfa, b, sfb, masked_m,
                                d=np.full((G, max_m, N), wl.SENTINEL_BF16, np.uint16))
    np.testing.assert_array_equal(gpu_masked(a, sfa, b, sfb, masked_m), ref)


def test_masked_random_tolerance(tile_n):
    G, max_m, N, K = 6, 256, 512, 1024
    mm = wl.masked_counts(G, max_m, seed=12)
    a, sfa, b, sfb, masked_m = masked_case(G, max_m, N, K, mm, seed=12, exact=False)
    out = gpu_masked(a, sfa, b, sfb, masked_m)
    ref = oracle.grouped_masked(a, sfa, b, sfb, masked_m,
                                d=np.full((G, max_m, N), wl.SENTINEL_BF16, np.uint16))
    for e in range(G):
        v = int(masked_m[e])
        if v:
            tolerance_check(bf16_bits_to_f32(out[e, :v]), bf16_bits_to_f32(ref[e, :v]), f"masked expert {e}")
        assert np.all(out[e, v:] == wl.SENTINEL_BF16)


def test_masked_expected_m_changes_the_plan_not_the_result():
    """expected_m only picks the tile width: a hint that narrows the tiles
    gives the same bits as no hint, on exact inputs equal to the oracle."""
    G, max_m, N, K = 4, 512, 4096, 512
    mm = [40, 0, 512, 17]
    a, sfa, b, sfb, masked_m = masked_case(G, max_m, N, K, mm, seed=41, exact=True)
    assert dg.dg_query_plan(dg.DG_LAYOUT_MASKED, max_m, N, K, G, expected_m=40)["block_n"] != \
        dg.dg_query_plan(dg.DG_LAYOUT_MASKED, max_m, N, K, G)["block_n"]
    outs = []
    for hint in (0, 40):
        d = sentinel_tensor((G, max_m, N))
        dg.dg_fp8_grouped_masked(dev(a), dev(sfa), dev(b), dev(sfb), dev(masked_m), d.view(torch.bfloat16),
                                 expected_m=hint)
        outs.append(bits(d.view(torch.bfloat16)))
    np.testing.assert_array_equal(outs[0], outs[1])
    ref = oracle.grouped_masked(a, sfa, b, sfb, masked_m, d=np.full(outs[0].shape, wl.SENTINEL_BF16, np.uint16))
    np.testing.assert_array_equal(outs[1], ref)


def test_masked_clamps_and_flags_bad_counts():
    a, sfa, b, sfb, _ = masked_case(3, 64, 128, 128, [0, 0, 0], seed=4, exact=True)
    masked_m = np.array([-5, 70, 10], np.int32)
    out = gpu_masked(a, sfa, b, sfb, masked_m)
    assert dg.dg_read_device_status() & dg.DG_DEVFLAG_MASKED_M_CLAMPED
    ref = oracle.grouped_masked(a, sfa, b, sfb, masked_m, d=np.full(out.shape, wl.SENTINEL_BF16, np.uint16))
    np.testing.assert_array_equal(out, ref)


def test_masked_cuda_graph_replay_follows_device_counts(tile_n):
    G, max_m, N, K = 4, 256, 256, 512
    a, sfa, b, sfb, _ = masked_case(G, max_m, N, K, [0] * G, seed=31, exact=True)
    ta, tsa, tb, tsb = dev(a), dev(sfa), dev(b), dev(sfb)
    mm_dev = torch.zeros(G, dtype=torch.int32, device="cuda")
    d = sentinel_tensor((G, max_m, N))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dg.dg_fp8_grouped_masked(ta, tsa, tb, tsb, mm_dev, d.view(torch.bfloat16))   # warm-up, outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.dg_fp8_grouped_masked(ta, tsa, tb, tsb, mm_dev, d.view(torch.bfloat16))
    for mm in ([5, 0, 256, 130], [256, 256, 1, 0], [0, 0, 0, 0]):
        masked_m = np.array(mm, np.int32)
        mm_dev.copy_(torch.from_numpy(masked_m))
        d.copy_(sentinel_tensor(d.shape))
        graph.replay()
        out = bits(d.view(torch.bfloat16))
        ref = oracle.grouped_masked(a, sfa, b, sfb, masked_m, d=np.full(out.shape, wl.SENTINEL_BF16, np.uint16))
        np.testing.assert_array_equal(out, ref)


def test_no_timeouts_were_flagged():
    assert not (dg.dg_read_device_status() & dg.DG_DEVFLAG_TIMEOUT)

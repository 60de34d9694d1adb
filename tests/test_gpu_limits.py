"""GPU GEMMs at the library's structural limits, bit for bit against the oracle.

Two limits come from what the kernels keep in shared memory:
- the CTA-pair kernel builds the contiguous layout's list of row pairs on the
  device, for at most 1024 blocks of 128 rows (131072 rows);
- the masked kernel builds its per-expert tile prefix on the device, for at
  most 1024 experts.
Both tests run exactly at the limit, in the plan the library picks, on
exact-arithmetic operands (values in {-2..2}, scales 2^[-3,0]), so every
result is unique."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg
import oracle
import workloads as wl
from helpers import QB, int_codes

pytestmark = pytest.mark.gpu

SENT = wl.SENTINEL_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    dg.load()
    dg.dg_read_device_status()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def codes(g: np.random.Generator, shape) -> np.ndarray:
    """E4M3 codes of values drawn from {-2..2}, built without int64
    temporaries (the contiguous operand has 268M entries)."""
    lut = int_codes(np.arange(-2, 3, dtype=np.int8))
    idx = g.integers(0, 5, shape, dtype=np.uint8)
    out = np.full(shape, lut[0], dtype=np.uint8)
    for k in range(1, 5):
        out[idx == k] = lut[k]
    return out


def test_contiguous_pair_list_at_capacity():
    """1024 blocks of 128 rows over 8 experts: odd and even block counts, and
    padding rows (-1) at the end of some experts' last blocks."""
    blocks = [131, 127, 128, 129, 125, 128, 127, 129]
    pad = [0, 37, 0, 100, 5, 0, 64, 1]
    assert sum(blocks) == 1024
    G, N, K = len(blocks), 256, 2048
    m_indices = np.concatenate([np.r_[np.full(nb * 128 - p, e, np.int32), np.full(p, -1, np.int32)]
                                for e, (nb, p) in enumerate(zip(blocks, pad))])
    sum_M = len(m_indices)
    assert sum_M == 1024 * 128
    plan = dg.dg_query_plan(dg.DG_LAYOUT_CONTIGUOUS, sum_M, N, K, G)
    assert plan["block_m"] == 256, plan          # the pair kernel, at its list's capacity

    g = np.random.default_rng(1024)
    a = codes(g, (sum_M, K))
    b = codes(g, (G, N, K))
    sfa = wl.exact_scales(g, (K // QB, sum_M))
    sfb = wl.exact_scales(g, (G, -(-N // QB), K // QB))
    d = torch.full((sum_M, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_fp8_grouped_contiguous(dev(a), dev(sfa), dev(b), dev(sfb), dev(m_indices), d.view(torch.bfloat16))
    out = bits(d.view(torch.bfloat16))
    assert dg.dg_read_device_status() == 0

    assert np.all(out[m_indices < 0] == SENT), "a padding row was written"
    starts = np.cumsum([0] + [nb * 128 for nb in blocks])[:-1]
    must = []
    for e, (s0, nb, p) in enumerate(zip(starts, blocks, pad)):
        last = int(s0 + nb * 128 - p - 1)
        must += [int(s0), int(s0) + 127, int(s0) + 128, last, int(s0 + nb * 128 - 128)]
    rows = wl.sample_rows(sum_M, 40, 1024, must=must)
    rows = rows[m_indices[rows] >= 0]
    ref = oracle.grouped_contiguous(a, sfa, b, sfb, m_indices, rows=rows, d=np.full((sum_M, N), SENT, np.uint16))
    np.testing.assert_array_equal(out[rows], ref[rows])


@pytest.mark.parametrize("expected_m", [0, 8])
def test_masked_at_expert_capacity(expected_m):
    """1024 experts (the limit of the device-side tile prefix), counts from 0
    to max_m, every row of the output compared."""
    G, max_m, N, K = 1024, 16, 128, 256
    g = np.random.default_rng(2048)
    masked_m = g.integers(0, max_m + 1, G).astype(np.int32)
    masked_m[[0, 1, 512, G - 1]] = [0, max_m, 1, max_m]
    ld = oracle.round_up(max_m, 4)
    a = codes(g, (G, max_m, K))
    b = codes(g, (G, N, K))
    sfa = np.zeros((G, K // QB, ld), np.float32)
    sfa[:, :, :max_m] = wl.exact_scales(g, (G, K // QB, max_m))
    sfb = wl.exact_scales(g, (G, -(-N // QB), K // QB))
    d = torch.full((G, max_m, N), SENT, dtype=torch.int16, device="cuda")
    dg.dg_fp8_grouped_masked(dev(a), dev(sfa), dev(b), dev(sfb), dev(masked_m), d.view(torch.bfloat16),
                             expected_m=expected_m)
    out = bits(d.view(torch.bfloat16))
    assert dg.dg_read_device_status() == 0
    ref = oracle.grouped_masked(a, sfa, b, sfb, masked_m, d=np.full((G, max_m, N), SENT, np.uint16))
    np.testing.assert_array_equal(out, ref)


# Operands with more than 2^31 elements: every element and byte offset in the
# kernels is 64-bit, which these tests check on the rows whose elements start
# past 2^31 (a 32-bit offset would wrap there).  The operands are generated on
# the device; the oracle gets only the sampled rows.
def rows_around(r0: int, M: int, seed: int) -> np.ndarray:
    return wl.sample_rows(M, 12, seed, must=[0, r0 - 1, r0, r0 + 1, M - 2, M - 1])


def test_quantiser_past_2g_elements():
    K = 8192
    r0 = (1 << 31) // K                       # the first row whose elements start at 2^31
    M = r0 + 64
    gen = torch.Generator(device="cuda").manual_seed(31)
    x = torch.randn((M, K), generator=gen, device="cuda", dtype=torch.float32)
    q, sfa = dg.dg_quant_act_1x128(x)
    torch.cuda.synchronize()
    rows = rows_around(r0, M, 31)
    idx = torch.from_numpy(rows).cuda()
    x_rows = x.index_select(0, idx).cpu().numpy()
    q_rows = q.index_select(0, idx).cpu().numpy()
    s_rows = sfa[:, idx].cpu().numpy()
    del x, q, sfa
    torch.cuda.empty_cache()
    ref_q, ref_s = oracle.quant_act_1x128(x_rows)
    np.testing.assert_array_equal(q_rows, ref_q)
    np.testing.assert_array_equal(s_rows, ref_s[:, :len(rows)])


def test_dense_gemm_past_2g_operand():
    N, K = 256, 7296
    r0 = -(-(1 << 31) // K)                   # the first row whose elements start past 2^31
    M = (r0 // 256 + 1) * 256                 # whole 256-row pair tiles
    assert M * K > (1 << 31)
    gen = torch.Generator(device="cuda").manual_seed(32)
    # values +1 / -1 (E4M3 0x38 / 0xB8) and power-of-two scales: exact sums
    a = torch.randint(0, 2, (M, K), generator=gen, device="cuda", dtype=torch.uint8).mul_(128).add_(0x38)
    b = torch.randint(0, 2, (N, K), generator=gen, device="cuda", dtype=torch.uint8).mul_(128).add_(0x38)
    g = np.random.default_rng(32)
    sfa = wl.exact_scales(g, (K // QB, M))
    sfb = wl.exact_scales(g, (-(-N // QB), K // QB))
    d = dg.dg_fp8_gemm_nt(a, dev(sfa), b, dev(sfb))
    out = bits(d)
    assert dg.dg_read_device_status() == 0
    rows = rows_around(r0, M, 32)
    a_rows = a.index_select(0, torch.from_numpy(rows).cuda()).cpu().numpy()
    b_h = b.cpu().numpy()
    del a, d
    torch.cuda.empty_cache()
    sfa_rows = np.zeros((K // QB, oracle.round_up(len(rows), 4)), np.float32)
    sfa_rows[:, :len(rows)] = sfa[:, rows]
    ref = oracle.gemm_nt(a_rows, sfa_rows, b_h, sfb)
    np.testing.assert_array_equal(out[rows], ref)

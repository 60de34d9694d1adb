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

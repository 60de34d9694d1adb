"""GPU quantisers against the oracle, bit for bit (every step is IEEE-exact:
max, fp32 division, round-to-nearest-even with saturation)."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    dg.load()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_act(x: np.ndarray):
    xt = dev(x)
    if x.dtype == np.uint16:
        xt = xt.view(torch.bfloat16)
    q, sfa = dg.dg_quant_act_1x128(xt)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sfa.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 128), (7, 256), (129, 512), (256, 2048), (1000, 7168)])
def test_quant_act_bit_exact(M, K):
    g = np.random.default_rng(M + K)
    x = wl.normal_matrix(g, (M, K), outliers=True)
    x *= np.ldexp(np.float32(1), g.integers(-8, 8, (M, 1))).astype(np.float32)
    q, sfa = run_act(x)
    q_ref, sfa_ref = oracle.quant_act_1x128(x)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sfa[:, :M], sfa_ref[:, :M])


def test_quant_act_bf16_bit_exact():
    g = np.random.default_rng(3)
    xf = wl.normal_matrix(g, (130, 1024), outliers=True)
    bits = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, sfa = run_act(bits)
    q_ref, sfa_ref = oracle.quant_act_1x128(bits)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sfa[:, :130], sfa_ref[:, :130])


def test_quant_act_rounding_ties_and_specials():
    """Groups whose scale is exactly 1 (amax = 448) so that x/s = x: every
    E4M3 midpoint, its fp32 neighbours, subnormals, zeros and -0."""
    t = oracle.e4m3_decode_table()[:0x7F]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                           t.astype(np.float32), np.array([0.0, -0.0, 2.0 ** -10, 2.0 ** -11], np.float32)])
    vals = np.concatenate([vals, -vals])
    per = 127
    groups = -(-len(vals) // per)
    x = np.zeros((groups, 128), dtype=np.float32)
    for i in range(groups):
        chunk = vals[i * per:(i + 1) * per]
        x[i, :len(chunk)] = chunk
        x[i, 127] = 448.0
    x = np.ascontiguousarray(x)
    q, sfa = run_act(x)
    q_ref, sfa_ref = oracle.quant_act_1x128(x)
    assert np.all(sfa_ref[0, :groups] == 1.0)
    np.testing.assert_array_equal(q, q_ref)
    # all-zero and tiny groups: scale from the 1e-4 floor
    z = np.zeros((3, 256), dtype=np.float32)
    z[1, 5] = 1e-7
    q, sfa = run_act(z)
    q_ref, sfa_ref = oracle.quant_act_1x128(z)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sfa[:, :3], sfa_ref[:, :3])


@pytest.mark.parametrize("G,N,K", [(1, 128, 128), (1, 2112, 512), (3, 200, 256)])
def test_quant_weight_bit_exact(G, N, K):
    g = np.random.default_rng(G * N + K)
    w = wl.normal_matrix(g, (G, N, K))
    w *= np.ldexp(np.float32(1), g.integers(-5, 5, (G, N, 1))).astype(np.float32)
    q, sfb = dg.dg_quant_weight_128x128(dev(w))
    torch.cuda.synchronize()
    q_ref, sfb_ref = oracle.quant_weight_128x128(w)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(sfb.cpu().numpy(), sfb_ref)

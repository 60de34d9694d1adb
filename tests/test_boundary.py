"""The C-ABI boundary without a GPU: the library builds for sm_103a, loads,
exports every entry point include/dg.h declares, rejects bad arguments with
the documented codes before touching the device, and plans tiles with the
arithmetic the pages give."""
import ctypes
import os
import re

import pytest

import moe_grouped_gemm_x128_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dg.build()
    return dg.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dg.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dg_\w+)\s*\(", text, flags=re.M)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(dg.EXPORTED)


def test_library_exports_every_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        s = dg.status_string(code)
        assert isinstance(s, str) and s
    assert dg.status_string(99) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def call(lib, name, *args):
    return getattr(lib, name)(*args)


def test_quant_validation(lib):
    assert call(lib, "dg_quant_act_1x128", None, 0, FAKE, FAKE, 4, 128, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_quant_act_1x128", FAKE, 7, FAKE, FAKE, 4, 128, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_quant_act_1x128", FAKE, 0, FAKE, FAKE, 0, 128, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_quant_act_1x128", FAKE, 0, FAKE, FAKE, 4, 100, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_quant_act_1x128", FAKE + 4, 0, FAKE, FAKE, 4, 128, None) == dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_quant_weight_128x128", FAKE, FAKE, None, 1, 128, 128, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_quant_weight_128x128", FAKE, FAKE, FAKE, 1, 128, 130, None) == dg.DG_ERR_UNSUPPORTED_SHAPE


def test_gemm_validation(lib):
    F = FAKE
    assert call(lib, "dg_fp8_gemm_nt", F, F, F, F, None, 128, 256, 512, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_fp8_gemm_nt", F, F, F, F, F, -1, 256, 512, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_fp8_gemm_nt", F, F, F, F, F, 128, 256, 500, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_gemm_nt", F, F, F, F, F, 128, 252, 512, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_gemm_nt", F, F + 8, F, F, F, 128, 256, 512, None) == dg.DG_ERR_MISALIGNED
    # contiguous: sum_M must be a multiple of 128, G > 0, m_indices non-null
    assert call(lib, "dg_fp8_grouped_contiguous", F, F, F, F, F, F, 200, 256, 512, 2, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_grouped_contiguous", F, F, F, F, F, None, 256, 256, 512, 2, None) == \
        dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_fp8_grouped_contiguous", F, F, F, F, F, F, 256, 256, 512, 0, None) == \
        dg.DG_ERR_INVALID_ARG
    # masked: G limit and alignment of masked_m
    assert call(lib, "dg_fp8_grouped_masked", F, F, F, F, F, F, 5000, 256, 256, 512, 0, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_grouped_masked", F, F, F, F, F, F, 1025, 256, 256, 512, 0, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE    # one expert past the device-side tile prefix
    assert call(lib, "dg_fp8_grouped_masked", F, F, F, F, F, F + 4, 4, 256, 256, 512, 0, None) == \
        dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_fp8_grouped_masked", F, F, F, F, F, F, 4, 0, 256, 512, 0, None) == dg.DG_ERR_INVALID_ARG


def test_requant_gemm_validation(lib):
    F = FAKE
    # q and sfo must both be given, N a multiple of 128, both 16-byte aligned
    assert call(lib, "dg_fp8_gemm_nt_q", F, F, F, F, F, None, 128, 256, 512, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_fp8_gemm_nt_q", F, F, F, F, None, F, 128, 256, 512, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_fp8_gemm_nt_q", F, F, F, F, F, F, 128, 192, 512, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_gemm_nt_q", F, F, F, F, F, F + 4, 128, 256, 512, None) == dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_fp8_gemm_nt_q", F, F, F, F, F + 8, F, 128, 256, 512, None) == dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_fp8_grouped_contiguous_q", F, F, F, F, F, F, F, 200, 256, 512, 2, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_grouped_contiguous_q", F, F, F, F, F, F, None, 256, 256, 512, 2, None) == \
        dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_fp8_grouped_contiguous_q", F, F, F, F, F, F, F, 256, 320, 512, 2, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_grouped_masked_q", F, F, F, F, F, F, F, 5000, 256, 256, 512, 0, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_fp8_grouped_masked_q", F, F, F, F, F, F, F + 4, 4, 256, 256, 512, 0, None) == \
        dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_fp8_grouped_masked_q", F, F, F, F, F, F, F, 4, 256, 384 + 64, 512, 0, None) == \
        dg.DG_ERR_UNSUPPORTED_SHAPE


def test_bf16_and_mx_validation(lib):
    F = FAKE
    assert call(lib, "dg_bf16_gemm_nt", None, F, F, 128, 256, 64, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_bf16_gemm_nt", F, F, F, 128, 256, 96, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_bf16_gemm_nt", F, F, F, 128, 252, 64, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_bf16_gemm_nt", F + 2, F, F, 128, 256, 64, None) == dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_quant_mx_1x32", F, F, None, 4, 128, None) == dg.DG_ERR_INVALID_ARG
    assert call(lib, "dg_quant_mx_1x32", F, F, F, 4, 96, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_mx_gemm_nt", F, F, F, F, F, 128, 256, 192, None) == dg.DG_ERR_UNSUPPORTED_SHAPE
    assert call(lib, "dg_mx_gemm_nt", F, F + 4, F, F, F, 128, 256, 256, None) == dg.DG_ERR_MISALIGNED
    assert call(lib, "dg_mx_gemm_nt", F, F, F, F, F, 0, 256, 256, None) == dg.DG_ERR_INVALID_ARG


def test_read_status_validation(lib):
    assert lib.dg_read_device_status(None, None) == dg.DG_ERR_INVALID_ARG


def test_selftest_limit_validation(lib):
    # the limit is checked before anything touches the device
    assert lib.dg_selftest_wait_timeout(999, None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_selftest_wait_timeout(4000000001, None) == dg.DG_ERR_INVALID_ARG


def golden_block_counts():
    """The pages' worked example (tests/golden/block_counts_m256_n7168.txt)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "block_counts_m256_n7168.txt")
    rows = []
    with open(path) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(int(v) for v in line.split()))
    return rows


def test_plan_tile_arithmetic_of_the_pages():
    # M=256, N=7168 ("DeepGEMM：一款支持FP8通用矩阵乘法(GEMM)的开源库", 非标准块大小支持):
    # 128-wide blocks keep 112 units busy, 112-wide ones 128; the plan's tile
    # count for a width is the same arithmetic (one tile per unit).
    rows = golden_block_counts()
    assert len(rows) == 2
    for M, N, bm, bn, busy in rows:
        assert -(-M // bm) * -(-N // bn) == busy
    # With 132 SMs the plan keeps 128-wide tiles (112 tiles, one wave) ...
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 256, 7168, 2048, 1, num_sms=132)
    assert (p["block_m"], p["block_n"], p["num_tiles"], p["grid"]) == (128, 128, 112, 112)
    # ... and with 152 SMs it narrows them to 96 so that 150 of 152 SMs work.
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 256, 7168, 2048, 1, num_sms=152)
    assert (p["block_n"], p["num_tiles"], p["grid"]) == (96, 150, 150)


def test_plan_width_override(monkeypatch):
    for bn in (96, 128, 192):
        monkeypatch.setenv("DG_FORCE_BN", str(bn))
        p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 7168, 2048, 1, num_sms=152)
        assert p["block_m"] == 128 and p["block_n"] == bn and p["num_tiles"] == 32 * -(-7168 // bn)
    # 256: the CTA-pair kernel, 256 x 256 tiles on two SMs, an even grid
    monkeypatch.setenv("DG_FORCE_BN", "256")
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 300, 520, 256, 1, num_sms=152)
    assert (p["block_m"], p["block_n"], p["num_tiles"], p["grid"]) == (256, 256, 2 * 3, 12)
    # forced: short K too
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 24576, 1536, 1, num_sms=152)
    assert p["block_m"] == 256
    # the masked layout has no pair kernel: the one-SM plan stays
    p = dg.dg_query_plan(dg.DG_LAYOUT_MASKED, 256, 7168, 2048, 16, num_sms=152)
    assert p["block_m"] == 128
    monkeypatch.setenv("DG_FORCE_BN", "100")   # not a compiled width: ignored
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 7168, 2048, 1, num_sms=152)
    assert (p["block_m"], p["block_n"]) == (256, 256)


def test_plan_picks_pair_tiles_for_a_full_wave_of_pairs():
    # a full wave of 256 x 256 pair tiles (76 pairs on 152 SMs) takes the
    # CTA-pair kernel; fewer keep the one-SM tiles (e.g. the skinny M=256 case)
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 7168, 18432, 1, num_sms=152)
    assert (p["block_m"], p["block_n"], p["num_tiles"], p["grid"]) == (256, 256, 16 * 28, 152)
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 256, 7168, 2048, 1, num_sms=152)
    assert p["block_m"] == 128
    # short K (fewer than 16 K blocks): the one-SM tiles amortise better
    p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 24576, 1536, 1, num_sms=152)
    assert (p["block_m"], p["block_n"]) == (128, 192)
    p = dg.dg_query_plan(dg.DG_LAYOUT_CONTIGUOUS, 33152, 4096, 7168, 8, num_sms=152)
    assert (p["block_m"], p["block_n"], p["grid"]) == (256, 256, 152)
    # contiguous pair rows live in shared memory: at most 1024 blocks of 128 rows
    p = dg.dg_query_plan(dg.DG_LAYOUT_CONTIGUOUS, 1025 * 128, 4096, 7168, 8, num_sms=152)
    assert p["block_m"] == 128
    p = dg.dg_query_plan(dg.DG_LAYOUT_CONTIGUOUS, 1024 * 128, 4096, 7168, 8, num_sms=152)
    assert p["block_m"] == 256


def test_masked_plan_follows_expected_m():
    # 4 experts with 512-row buffers, N = 4096: every buffer full makes 16
    # m-blocks, 352 tiles of 128 x 192; a hint of 40 rows per expert leaves 4
    # m-blocks, 88 such tiles on 152 SMs, so the plan narrows them to 128
    # (128 tiles, one wave)
    full = dg.dg_query_plan(dg.DG_LAYOUT_MASKED, 512, 4096, 2048, 4, num_sms=152)
    assert full["block_n"] == 192
    hint = dg.dg_query_plan(dg.DG_LAYOUT_MASKED, 512, 4096, 2048, 4, num_sms=152, expected_m=40)
    assert hint["block_n"] == 128
    # the grid and the tile bound stay those of full buffers (the kernel reads
    # masked_m on the device), and the hint never exceeds max_m
    assert hint["grid"] == 152 and hint["num_tiles"] == 4 * 4 * 32
    assert dg.dg_query_plan(dg.DG_LAYOUT_MASKED, 512, 4096, 2048, 4, num_sms=152, expected_m=5000) == full
    # the other layouts ignore the hint
    assert dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 7168, 2048, 1, num_sms=152, expected_m=7) == \
        dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 4096, 7168, 2048, 1, num_sms=152)
    with pytest.raises(dg.DgError):
        dg.dg_query_plan(dg.DG_LAYOUT_MASKED, 512, 7168, 2048, 4, num_sms=152, expected_m=-1)


def test_plan_shapes():
    for (M, N, K) in [(128, 256, 512), (4096, 7168, 18432), (4096, 24576, 1536), (4096, 2112, 7168), (1, 8, 128)]:
        p = dg.dg_query_plan(dg.DG_LAYOUT_DENSE, M, N, K, 1, num_sms=152)
        tiles = -(-M // p["block_m"]) * -(-N // p["block_n"])
        assert p["num_tiles"] == tiles
        if p["block_m"] == 256:
            assert p["grid"] == 2 * min(tiles, 76)
        else:
            assert p["grid"] == min(tiles, 152)
        assert p["smem_bytes"] <= 232448
    # masked: fixed grid = SM count (the real tile count lives on the device)
    p = dg.dg_query_plan(dg.DG_LAYOUT_MASKED, 256, 7168, 2048, 16, num_sms=152)
    assert p["grid"] == 152
    assert p["num_tiles"] == 16 * 2 * -(-7168 // p["block_n"])
    with pytest.raises(dg.DgError):
        dg.dg_query_plan(dg.DG_LAYOUT_DENSE, 128, 256, 100, 1, num_sms=152)

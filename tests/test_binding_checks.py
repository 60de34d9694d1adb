"""The binding's argument checks, on the CPU.

The C entry points take bare pointers, so the Python binding checks every
tensor's shape, dtype, layout and device before calling them.  These tests
run each binding with CPU tensors: once with the device check and the
library replaced by stand-ins, on every call pattern the benchmark, the smoke
check and the GPU tests use (all must pass the checks), and once as is, on
wrong arguments (each must raise before any CUDA call)."""
import pytest
import torch

import moe_grouped_gemm_x128_gb300 as dg

U8, F32, BF16, I32 = torch.uint8, torch.float32, torch.bfloat16, torch.int32


class _Calls:
    """Stands in for libdg.so: records the entry points called, returns DG_OK."""

    def __init__(self):
        self.names = []

    def __getattr__(self, name):
        def call(*args):
            self.names.append(name)
            return dg.DG_OK
        return call


@pytest.fixture
def fake(monkeypatch):
    lib = _Calls()
    monkeypatch.setattr(dg, "load", lambda: lib)
    monkeypatch.setattr(dg, "_on_device", lambda *named: None)
    monkeypatch.setattr(dg, "_stream", lambda s: 0)
    return lib


def z(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


def dense(M, N, K):
    return z((M, K), U8), z((K // 128, dg.round_up(M, 4)), F32), z((N, K), U8), z((-(-N // 128), K // 128), F32)


def test_call_patterns_pass(fake):
    # quantisers: fp32 and bf16 activations, given or allocated outputs; 2-D and 3-D weights
    for M, K in [(256, 2048), (1, 128), (130, 640)]:
        dg.dg_quant_act_1x128(z((M, K), F32))
        dg.dg_quant_act_1x128(z((M, K), BF16))
        dg.dg_quant_act_1x128(z((M, K), F32), z((M, K), U8), z((K // 128, dg.round_up(M, 4)), F32))
    q, sfb = dg.dg_quant_weight_128x128(z((7168, 2048), F32))
    assert q.shape == (7168, 2048) and sfb.shape == (56, 16)
    q, sfb = dg.dg_quant_weight_128x128(z((3, 200, 256), F32))
    assert q.shape == (3, 200, 256) and sfb.shape == (3, 2, 2)
    q2, s2 = dg.dg_quant_weight_128x128(z((200, 256), F32), z((200, 256), U8), z((2, 2), F32))
    assert q2.shape == (200, 256) and s2.shape == (2, 2)
    # dense GEMM, as the benchmark and the tests call it (uint8 or float8 operands)
    for M, N, K in [(256, 7168, 2048), (3, 8, 256), (129, 136, 384), (65, 96, 18432)]:
        a, sfa, b, sfb = dense(M, N, K)
        dg.dg_fp8_gemm_nt(a, sfa, b, sfb)
        dg.dg_fp8_gemm_nt(a, sfa, b, sfb, z((M, N), BF16))
        dg.dg_fp8_gemm_nt(a.view(torch.float8_e4m3fn), sfa, b.view(torch.float8_e4m3fn), sfb)
    # contiguous: sum_M a multiple of 128, sfa [K/128, sum_M]
    G, sum_M, N, K = 4, 1024, 392, 384
    args = (z((sum_M, K), U8), z((K // 128, sum_M), F32), z((G, N, K), U8), z((G, 4, K // 128), F32),
            z((sum_M,), I32))
    dg.dg_fp8_grouped_contiguous(*args)
    dg.dg_fp8_grouped_contiguous(*args, z((sum_M, N), torch.int16).view(BF16))
    # masked: sfa [G, K/128, round_up(max_m, 4)], d given as a bf16 view of int16
    G, max_m, N, K = 5, 130, 8, 640
    margs = (z((G, max_m, K), U8), z((G, K // 128, 132), F32), z((G, N, K), U8), z((G, 1, K // 128), F32),
             z((G,), I32))
    dg.dg_fp8_grouped_masked(*margs)
    dg.dg_fp8_grouped_masked(*margs, z((G, max_m, N), torch.int16).view(BF16))
    # re-quantised outputs, given and allocated
    a, sfa, b, sfb = dense(300, 640, 640)
    q, sfo = dg.dg_fp8_gemm_nt_q(a, sfa, b, sfb)
    assert q.shape == (300, 640) and sfo.shape == (5, 300)
    dg.dg_fp8_gemm_nt_q(a, sfa, b, sfb, z((300, 640), U8), z((5, 300), F32))
    G, sum_M, N, K = 3, 384, 384, 384
    cargs = (z((sum_M, K), U8), z((K // 128, sum_M), F32), z((G, N, K), U8), z((G, 3, K // 128), F32),
             z((sum_M,), I32))
    q, sfo = dg.dg_fp8_grouped_contiguous_q(*cargs)
    assert q.shape == (sum_M, N) and sfo.shape == (3, sum_M)
    G, max_m, N, K = 4, 256, 256, 512
    margs = (z((G, max_m, K), U8), z((G, K // 128, max_m), F32), z((G, N, K), U8), z((G, 2, K // 128), F32),
             z((G,), I32))
    q, sfo = dg.dg_fp8_grouped_masked_q(*margs)
    assert q.shape == (G, max_m, N) and sfo.shape == (G, 2, max_m)
    dg.dg_fp8_grouped_masked_q(*margs, z((G, max_m, N), U8), z((G, 2, max_m), F32))
    assert "dg_fp8_grouped_masked_q" in fake.names and "dg_quant_weight_128x128" in fake.names


def test_wrong_arguments_raise_before_any_cuda_call(fake):
    a, sfa, b, sfb = dense(128, 256, 512)
    with pytest.raises(ValueError, match="sfa: expected shape"):
        dg.dg_fp8_gemm_nt(a, z((4, 132), F32), b, sfb)            # ld must be round_up(M, 4)
    with pytest.raises(ValueError, match="b: expected shape"):
        dg.dg_fp8_gemm_nt(a, sfa, z((256, 256), U8), sfb)          # K differs from A's
    with pytest.raises(TypeError, match="a: expected dtype"):
        dg.dg_fp8_gemm_nt(a.float(), sfa, b, sfb)
    with pytest.raises(TypeError, match="d: expected dtype"):
        dg.dg_fp8_gemm_nt(a, sfa, b, sfb, z((128, 256), F32))
    with pytest.raises(ValueError, match="must be contiguous"):
        dg.dg_fp8_gemm_nt(a, sfa, z((512, 256), U8).t(), sfb)
    with pytest.raises(TypeError, match="sfb: expected a torch.Tensor"):
        dg.dg_fp8_gemm_nt(a, sfa, b, None)
    with pytest.raises(ValueError, match="a: expected 2 dimensions"):
        dg.dg_fp8_gemm_nt(a[None], sfa, b, sfb)
    with pytest.raises(ValueError, match="masked_m: expected shape"):
        dg.dg_fp8_grouped_masked(z((2, 64, 128), U8), z((2, 1, 64), F32), z((2, 128, 128), U8),
                                 z((2, 1, 1), F32), z((3,), I32))
    with pytest.raises(TypeError, match="m_indices: expected dtype"):
        dg.dg_fp8_grouped_contiguous(z((128, 128), U8), z((1, 128), F32), z((2, 128, 128), U8),
                                     z((2, 1, 1), F32), z((128,), torch.int64))
    with pytest.raises(TypeError, match="x: expected dtype"):
        dg.dg_quant_act_1x128(z((4, 128), torch.float16))
    with pytest.raises(ValueError, match="sfo: expected shape"):
        dg.dg_fp8_gemm_nt_q(a, sfa, b, sfb, z((128, 256), U8), z((2, 4), F32))
    assert fake.names == []


def test_cpu_tensors_are_refused():
    a, sfa, b, sfb = dense(128, 256, 512)
    with pytest.raises(ValueError, match="a CUDA tensor is required"):
        dg.dg_fp8_gemm_nt(a, sfa, b, sfb)
    with pytest.raises(ValueError, match="a CUDA tensor is required"):
        dg.dg_quant_act_1x128(z((4, 128), F32))

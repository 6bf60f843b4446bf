"""GPU parity of calls that consume the previous call's output directly.

The quantizers and the W4A16 GEMMs start under programmatic dependent launch:
a kernel may begin while the kernel before it on the stream is still running.
Here every call reads what the call right before it wrote, on one stream, with
no copy, synchronisation or other kernel in between, and the whole chain must
equal the oracle's composition of the same steps bit for bit (the GEMMs within
the usual bound):

  FP8 1x128 dequant -> FP8 per-tensor (its scale becomes the next call's given
  amax) -> NVFP4 with that given amax -> INT4 g128 of the NVFP4 dequant ->
  W4A16 on those weights at once, directly and after another W4A16 launch;
  likewise the zero-point INT4 quantizer and its GEMM.

The W4A16 kernels read their weights before waiting for the previous kernel;
the library launches them after the stream's earlier work when an INT4
quantizer call may still be writing those weights."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_same_bytes, check_gemm, dev_bf16, dev_f32, host

pytestmark = pytest.mark.gpu

REL = 1e-3
K, N = 256, 1024


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def seeded(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((K, N)) * 0.05).astype(np.float32)
    x[:, rng.choice(N, 8, replace=False)] *= np.float32(30)         # outlier columns
    a = rng.standard_normal((64, K)).astype(np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)               # bf16 by truncation: any bits do
    return x, bits


def oracle_chain(x):
    _, _, d1 = oracle.quant_fp8(x, oracle.FP8_GROUP_1x128)
    c2, s2, d2 = oracle.quant_fp8(d1, oracle.FP8_PER_TENSOR)
    c3, s3, g3, d3 = oracle.quant_nvfp4(d2, amax_in=float(s2[0]))
    return (c2, s2, d2), (c3, s3, g3, d3)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_quantizer_chain_back_to_back(qz, seed):
    x, _ = seeded(seed)
    x_d = dev_f32(x)
    _, _, d1 = qz.qz_quantize_fp8(x_d, oracle.FP8_GROUP_1x128, dequant=True)
    c2, s2, d2 = qz.qz_quantize_fp8(d1, oracle.FP8_PER_TENSOR, dequant=True)
    c3, s3, g3, d3 = qz.qz_quantize_nvfp4(d2, global_amax_in=s2, dequant=True)
    qw, sc, d4 = qz.qz_quantize_int4_g128(d3, dequant=True)
    torch.cuda.synchronize()
    (rc2, rs2, rd2), (rc3, rs3, rg3, rd3) = oracle_chain(x)
    rqw, rsc, rd4 = oracle.quant_int4_g128(rd3)
    assert_same_bytes(host(c2), rc2, "fp8 tensor codes")
    assert_same_bytes(host(s2), rs2, "fp8 tensor scale")
    assert_same_bytes(host(d2), rd2, "fp8 tensor dequant")
    assert_same_bytes(host(c3), rc3, "nvfp4 codes (given amax)")
    assert_same_bytes(host(s3).reshape(rs3.shape), rs3, "nvfp4 block scales (given amax)")
    assert_same_bytes(host(g3).reshape(np.shape(rg3)), np.asarray(rg3, np.float32), "nvfp4 global scale")
    assert_same_bytes(host(d3), rd3, "nvfp4 dequant (given amax)")
    assert_same_bytes(host(qw), rqw, "int4 codes")
    assert_same_bytes(host(sc).view(np.uint16), rsc, "int4 scales")
    assert_same_bytes(host(d4), rd4, "int4 dequant")


@pytest.mark.parametrize("M", [1, 4, 12, 24, 48])
def test_int4_quantizer_then_w4a16_at_once(qz, M):
    """INT4 quantizer, then at once a W4A16 GEMM on other weights, then one on the
    new weights; and the new weights' GEMM directly after the quantizer."""
    x, a_bits = seeded(10 + M)
    A = a_bits[:M]
    A_d = dev_bf16(A)
    w_old = (np.random.default_rng(M).standard_normal((K, N)) * 0.02).astype(np.float32)
    rq_old, rs_old, _ = oracle.quant_int4_g128(w_old, want_deq=False)
    qw_old = torch.from_numpy(rq_old).cuda()
    sc_old = torch.from_numpy(rs_old.view(np.int16)).cuda().view(torch.bfloat16)
    x_d = dev_f32(x)
    torch.cuda.synchronize()
    for rnd in range(3):
        src = x_d * float(rnd + 1) if rnd else x_d                  # a torch kernel, then the chain
        qw, sc, _ = qz.qz_quantize_int4_g128(src)
        y_direct = qz.qz_gemm_w4a16(A_d, qw, sc)
        qw2, sc2, _ = qz.qz_quantize_int4_g128(src)
        y_other = qz.qz_gemm_w4a16(A_d, qw_old, sc_old)
        y_after = qz.qz_gemm_w4a16(A_d, qw2, sc2)
        torch.cuda.synchronize()
        rq, rs, _ = oracle.quant_int4_g128(x * np.float32(rnd + 1), want_deq=False)
        y_ref, bound = oracle.gemm_w4a16(A, rq, rs)
        check_gemm(host(y_direct), y_ref, bound, f"M={M} round {rnd}: directly after the quantizer", REL)
        check_gemm(host(y_after), y_ref, bound, f"M={M} round {rnd}: after another W4A16 launch", REL)
        y_ref_o, bound_o = oracle.gemm_w4a16(A, rq_old, rs_old)
        check_gemm(host(y_other), y_ref_o, bound_o, f"M={M} round {rnd}: other weights", REL)


@pytest.mark.parametrize("M", [1, 16])
def test_int4_zp_quantizer_then_gemm_at_once(qz, M):
    x, a_bits = seeded(30 + M)
    A = a_bits[:M]
    A_d = dev_bf16(A)
    x_d = dev_f32(x)
    torch.cuda.synchronize()
    qw, sc, z, _ = qz.qz_quantize_int4_g128_zp(x_d)
    y = qz.qz_gemm_w4a16_zp(A_d, qw, sc, z)
    torch.cuda.synchronize()
    rq, rs, rz, _ = oracle.quant_int4_g128_zp(x, want_deq=False)
    assert_same_bytes(host(qw), rq, "zp codes")
    assert_same_bytes(host(z), rz, "zero points")
    y_ref, bound = oracle.gemm_w4a16_zp(A, rq, rs, rz)
    check_gemm(host(y), y_ref, bound, f"zp M={M} directly after the quantizer", REL)

"""GPU parity of the variants beyond the base formats, against the oracle:

* INT4 with a zero point (quantizer bit-exact; W4A16 GEMM within the GEMM bound);
* weight-only FP4 GEMMs (NVFP4 and MXFP4 weights, bf16 activations);
* FP8 KV writes with per-head scales (computed and given) and with K per channel
  plus a zero point and V per token (bit-exact);
* SmoothQuant statistics and factors, INT8 per-row quantization (bit-exact) and the
  INT8 W8A8 GEMM;
* the FP8 block GEMM whose epilogue quantizes its output to FP8 1x128.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import assert_same_bytes, bf16_bits_to_f64, check_gemm, dev_bf16, dev_f32, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def f32_of(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------ INT4 zero point

def zp_weight(K, N, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    w[:, 3] = np.abs(w[:, 3])                                  # all positive: z = 0
    w[:, 5] = np.float32(1.0) + np.abs(w[:, 5])                # far above zero
    w[:128, 7] = 0.0                                           # an all-zero group
    w[:, 9] += np.float32(0.05)                                # shifted range
    return w


@pytest.mark.parametrize("bf16", [False, True])
def test_int4_zp_quantizer_bit_exact(qz, bf16):
    w = zp_weight(512, 192, seed=1)
    x = syn.to_bf16_bits(w) if bf16 else w
    qw, sc, zp, deq = qz.qz_quantize_int4_g128_zp(dev_bf16(x) if bf16 else dev_f32(x), dequant=True)
    rq, rs, rz, rd = oracle.quant_int4_g128_zp(x)
    assert_same_bytes(host(qw), rq, "qweight")
    assert_same_bytes(host(sc), rs, "scales")
    assert_same_bytes(host(zp), rz, "zero points")
    assert_same_bytes(host(deq), rd, "dequant")


def activations(M, K, seed):
    rng = np.random.default_rng(seed + 1000)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[:, rng.choice(K, max(1, K // 100), replace=False)] *= np.float32(20)
    return syn.to_bf16_bits(a)


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_w4a16_zp_gemm(qz, M):
    K, N = 1024, 192
    rq, rs, rz, _ = oracle.quant_int4_g128_zp(zp_weight(K, N, seed=M), want_deq=False)
    A = activations(M, K, seed=M)
    y = host(qz.qz_gemm_w4a16_zp(dev_bf16(A), dev(rq), dev(rs.view(np.int16)).view(torch.bfloat16), dev(rz)))
    y_ref, bound = oracle.gemm_w4a16_zp(A, rq, rs, rz)
    check_gemm(y, y_ref, bound, f"w4a16 zp M={M}")


@pytest.mark.parametrize("M", [1, 16])
def test_w4a16_zp_llama_shape_sampled(qz, M):
    A, w = syn.w4a16_decode_inputs(M=M, seed=3)
    qw, sc, zp, _ = qz.qz_quantize_int4_g128_zp(dev_f32(w))
    rq, rs, rz, _ = oracle.quant_int4_g128_zp(w, want_deq=False)
    assert np.array_equal(host(qw), rq) and np.array_equal(host(zp), rz)
    y = host(qz.qz_gemm_w4a16_zp(dev_bf16(A), qw, sc, zp))
    rng = np.random.default_rng(M)
    ii, jj = rng.integers(0, M, 2000), rng.integers(0, w.shape[1], 2000)
    y_ref, bound = oracle.gemm_w4a16_zp(A, rq, rs, rz, ii, jj)
    check_gemm(y[ii, jj], y_ref, bound, f"w4a16 zp llama M={M}")


# ------------------------------------------------- weight-only FP4 GEMMs

def fp4_weight(N, K, seed):
    rng = np.random.default_rng(seed)
    return syn.to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))


@pytest.mark.parametrize("M", [1, 5, 8, 16])
@pytest.mark.parametrize("K,N", [(128, 32), (512, 96), (2048, 256)])
def test_w4a16_nvfp4_and_mxfp4(qz, M, K, N):
    bt = fp4_weight(N, K, seed=M + K)
    A = activations(M, K, seed=K + M)
    cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
    y = host(qz.qz_gemm_w4a16_nvfp4(dev_bf16(A), dev(cb), dev(sb), dev_f32(np.float32([gb]))))
    y_ref, bound = oracle.gemm_w4a16_nvfp4(A, cb, sb, gb)
    check_gemm(y, y_ref, bound, f"w4a16 nvfp4 M={M} K={K} N={N}")
    cm, em, _ = oracle.quant_mxfp4(bt, want_deq=False)
    y = host(qz.qz_gemm_w4a16_mxfp4(dev_bf16(A), dev(cm), dev(em)))
    y_ref, bound = oracle.gemm_w4a16_mxfp4(A, cm, em)
    check_gemm(y, y_ref, bound, f"w4a16 mxfp4 M={M} K={K} N={N}")


def test_w4a16_fp4_every_code_and_scale_exact(qz):
    """Weights that visit every E2M1 code (including +-0.5, the one whose bf16 form is
    subnormal before scaling) with power-of-two scales and integer activations: every
    product and sum is exact, so the output is the oracle's exact value rounded once
    to bf16."""
    rng = np.random.default_rng(7)
    M, N, K = 4, 64, 256
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    qB = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sB = np.full((N, K // 16), 0x38, np.uint8)                         # E4M3 1.0
    eB = np.full((N, K // 32), 127, np.uint8)                          # 2^0
    A = syn.to_bf16_bits(rng.integers(-3, 4, (M, K)).astype(np.float32))
    y = host(qz.qz_gemm_w4a16_nvfp4(dev_bf16(A), dev(qB), dev(sB), dev_f32(np.float32([0.5]))))
    y_ref, _ = oracle.gemm_w4a16_nvfp4(A, qB, sB, 0.5)
    assert np.array_equal(y, syn.to_bf16_bits(y_ref.astype(np.float32)))
    y = host(qz.qz_gemm_w4a16_mxfp4(dev_bf16(A), dev(qB), dev(eB)))
    y_ref, _ = oracle.gemm_w4a16_mxfp4(A, qB, eB)
    assert np.array_equal(y, syn.to_bf16_bits(y_ref.astype(np.float32)))


@pytest.mark.parametrize("M", [1, 16])
def test_w4a16_nvfp4_llama_shape_sampled(qz, M):
    A, w = syn.w4a16_decode_inputs(M=M, seed=4)
    bt = syn.to_bf16_bits(np.ascontiguousarray(w.T))
    cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
    y = host(qz.qz_gemm_w4a16_nvfp4(dev_bf16(A), dev(cb), dev(sb), dev_f32(np.float32([gb]))))
    rng = np.random.default_rng(M + 50)
    ii, jj = rng.integers(0, M, 2000), rng.integers(0, bt.shape[0], 2000)
    y_ref, bound = oracle.gemm_w4a16_nvfp4(A, cb, sb, gb, ii, jj)
    check_gemm(y[ii, jj], y_ref, bound, f"w4a16 nvfp4 llama M={M}")


# --------------------------------------------------------- KV variants

@pytest.mark.parametrize("T", [1, 17, 4096])
def test_kv_per_head_compute_and_given(qz, T):
    k, v = syn.kv_cache_inputs(seed=T, T=T)
    kc, vc, ks, vs = qz.qz_kv_write_fp8_per_head(dev_bf16(k), dev_bf16(v))
    rkc, rvc, rks, rvs, _, _ = oracle.kv_write_fp8_per_head(k, v)
    assert_same_bytes(host(kc), rkc, "k codes")
    assert_same_bytes(host(vc), rvc, "v codes")
    assert_same_bytes(host(ks), rks, "k scales")
    assert_same_bytes(host(vs), rvs, "v scales")
    given = (np.arange(1, 9, dtype=np.float32).reshape(1, 8) * np.float32(0.01))
    kc, vc, _, _ = qz.qz_kv_write_fp8_per_head(dev_bf16(k), dev_bf16(v), k_scale=dev_f32(given),
                                               v_scale=dev_f32(given * 2), mode=qz.SCALE_GIVEN)
    assert_same_bytes(host(kc), oracle.kv_fp8_per_head_given(k, given)[0], "k codes, given scales")
    assert_same_bytes(host(vc), oracle.kv_fp8_per_head_given(v, given * 2)[0], "v codes, given scales")


@pytest.mark.parametrize("B,H,T,D", [(1, 8, 4096, 128), (2, 3, 17, 64), (1, 2, 1, 128), (1, 1, 40, 256)])
def test_kv_channel_zero_point(qz, B, H, T, D):
    k, v = syn.kv_cache_inputs(seed=B * T + D, B=B, H=H, T=T, D=D)
    kc, vc, ksc, kzp, vsc = qz.qz_kv_write_fp8_channel_zp(dev_bf16(k), dev_bf16(v))
    rkc, rks, rkz, _ = oracle.kv_k_channel_zp(k)
    assert_same_bytes(host(kc), rkc, "k codes")
    assert_same_bytes(host(ksc), rks, "k scales")
    assert_same_bytes(host(kzp), rkz, "k zero points")
    rvc, rvs, _ = oracle.quant_fp8(v.reshape(B * H * T, D), oracle.FP8_PER_ROW, want_deq=False)
    assert_same_bytes(host(vc).reshape(B * H * T, D), rvc, "v codes (per token)")
    assert_same_bytes(host(vsc).reshape(-1), rvs, "v scales (per token)")


# -------------------------------------------------- SmoothQuant + INT8

def test_col_amax_and_smooth_factors(qz):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((300, 512)).astype(np.float32)
    x[:, rng.choice(512, 6, replace=False)] *= np.float32(40.0)
    wt = syn.to_bf16_bits((rng.standard_normal((768, 512)) * 0.02).astype(np.float32))
    xm = host(qz.qz_col_amax(dev_f32(x)))
    wm = host(qz.qz_col_amax(dev_bf16(wt)))
    assert_same_bytes(xm, oracle.col_amax(x), "activation amax")
    assert_same_bytes(wm, oracle.col_amax(wt), "weight amax")
    xm[3] = 0.0                                                       # the 1e-12 floor
    s = host(qz.qz_smooth_factors(dev_f32(xm), dev_f32(wm)))
    assert_same_bytes(s, oracle.smooth_factors(xm, wm), "smooth factors")


@pytest.mark.parametrize("bf16", [False, True])
def test_int8_rows_bit_exact(qz, bf16):
    rng = np.random.default_rng(22)
    x = rng.standard_normal((77, 1024)).astype(np.float32)
    x[:, 5] *= np.float32(50.0)
    x[10] = 0.0                                                       # an all-zero row
    xin = syn.to_bf16_bits(x) if bf16 else x
    f = rng.uniform(0.1, 8.0, 1024).astype(np.float32)
    for op, name in ((qz.SMOOTH_NONE, "none"), (qz.SMOOTH_DIVIDE, "divide"), (qz.SMOOTH_MULTIPLY, "multiply")):
        d = dev_bf16(xin) if bf16 else dev_f32(xin)
        q, s, deq = qz.qz_quantize_int8_rows(d, dev_f32(f) if op else None, op, dequant=True)
        rq, rs, rd = oracle.quant_int8_rows(xin, f if op else None, op)
        assert_same_bytes(host(q).view(np.uint8), rq.view(np.uint8), f"codes {name}")
        assert_same_bytes(host(s), rs, f"scales {name}")
        assert_same_bytes(host(deq), rd, f"dequant {name}")


def int8_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K)).astype(np.float32)
    X[:, rng.choice(K, max(1, K // 100), replace=False)] *= np.float32(20.0)
    Wt = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xb, wb = syn.to_bf16_bits(X), syn.to_bf16_bits(Wt)
    s = oracle.smooth_factors(oracle.col_amax(xb), oracle.col_amax(wb))
    qa, sa, _ = oracle.quant_int8_rows(xb, s, oracle.INT8_DIVIDE, want_deq=False)
    qb, sb, _ = oracle.quant_int8_rows(wb, s, oracle.INT8_MULTIPLY, want_deq=False)
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (128, 256, 512), (256, 512, 1024), (384, 768, 192),
                                   (640, 512, 256)])
def test_int8_gemm_full_check(qz, M, N, K):
    qa, sa, qb, sb = int8_operands(M, N, K, seed=M + N + K)
    y = host(qz.qz_gemm_int8(dev(qa), dev_f32(sa), dev(qb), dev_f32(sb)))
    y_ref, bound = oracle.gemm_int8(qa, sa, qb, sb)
    check_gemm(y, y_ref, bound, f"int8 {M}x{N}x{K}")


def test_int8_gemm_integer_case_is_exact(qz):
    """Unit scales and codes in -1..1 over K = 256: the output is the integer matmul,
    exactly representable in bf16 (|y| <= 256); the extreme codes -128 and 127 are
    covered by a second case whose sums stay within 2^24."""
    rng = np.random.default_rng(23)
    M, N, K = 128, 256, 256
    qa = rng.integers(-1, 2, (M, K)).astype(np.int8)
    qb = rng.integers(-1, 2, (N, K)).astype(np.int8)
    ones_m, ones_n = np.ones(M, np.float32), np.ones(N, np.float32)
    y = host(qz.qz_gemm_int8(dev(qa), dev_f32(ones_m), dev(qb), dev_f32(ones_n)))
    ref = qa.astype(np.int64) @ qb.T.astype(np.int64)
    assert np.array_equal(bf16_bits_to_f64(y), ref.astype(np.float64))
    qa = rng.choice(np.array([-128, 127, 0, 1], np.int8), (M, K))
    qb = rng.choice(np.array([-128, 127, -1, 0], np.int8), (N, K))
    y = host(qz.qz_gemm_int8(dev(qa), dev_f32(ones_m), dev(qb), dev_f32(ones_n)))
    ref = (qa.astype(np.int64) @ qb.T.astype(np.int64)).astype(np.float32)    # |sums| < 2^24: exact in fp32
    assert np.array_equal(y, syn.to_bf16_bits(ref))


def test_int8_gemm_prefill_shape_sampled(qz):
    """The FP8 prefill workload's shape (2048 x 14336 x 4096) in W8A8 INT8 with
    SmoothQuant; 3000 sampled outputs."""
    M, N, K = 2048, 14336, 4096
    qa, sa, qb, sb = int8_operands(M, N, K, seed=5)
    y = host(qz.qz_gemm_int8(dev(qa), dev_f32(sa), dev(qb), dev_f32(sb)))
    rng = np.random.default_rng(6)
    ii, jj = rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    y_ref, bound = oracle.gemm_int8(qa, sa, qb, sb, ii, jj)
    check_gemm(y[ii, jj], y_ref, bound, "int8 prefill shape")
    assert qz.qz_device_error() == 0


def test_smoothquant_pipeline_on_gpu(qz):
    """Statistics, factors and both INT8 quantizers on the GPU (each bit-exact), then
    the GEMM within the bound."""
    rng = np.random.default_rng(24)
    M, N, K = 256, 512, 768
    X = rng.standard_normal((M, K)).astype(np.float32)
    X[:, [3, 100, 500]] *= np.float32(60.0)
    Wt = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xb, wb = syn.to_bf16_bits(X), syn.to_bf16_bits(Wt)
    xd, wd = dev_bf16(xb), dev_bf16(wb)
    s = qz.qz_smooth_factors(qz.qz_col_amax(xd), qz.qz_col_amax(wd))
    qa, sa, _ = qz.qz_quantize_int8_rows(xd, s, qz.SMOOTH_DIVIDE)
    qb, sb, _ = qz.qz_quantize_int8_rows(wd, s, qz.SMOOTH_MULTIPLY)
    rs = oracle.smooth_factors(oracle.col_amax(xb), oracle.col_amax(wb))
    assert_same_bytes(host(s), rs, "factors")
    rqa, rsa, _ = oracle.quant_int8_rows(xb, rs, oracle.INT8_DIVIDE, want_deq=False)
    rqb, rsb, _ = oracle.quant_int8_rows(wb, rs, oracle.INT8_MULTIPLY, want_deq=False)
    assert_same_bytes(host(qa).view(np.uint8), rqa.view(np.uint8), "activation codes")
    assert_same_bytes(host(qb).view(np.uint8), rqb.view(np.uint8), "weight codes")
    y = host(qz.qz_gemm_int8(qa, sa, qb, sb))
    y_ref, bound = oracle.gemm_int8(rqa, rsa, rqb, rsb)
    check_gemm(y, y_ref, bound, "smoothquant int8")


# ---------------------------------------- FP8 GEMM with quantized output

def test_fp8_gemm_quantized_output_exact_case(qz):
    """Unit scales and small integer operands make every sum exact, so the output the
    epilogue quantizes is the oracle's exact product: codes and scales bit-exact against
    the oracle's 1x128 FP8 quantizer of the bf16-rounded exact output."""
    rng = np.random.default_rng(25)
    M, N, K = 256, 512, 384
    vals = np.array([0x00, 0x38, 0x40, 0x44, 0xB8, 0xC0, 0x30], np.uint8)   # 0, 1, 2, 3, -1, -2, 0.5
    qa = vals[rng.integers(0, len(vals), (M, K))]
    qb = vals[rng.integers(0, len(vals), (N, K))]
    sa = np.ones((M, K // 128), np.float32)
    sb = np.ones((N // 128, K // 128), np.float32)
    codes, scales, Y = qz.qz_gemm_fp8_block_quant(dev(qa), dev_f32(sa), dev(qb), dev_f32(sb), want_y=True)
    y_ref, _ = oracle.gemm_fp8_block(qa, sa, qb, sb)
    ybf = syn.to_bf16_bits(y_ref.astype(np.float32))                 # exact values: one rounding to bf16
    assert np.array_equal(host(Y), ybf)
    rc, rs, _ = oracle.quant_fp8(ybf, oracle.FP8_GROUP_1x128, want_deq=False)
    assert_same_bytes(host(codes), rc, "output codes")
    assert_same_bytes(host(scales), rs, "output scales")


def test_fp8_gemm_quantized_output_prefill_shape(qz):
    """The prefill shape with realistic operands: the bf16 output equals the plain FP8
    GEMM's bit for bit, the fused codes and scales equal the 1x128 quantizer applied to
    that output, and the output stays within the GEMM bound of the oracle."""
    a, bt = syn.fp8_block_gemm_inputs(seed=2, M=512, K=1024, N=2048)
    qa, sa, _ = oracle.quant_fp8(a, oracle.FP8_GROUP_1x128, want_deq=False)
    qb, sb, _ = oracle.quant_fp8(bt, oracle.FP8_BLOCK_128x128, want_deq=False)
    d = [dev(qa), dev_f32(sa), dev(qb), dev_f32(sb)]
    codes, scales, Y = qz.qz_gemm_fp8_block_quant(*d, want_y=True)
    y_plain = qz.qz_gemm_fp8_block(*d)
    assert np.array_equal(host(Y), host(y_plain))
    c2, s2, _ = qz.qz_quantize_fp8(y_plain, qz.FP8_GROUP_1x128)
    assert np.array_equal(host(codes), host(c2)) and np.array_equal(host(scales), host(s2))
    codes_only, scales_only, none = qz.qz_gemm_fp8_block_quant(*d)
    assert none is None and np.array_equal(host(codes_only), host(codes))
    rng = np.random.default_rng(8)
    ii, jj = rng.integers(0, 512, 2000), rng.integers(0, 2048, 2000)
    y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)
    check_gemm(host(Y)[ii, jj], y_ref, bound, "fp8 gemm with quantized output")
    assert qz.qz_device_error() == 0

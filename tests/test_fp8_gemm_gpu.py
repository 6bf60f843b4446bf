"""GPU parity of the block-scaled FP8 GEMM (tcgen05) against the oracle's FP64
reference: |y_gpu - y_ref| <= 1e-3 * sum_k |a_ik * b_kj| plus half a bf16 ulp
of y_ref (the rounding of the bf16 output), on the exactly dequantized operands. Operands come from the oracle's quantizers (1x128 for A,
128x128 for B^T). Shapes cover one tile, several tiles in both directions with
more tiles than a wave of CTAs, long K, and the full prefill size (sampled)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import bf16_bits_to_f64, check_gemm, host

pytestmark = pytest.mark.gpu

REL = 1e-3


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def operands(M, N, K, seed, outliers=True):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    if outliers:
        a[:, rng.choice(K, max(1, K // 100), replace=False)] *= np.float32(20)
    bt = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qa, sa, _ = oracle.quant_fp8(syn.to_bf16_bits(a), oracle.FP8_GROUP_1x128, want_deq=False)
    qb, sb, _ = oracle.quant_fp8(syn.to_bf16_bits(bt), oracle.FP8_BLOCK_128x128, want_deq=False)
    return qa, sa, qb, sb


def run(qz, qa, sa, qb, sb):
    d = [torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in (qa, sa, qb, sb)]
    return host(qz.qz_gemm_fp8_block(*d))


def check(y_bits, y_ref, bound, what):
    check_gemm(y_bits, y_ref, bound, what, REL)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (128, 256, 512), (256, 512, 256), (384, 768, 384),
                                   (128, 256, 2048)])
def test_fp8_block_gemm_full_check(qz, M, N, K):
    qa, sa, qb, sb = operands(M, N, K, seed=M + N + K)
    y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb)
    check(run(qz, qa, sa, qb, sb), y_ref, bound, f"{M}x{N}x{K}")


def test_fp8_block_gemm_many_tiles(qz):
    """More output tiles than SMs (persistent CTAs loop over several tiles)."""
    M, N, K = 2048, 4096, 256
    qa, sa, qb, sb = operands(M, N, K, seed=7)
    y = run(qz, qa, sa, qb, sb)
    rng = np.random.default_rng(7)
    ii, jj = rng.integers(0, M, 4000), rng.integers(0, N, 4000)
    y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)
    check(y[ii, jj], y_ref, bound, "many tiles")
    # every tile's corner elements
    ti, tj = np.meshgrid(np.arange(0, M, 128), np.arange(0, N, 256), indexing="ij")
    for di, dj in ((0, 0), (127, 255), (64, 131)):
        ii, jj = (ti + di).ravel(), (tj + dj).ravel()
        y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)
        check(y[ii, jj], y_ref, bound, f"tile corners +{di},{dj}")


def test_fp8_block_gemm_integer_exact(qz):
    """Integer-valued operands with unit scales: exact integer matmul (bf16-rounded)."""
    rng = np.random.default_rng(3)
    M, N, K = 128, 256, 256
    a = rng.integers(-4, 5, (M, K))
    b = rng.integers(-4, 5, (N, K))
    qa = oracle.e4m3_encode_array(a.astype(np.float32)).reshape(M, K)
    qb = oracle.e4m3_encode_array(b.astype(np.float32)).reshape(N, K)
    y = bf16_bits_to_f64(run(qz, qa, np.ones((M, K // 128), np.float32), qb,
                             np.ones((N // 128, K // 128), np.float32)))
    ref = (a @ b.T).astype(np.float32)
    assert np.array_equal(y, bf16_bits_to_f64(syn.to_bf16_bits(ref)))


def test_fp8_block_gemm_scales_per_block(qz):
    """Distinct power-of-two scales per (row, k-block) and per 128x128 block: a scale
    applied to the wrong block shows up as a large error."""
    rng = np.random.default_rng(4)
    M, N, K = 256, 512, 512
    a = rng.integers(-3, 4, (M, K)).astype(np.float32)
    b = rng.integers(-3, 4, (N, K)).astype(np.float32)
    qa = oracle.e4m3_encode_array(a).reshape(M, K)
    qb = oracle.e4m3_encode_array(b).reshape(N, K)
    sa = np.ldexp(1.0, rng.integers(-6, 7, (M, K // 128))).astype(np.float32)
    sb = np.ldexp(1.0, rng.integers(-6, 7, (N // 128, K // 128))).astype(np.float32)
    y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb)
    check(run(qz, qa, sa, qb, sb), y_ref, bound, "per-block scales")


def test_fp8_block_gemm_prefill_full_size_sampled(qz):
    """Config 3 at full size (M=2048, N=14336, K=4096) in the bench's launch
    configuration; operands from the oracle's quantizers; sampled outputs."""
    a, bt = syn.fp8_block_gemm_inputs(seed=0)
    qa, sa, _ = oracle.quant_fp8(a, oracle.FP8_GROUP_1x128, want_deq=False)
    # B^T 128x128 quantization, block row by block row (independent blocks)
    qb = np.empty(bt.shape, np.uint8)
    sb = np.empty((bt.shape[0] // 128, bt.shape[1] // 128), np.float32)
    for i in range(bt.shape[0] // 128):
        qb[i * 128:(i + 1) * 128], sb[i:i + 1], _ = oracle.quant_fp8(bt[i * 128:(i + 1) * 128],
                                                                     oracle.FP8_BLOCK_128x128, want_deq=False)
    y = run(qz, qa, sa, qb, sb)
    rng = np.random.default_rng(0)
    ii, jj = rng.integers(0, a.shape[0], 3000), rng.integers(0, bt.shape[0], 3000)
    y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)
    check(y[ii, jj], y_ref, bound, "prefill sampled")

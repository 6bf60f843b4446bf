"""GPU parity of the W4A16 GEMM against the oracle's FP64 reference.

Acceptance (the GEMM tolerance): |y_gpu - y_ref| <= 1e-3 * sum_k |a_ik * b_kj| plus
half a bf16 ulp of y_ref (the rounding of the bf16 output), on the exactly
dequantized operands. The INT4 weights fed to both sides come from
the oracle's quantizer, never from the GPU. Shapes cover ragged token counts
(M = 1..64), several tiles, the half-depth last K stage (K % 256 == 128), the
full Llama-3.1-8B MLP size (sampled outputs) and a grouped launch."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from gpu_util import bf16_bits_to_f64, check_gemm, dev_bf16, host

import torch

pytestmark = pytest.mark.gpu

REL = 1e-3


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def quantized_weight(K, N, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
    return qw, sc


def activations(M, K, seed):
    rng = np.random.default_rng(seed + 1000)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[:, rng.choice(K, max(1, K // 100), replace=False)] *= np.float32(20)
    return syn.to_bf16_bits(a)


def check(y_gpu_bits, y_ref, bound, what):
    check_gemm(y_gpu_bits, y_ref, bound, what, REL)


def run(qz, A, qw, sc):
    qw_d = torch.from_numpy(qw).cuda()
    sc_d = torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16)
    return host(qz.qz_gemm_w4a16(dev_bf16(A), qw_d, sc_d))


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 16, 17, 32, 33, 64])
def test_w4a16_tokens(qz, M):
    K, N = 512, 384
    qw, sc = quantized_weight(K, N, seed=M)
    A = activations(M, K, seed=M)
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc)
    check(run(qz, A, qw, sc), y_ref, bound, f"M={M}")


@pytest.mark.parametrize("K,N", [(128, 64), (384, 192), (640, 1024), (1024, 2048), (4096, 128)])
def test_w4a16_shapes(qz, K, N):
    M = 5
    qw, sc = quantized_weight(K, N, seed=K + N)
    A = activations(M, K, seed=K)
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc)
    check(run(qz, A, qw, sc), y_ref, bound, f"K={K} N={N}")


@pytest.mark.parametrize("M,K,N", [(24, 256, 192), (64, 640, 320), (12, 128, 64)])
def test_w4a16_partial_column_tiles(qz, M, K, N):
    """N not a multiple of the 128-column tiles of the tensor-core kernel (9-64 tokens):
    the columns past N are read as zeros and never stored."""
    qw, sc = quantized_weight(K, N, seed=N)
    A = activations(M, K, seed=M)
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc)
    check(run(qz, A, qw, sc), y_ref, bound, f"M={M} K={K} N={N}")


def test_w4a16_integer_exact(qz):
    """Unit scales and small integer activations: the result is an exact integer
    (a plain integer matmul), so the GPU must match it exactly after bf16 rounding."""
    rng = np.random.default_rng(5)
    M, K, N = 8, 256, 128
    q = rng.integers(-8, 8, (K, N))
    qw = np.zeros((K // 8, N), np.uint32)
    for k in range(K):
        qw[k // 8] |= (q[k].astype(np.uint32) & 0xF) << np.uint32(4 * (k % 8))
    a = rng.integers(-3, 4, (M, K)).astype(np.float32)
    A = syn.to_bf16_bits(a)
    sc = np.full((K // 128, N), 0x3F80, np.uint16)
    y = bf16_bits_to_f64(run(qz, A, qw.view(np.int32), sc))
    ref = (a.astype(np.int64) @ q).astype(np.float64)
    ref_bf16 = bf16_bits_to_f64(syn.to_bf16_bits(ref.astype(np.float32)))
    assert np.array_equal(y, ref_bf16)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a16_llama_mlp_full_size_sampled(qz, M):
    """Config 2 at full size (K=4096, N=14336) in the bench's launch configuration,
    with the oracle's INT4 weights; 3000 sampled outputs checked one by one."""
    A, w = syn.w4a16_decode_inputs(M=M, seed=0)
    qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
    y = run(qz, A, qw, sc)
    rng = np.random.default_rng(M)
    ii, jj = rng.integers(0, M, 3000), rng.integers(0, w.shape[1], 3000)
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc, ii, jj)
    check(y[ii, jj], y_ref, bound, f"llama M={M}")
    # the tail of the last tile is covered too
    jt = np.arange(w.shape[1] - 64, w.shape[1])
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc, np.zeros(64, np.int64), jt)
    check(y[0, jt], y_ref, bound, "last columns")


def test_w4a16_gpu_quantizer_composes(qz):
    """GPU INT4 quantizer -> GPU GEMM equals the oracle composition."""
    A = activations(3, 1024, seed=9)
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((1024, 512)) * 0.02).astype(np.float32)
    qw_d, sc_d, _ = qz.qz_quantize_int4_g128(torch.from_numpy(w).cuda())
    y = host(qz.qz_gemm_w4a16(dev_bf16(A), qw_d, sc_d))
    qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc)
    check(y, y_ref, bound, "composed")


def test_w4a16_grouped_qwen_shapes(qz):
    """One grouped launch of one Qwen3-0.6B layer's seven linears at 64 tokens."""
    probs, refs = [], []
    for layer, name, A, w in syn.qwen3_decode_linears(layers=1, tokens=64, seed=0):
        qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
        K, N = w.shape
        Y = torch.empty((64, N), dtype=torch.bfloat16, device="cuda")
        probs.append((dev_bf16(A), torch.from_numpy(qw).cuda(),
                      torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16), Y))
        rng = np.random.default_rng(K + N)
        ii, jj = rng.integers(0, 64, 400), rng.integers(0, N, 400)
        refs.append((name, ii, jj) + oracle.gemm_w4a16(A, qw, sc, ii, jj))
    qz.qz_gemm_w4a16_grouped(probs)
    for (name, ii, jj, y_ref, bound), (_, _, _, Y) in zip(refs, probs):
        check(host(Y)[ii, jj], y_ref, bound, f"grouped {name}")


@pytest.mark.parametrize("tokens", [3, 16])
def test_w4a16_grouped_decode_tokens(qz, tokens):
    """Grouped launch at decode batch sizes (the register-direct kernel): one
    Qwen3-0.6B layer's seven linears with mixed K and N, every output checked."""
    probs, refs = [], []
    for layer, name, A, w in syn.qwen3_decode_linears(layers=1, tokens=tokens, seed=1):
        qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
        K, N = w.shape
        Y = torch.empty((tokens, N), dtype=torch.bfloat16, device="cuda")
        probs.append((dev_bf16(A), torch.from_numpy(qw).cuda(),
                      torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16), Y))
        refs.append((name,) + oracle.gemm_w4a16(A, qw, sc))
    qz.qz_gemm_w4a16_grouped(probs)
    for (name, y_ref, bound), (_, _, _, Y) in zip(refs, probs):
        check(host(Y), y_ref, bound, f"grouped {name} tokens={tokens}")


@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("K,N", [(128, 64), (1152, 192), (2944, 64), (8192, 128), (8320, 64)])
def test_w4a16_staging_depths(qz, M, K, N):
    """Up to 8 tokens, K from one 128-deep group to the deepest K staged whole in shared
    memory (8192), odd group counts (a half-filled last box), and one group deeper
    (8320, the register-direct kernel)."""
    qw, sc = quantized_weight(K, N, seed=K + M)
    A = activations(M, K, seed=K + 7 * M)
    y_ref, bound = oracle.gemm_w4a16(A, qw, sc)
    check(run(qz, A, qw, sc), y_ref, bound, f"M={M} K={K} N={N}")


def grouped_case(qz, shapes, seed):
    rng = np.random.default_rng(seed)
    probs, refs = [], []
    for i, (M, K, N) in enumerate(shapes):
        qw, sc = quantized_weight(K, N, seed=seed + i)
        A = activations(M, K, seed=seed + 3 * i)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        probs.append((dev_bf16(A), torch.from_numpy(qw).cuda(),
                      torch.from_numpy(sc.view(np.int16)).cuda().view(torch.bfloat16), Y))
        refs.append(oracle.gemm_w4a16(A, qw, sc))
    qz.qz_gemm_w4a16_grouped(probs)
    for i, ((y_ref, bound), (_, _, _, Y)) in enumerate(zip(refs, probs)):
        check(host(Y), y_ref, bound, f"problem {i} {shapes[i]}")


def test_w4a16_grouped_single_token_many_problems(qz):
    """130 single-token problems of mixed K and N: more than one launch's problem table."""
    shapes = [(1, 128 * (1 + i % 5), 64 * (1 + i % 3)) for i in range(130)]
    grouped_case(qz, shapes, seed=40)


def test_w4a16_grouped_mixed_tokens_and_depths(qz):
    """One token next to several in one launch, and a group that holds one K deeper than
    8192 (the whole group then runs register-direct)."""
    grouped_case(qz, [(1, 1024, 128), (2, 384, 64), (8, 2048, 192), (1, 128, 64)], seed=50)
    grouped_case(qz, [(1, 1024, 128), (4, 8320, 64), (1, 256, 64)], seed=60)


def test_w4a16_grouped_split_into_shares(qz):
    """Groups larger than one launch's problem table at 9-16 tokens (70 problems: two
    launches of 35) and at 17-64 tokens (90 problems: two launches of 45)."""
    grouped_case(qz, [(12, 128 * (1 + i % 4), 64 * (1 + i % 3)) for i in range(70)], seed=70)
    grouped_case(qz, [(40, 128 * (1 + i % 4), 128 * (1 + i % 2)) for i in range(90)], seed=80)

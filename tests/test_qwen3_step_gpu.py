"""The Qwen3-0.6B-shaped decode step (28 layers x 7 linears = 196 GEMMs at 64 tokens)
run exactly as the bench runs it, checked problem by problem against the oracle.

W4A16: all 196 problems in one qz_gemm_w4a16_grouped call (the library splits them
into equal launch shares). NVFP4: all 196 activations quantized by one
qz_quantize_nvfp4_grouped call (codes, block scales and global scale compared bit for
bit with the oracle), the weights' scales re-laid once by qz_prepare_fp4_scales, and
all 196 GEMMs in one qz_gemm_nvfp4_grouped call (several launches). Weights are
quantized by the oracle, so every GEMM operand the GPU reads is the oracle's. Every
problem gets 64 sampled outputs, so the problems past each launch boundary are
covered.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import assert_same_bytes, check_gemm, dev_bf16, host

pytestmark = pytest.mark.gpu

TOKENS = 64
SAMPLES = 64


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _samples(N, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, TOKENS, SAMPLES), rng.integers(0, N, SAMPLES)


def _oracle_map(fn):
    """fn over the 196 linears, on host threads (each oracle call is single-threaded C
    and releases the interpreter lock); results in the linears' order."""
    linears = list(enumerate(syn.qwen3_decode_linears(layers=28, tokens=TOKENS, seed=0)))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        return list(ex.map(lambda item: fn(*item), linears))


def test_qwen3_decode_step_w4a16_all_196(qz):
    def prep(i, item):
        layer, name, A, w = item
        qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
        ii, jj = _samples(w.shape[1], 1000 + i)
        return A, qw, sc, (f"L{layer} {name}", ii, jj) + oracle.gemm_w4a16(A, qw, sc, ii, jj)

    probs, refs = [], []
    for A, qw, sc, ref in _oracle_map(prep):
        Y = torch.empty((TOKENS, qw.shape[1]), dtype=torch.bfloat16, device="cuda")
        probs.append((dev_bf16(A), dev(qw), dev(sc.view(np.int16)).view(torch.bfloat16), Y))
        refs.append(ref)
    assert len(probs) == 196
    qz.qz_gemm_w4a16_grouped(probs)
    torch.cuda.synchronize()
    for (what, ii, jj, y_ref, bound), p in zip(refs, probs):
        check_gemm(host(p[3])[ii, jj], y_ref, bound, f"w4a16 step {what}")
    assert qz.qz_device_error() == 0


def test_qwen3_decode_step_nvfp4_all_196(qz):
    def prep(i, item):
        layer, name, A, w = item
        bt = syn.to_bf16_bits(np.ascontiguousarray(w.T))          # the weight as B^T [N, K]
        cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
        ca, sa, ga, _ = oracle.quant_nvfp4(A, want_deq=False)
        ii, jj = _samples(w.shape[1], 2000 + i)
        ref = (f"L{layer} {name}", ii, jj) + oracle.gemm_nvfp4(ca, sa, ga, cb, sb, gb, ii, jj)
        return A, (ca, sa, ga), (cb, sb, gb, w.shape[0], w.shape[1]), ref

    acts, act_ref, weights, refs = [], [], [], []
    for A, aref, (cb, sb, gb, K, N), ref in _oracle_map(prep):
        acts.append(dev_bf16(A))
        act_ref.append(aref)
        weights.append((dev(cb), qz.qz_prepare_fp4_scales(dev(sb), K, nv=True), dev(np.float32([gb])), K, N))
        refs.append(ref)
    assert len(acts) == 196
    # the activations: one grouped quantizer call, bit-exact per tensor
    quant = qz.qz_quantize_nvfp4_grouped(acts)
    torch.cuda.synchronize()
    for t, ((ca, sa, ga), (gca, gsa, gga)) in enumerate(zip(act_ref, quant)):
        assert_same_bytes(host(gca), ca, f"activation {t} codes")
        assert_same_bytes(host(gsa), sa, f"activation {t} block scales")
        assert_same_bytes(host(gga), np.float32([ga]), f"activation {t} global scale")
    # the GEMMs: one grouped call over the GPU-quantized activations
    probs = []
    for (gca, gsa, gga), (cb, sbp, gb, K, N) in zip(quant, weights):
        Y = torch.empty((TOKENS, N), dtype=torch.bfloat16, device="cuda")
        probs.append((gca, gsa, gga, cb, sbp, gb, Y))
    qz.qz_gemm_nvfp4_grouped(probs)
    torch.cuda.synchronize()
    for (what, ii, jj, y_ref, bound), p in zip(refs, probs):
        check_gemm(host(p[6])[ii, jj], y_ref, bound, f"nvfp4 step {what}")
    assert qz.qz_device_error() == 0

"""The allocation-free NVFP4 GEMM (qz_gemm_nvfp4_noalloc), called through the C ABI.

It exists for callers that cannot allocate device memory or pass a workspace —
runtimes that plan all device memory once at start-up and give plug-ins no
allocator, or latency-critical loops that cannot risk cudaMalloc synchronising
the device. Its scratch is a fixed array inside the library, shared by every
call. This test checks, on two calls in a row with different problems (so the
second call sees the first call's leftovers in that array), that each result
equals the workspace entry point qz_gemm_nvfp4 bit for bit (the same kernels
run on the same operands, so any difference would mean stale scratch was read)
and lies within the GEMM tolerance the other tests use; that the Python wrapper
of the same name gives the same bits; and that a problem too large for the
fixed array is rejected with QZ_ERR_SHAPE before anything is launched. It runs
last (file name) and also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import bf16_bits_to_f64, gemm_tolerance, host

pytestmark = pytest.mark.gpu

QZ_ERR_SHAPE = 2
SCRATCH_BYTES = 4 << 20            # QZ_NVFP4_NOALLOC_SCRATCH_BYTES in include/qz.h


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[:, rng.choice(K, max(1, K // 200), replace=False)] *= np.float32(30)
    bt = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    ca, sa, ga, _ = oracle.quant_nvfp4(syn.to_bf16_bits(a), want_deq=False)
    cb, sb, gb, _ = oracle.quant_nvfp4(syn.to_bf16_bits(bt), want_deq=False)
    return ca, sa, ga, cb, sb, gb


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_nvfp4_noalloc_matches_workspace_entry_point():
    import bit_quantized_linear_quantizers_gb300 as qz
    lib = qz.lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (M, N, K, seed) in enumerate([(256, 512, 1024, 1), (384, 256, 512, 2)]):
        ca, sa, ga, cb, sb, gb = _operands(M, N, K, seed)
        d = [_dev(x) for x in (ca, sa, np.float32([ga]), cb, sb, np.float32([gb]))]
        y_noalloc = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        rc = lib.qz_gemm_nvfp4_noalloc(*[_p(t) for t in d], _p(y_noalloc), M, N, K, stream)
        assert rc == 0, qz.qz_status_string(rc)
        y_ws = qz.qz_gemm_nvfp4(*d)                       # the workspace entry point
        y_py = qz.qz_gemm_nvfp4_noalloc(*d)               # the Python wrapper of the C call
        torch.cuda.synchronize()
        assert np.array_equal(host(y_noalloc), host(y_ws)), f"call {call}: differs from qz_gemm_nvfp4"
        assert np.array_equal(host(y_py), host(y_ws)), f"call {call}: the wrapper differs from qz_gemm_nvfp4"
        y_ref, bound = oracle.gemm_nvfp4(ca, sa, ga, cb, sb, gb)
        a = bf16_bits_to_f64(host(y_noalloc))
        assert np.all(np.abs(a - y_ref) <= gemm_tolerance(y_ref, bound)), f"call {call}: outside the GEMM tolerance"


def test_nvfp4_noalloc_rejects_problems_beyond_its_scratch():
    import bit_quantized_linear_quantizers_gb300 as qz
    M, N, K = 16384, 256, 4096            # needs (M + N) * K / 16 bytes > 4 MiB of scratch
    assert (M + N) * K // 16 > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: the call is rejected first
    rc = qz.lib.qz_gemm_nvfp4_noalloc(fake, fake, fake, fake, fake, fake, fake, M, N, K, None)
    assert rc == QZ_ERR_SHAPE

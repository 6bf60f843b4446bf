"""The C ABI on the host (no GPU needed): libqz.so loads, exports every function
include/qz.h declares, sizes workspaces, and rejects invalid calls during host
validation, before anything could reach a GPU. Every call below carries at least
one invalid argument, so none of them can launch a kernel on any machine."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qz.h")


def _lib():
    import __graft_entry__
    b = __graft_entry__._build_module()
    return ctypes.CDLL(b.build())


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qz_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["qz_quantize_fp8", "qz_quantize_mxfp4", "qz_quantize_nvfp4", "qz_quantize_int4_g128",
                     "qz_kv_write_fp8", "qz_gemm_w4a16", "qz_gemm_fp8_block", "qz_gemm_nvfp4",
                     "qz_gemm_mxfp4", "qz_workspace_size", "qz_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = _lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def test_status_strings(qz):
    assert qz.qz_status_string(0) == "QZ_OK"
    for s in range(1, 8):
        assert qz.qz_status_string(s).startswith("QZ_ERR_")


def test_workspace_sizes(qz):
    assert qz.qz_workspace_size(qz.OP_QUANTIZE_FP8, 1024, 1024, qz.FP8_PER_TENSOR) > 0
    assert qz.qz_workspace_size(qz.OP_QUANTIZE_FP8, 1024, 1024, qz.FP8_PER_ROW) == 0
    assert qz.qz_workspace_size(qz.OP_KV_WRITE_FP8, 1 << 22) >= 2 * 4
    assert qz.qz_workspace_size(qz.OP_GEMM_W4A16, 16, 14336, 4096) == 0
    assert qz.qz_workspace_size(99, 1, 1, 1) == 0


FAKE = ctypes.c_void_p(0x10000)        # aligned, never dereferenced: validation fails first
ODD = ctypes.c_void_p(0x10001)
NULL = None


@pytest.mark.parametrize("args,expect", [
    # x, dtype, rows, cols, ldx, gran, codes, scales, deq, ws, ws_bytes, stream
    ((FAKE, 0, 4, 128, 128, 9, FAKE, FAKE, NULL, NULL, 0, NULL), 1),        # bad granularity
    ((FAKE, 7, 4, 128, 128, 1, FAKE, FAKE, NULL, NULL, 0, NULL), 1),        # bad dtype
    ((FAKE, 0, 4, 128, 64, 1, FAKE, FAKE, NULL, NULL, 0, NULL), 1),         # ldx < cols
    ((NULL, 0, 4, 128, 128, 1, FAKE, FAKE, NULL, NULL, 0, NULL), 1),        # null x
    ((FAKE, 0, 4, 100, 100, 3, FAKE, FAKE, NULL, NULL, 0, NULL), 2),        # 1x128 needs cols % 128
    ((FAKE, 0, 200, 128, 128, 2, FAKE, FAKE, NULL, NULL, 0, NULL), 2),      # 128x128 needs rows % 128
    ((ODD, 0, 4, 128, 128, 3, FAKE, FAKE, NULL, NULL, 0, NULL), 3),         # misaligned x, group path
    ((FAKE, 0, 4, 128, 128, 0, FAKE, FAKE, NULL, NULL, 0, NULL), 7),        # per-tensor without ws
    ((FAKE, 0, 0, 128, 128, 0, FAKE, FAKE, NULL, NULL, 0, NULL), 2),        # empty per-tensor
])
def test_quantize_fp8_validation(qz, args, expect):
    assert qz.lib.qz_quantize_fp8(*args) == expect


def test_empty_inputs_are_noops(qz):
    # rows == 0: nothing to do, no device touched (pointers are fake)
    assert qz.lib.qz_quantize_fp8(FAKE, 0, 0, 128, 128, 1, FAKE, FAKE, NULL, NULL, 0, NULL) == 0
    assert qz.lib.qz_quantize_mxfp4(FAKE, 0, 0, 64, 64, FAKE, FAKE, NULL, NULL) == 0
    assert qz.lib.qz_quantize_int4_g128(FAKE, 0, 0, 64, 64, FAKE, FAKE, NULL, NULL) == 0
    assert qz.lib.qz_kv_write_fp8(FAKE, FAKE, 0, 8, 16, 128, FAKE, FAKE, FAKE, FAKE, 1, NULL, 0, NULL) == 0


def test_fp4_and_int4_validation(qz):
    L = qz.lib
    assert L.qz_quantize_mxfp4(FAKE, 0, 4, 48, 48, FAKE, FAKE, NULL, NULL) == 2          # cols % 32
    assert L.qz_quantize_mxfp4(FAKE, 0, 4, 64, 63, FAKE, FAKE, NULL, NULL) == 1          # ldx < cols
    assert L.qz_quantize_mxfp4(ODD, 0, 4, 64, 64, FAKE, FAKE, NULL, NULL) == 3
    assert L.qz_quantize_nvfp4(FAKE, 0, 4, 24, 24, FAKE, FAKE, FAKE, NULL, NULL, NULL, 0, NULL) == 2
    assert L.qz_quantize_nvfp4(FAKE, 0, 4, 32, 32, FAKE, FAKE, FAKE, NULL, NULL, NULL, 0, NULL) == 7
    assert L.qz_quantize_nvfp4(FAKE, 0, 4, 32, 32, FAKE, FAKE, NULL, NULL, NULL, FAKE, 1 << 20, NULL) == 1
    assert L.qz_quantize_int4_g128(FAKE, 0, 100, 64, 64, FAKE, FAKE, NULL, NULL) == 2    # K % 128
    assert L.qz_quantize_int4_g128(FAKE, 0, 128, 40, 40, FAKE, FAKE, NULL, NULL) == 2    # N % 64
    assert L.qz_kv_write_fp8(FAKE, FAKE, 1, 8, 16, 128, FAKE, FAKE, FAKE, FAKE, 5, NULL, 0, NULL) == 1
    assert L.qz_kv_write_fp8(FAKE, FAKE, 1, 8, 16, 128, FAKE, FAKE, FAKE, FAKE, 0, NULL, 0, NULL) == 7
    assert L.qz_kv_write_fp8(ODD, FAKE, 1, 8, 16, 128, FAKE, FAKE, FAKE, FAKE, 1, NULL, 0, NULL) == 3


def test_gemm_validation(qz):
    L = qz.lib
    # A, qweight, scale, Y, M, N, K, ws, ws_bytes, stream
    assert L.qz_gemm_w4a16(FAKE, FAKE, FAKE, FAKE, 65, 128, 128, NULL, 0, NULL) == 2     # M > 64
    assert L.qz_gemm_w4a16(FAKE, FAKE, FAKE, FAKE, 4, 100, 128, NULL, 0, NULL) == 2      # N % 64
    assert L.qz_gemm_w4a16(FAKE, FAKE, FAKE, FAKE, 4, 128, 96, NULL, 0, NULL) == 2       # K % 128
    assert L.qz_gemm_w4a16(NULL, FAKE, FAKE, FAKE, 4, 128, 128, NULL, 0, NULL) == 1
    assert L.qz_gemm_w4a16(ODD, FAKE, FAKE, FAKE, 4, 128, 128, NULL, 0, NULL) == 3
    assert L.qz_gemm_w4a16(FAKE, FAKE, FAKE, FAKE, 0, 128, 128, NULL, 0, NULL) == 1
    assert L.qz_gemm_w4a16_grouped(None, 0, NULL, 0, NULL) == 1
    assert L.qz_gemm_fp8_block(FAKE, FAKE, FAKE, FAKE, FAKE, 100, 256, 128, NULL, 0, NULL) == 2
    assert L.qz_gemm_fp8_block(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 100, NULL, 0, NULL) == 2
    assert L.qz_gemm_fp8_block(FAKE, FAKE, NULL, FAKE, FAKE, 128, 256, 128, NULL, 0, NULL) == 1
    assert L.qz_gemm_nvfp4(FAKE, FAKE, NULL, FAKE, FAKE, FAKE, FAKE, 128, 256, 256, NULL, 0, NULL) == 1
    assert L.qz_gemm_nvfp4(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 200, 256, NULL, 0, NULL) == 2
    assert L.qz_gemm_mxfp4(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 100, NULL, 0, NULL) == 2
    assert L.qz_gemm_mxfp4(ODD, FAKE, FAKE, FAKE, FAKE, 128, 256, 256, NULL, 0, NULL) == 3
    # qA, sA, gA, qB, sB, gB, y_amax, y_codes, y_scales, y_global, M, N, K, ws, ws_bytes, stream
    q = L.qz_gemm_nvfp4_quant
    assert q(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, FAKE, FAKE, 128, 256, 256, NULL, 0, NULL) == 1  # amax
    assert q(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, 128, 256, 256, NULL, 0, NULL) == 1
    assert q(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 200, 256, NULL, 0, NULL) == 2  # N
    assert q(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ODD, FAKE, FAKE, 128, 256, 256, NULL, 0, NULL) == 3   # codes
    assert q(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 256, NULL, 0, NULL) == 7  # ws
    # qA, eA, qB, eB, y_codes, y_e8m0, M, N, K, ws, ws_bytes, stream
    mq = L.qz_gemm_mxfp4_quant
    assert mq(FAKE, FAKE, FAKE, FAKE, NULL, FAKE, 128, 256, 256, NULL, 0, NULL) == 1
    assert mq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 100, NULL, 0, NULL) == 2                 # K
    assert mq(FAKE, FAKE, FAKE, FAKE, FAKE, ODD, 128, 256, 256, NULL, 0, NULL) == 3                  # e8m0
    assert mq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 256, 256, NULL, 0, NULL) == 7                 # ws


def test_grouped_nvfp4_and_prepare_validation(qz):
    L = qz.lib
    P = qz._Nvfp4Problem

    def one(**kw):
        f = dict(qA=0x10000, sA=0x10000, gA=0x10000, qB=0x10000, sB_prepared=0x10000, gB=0x10000,
                 Y=0x10000, M=64, N=1024, K=1024)
        f.update(kw)
        arr = (P * 1)()
        arr[0] = P(**f)
        return arr

    ws_need = qz.qz_workspace_size(qz.OP_GEMM_NVFP4_GROUPED, 1, 1024)
    assert ws_need == 128 * 1024 // 16
    assert L.qz_gemm_nvfp4_grouped(None, 1, FAKE, ws_need, NULL) == 1
    assert L.qz_gemm_nvfp4_grouped(one(), 0, FAKE, ws_need, NULL) == 1                  # count < 1
    assert L.qz_gemm_nvfp4_grouped(one(), 257, FAKE, ws_need, NULL) == 1                # count > 256
    assert L.qz_gemm_nvfp4_grouped(one(M=129), 1, FAKE, ws_need, NULL) == 2             # decode: M <= 128
    assert L.qz_gemm_nvfp4_grouped(one(N=1000), 1, FAKE, ws_need, NULL) == 2            # N % 256
    assert L.qz_gemm_nvfp4_grouped(one(K=1000), 1, FAKE, ws_need, NULL) == 2            # K % 256
    assert L.qz_gemm_nvfp4_grouped(one(gB=0), 1, FAKE, ws_need, NULL) == 1
    assert L.qz_gemm_nvfp4_grouped(one(qB=0x10008), 1, FAKE, ws_need, NULL) == 3        # 16-byte alignment
    assert L.qz_gemm_nvfp4_grouped(one(sA=0x10002), 1, FAKE, ws_need, NULL) == 3        # 4-byte alignment
    assert L.qz_gemm_nvfp4_grouped(one(), 1, FAKE, ws_need - 1, NULL) == 7              # workspace too small
    assert L.qz_gemm_nvfp4_grouped(one(), 1, NULL, ws_need, NULL) == 7
    # scales, rows, K, nv, out, stream
    assert qz.qz_workspace_size(qz.OP_PREPARE_FP4_SCALES, 200, 1024, 1) == 256 * 64
    assert qz.qz_workspace_size(qz.OP_PREPARE_FP4_SCALES, 200, 1024, 0) == 256 * 32
    assert L.qz_prepare_fp4_scales(NULL, 128, 256, 1, FAKE, NULL) == 1
    assert L.qz_prepare_fp4_scales(FAKE, 128, 256, 2, FAKE, NULL) == 1                 # nv must be 0 or 1
    assert L.qz_prepare_fp4_scales(FAKE, 0, 256, 1, FAKE, NULL) == 1
    assert L.qz_prepare_fp4_scales(FAKE, 128, 100, 1, FAKE, NULL) == 2                 # K % 256
    assert L.qz_prepare_fp4_scales(FAKE, 128, 256, 1, ODD, NULL) == 3


def test_grouped_nvfp4_quantize_validation(qz):
    L = qz.lib
    T = qz._Nvfp4Tensor

    def one(n=1, **kw):
        f = dict(x=0x10000, rows=4, cols=1024, codes=0x10000, scale_e4m3=0x10000, global_scale=0x10000)
        f.update(kw)
        arr = (T * n)()
        for i in range(n):
            arr[i] = T(**f)
        return arr

    ws_need = qz.qz_workspace_size(qz.OP_QUANTIZE_NVFP4_GROUPED, 3)
    assert ws_need == 3 * 4 * 4
    assert qz.qz_workspace_size(qz.OP_QUANTIZE_NVFP4_GROUPED, 257) == 0
    assert L.qz_quantize_nvfp4_grouped(None, 1, 0, FAKE, ws_need, NULL) == 1
    assert L.qz_quantize_nvfp4_grouped(one(), 0, 0, FAKE, ws_need, NULL) == 1             # count < 1
    assert L.qz_quantize_nvfp4_grouped(one(257), 257, 1, FAKE, 1 << 20, NULL) == 1        # count > 256
    assert L.qz_quantize_nvfp4_grouped(one(), 1, 5, FAKE, ws_need, NULL) == 1             # dtype
    assert L.qz_quantize_nvfp4_grouped(one(rows=0), 1, 0, FAKE, ws_need, NULL) == 1
    assert L.qz_quantize_nvfp4_grouped(one(global_scale=0), 1, 0, FAKE, ws_need, NULL) == 1
    assert L.qz_quantize_nvfp4_grouped(one(cols=40), 1, 0, FAKE, ws_need, NULL) == 2      # cols % 16
    assert L.qz_quantize_nvfp4_grouped(one(x=0x10008), 1, 0, FAKE, ws_need, NULL) == 3    # x 16-byte
    assert L.qz_quantize_nvfp4_grouped(one(codes=0x10002), 1, 0, FAKE, ws_need, NULL) == 3
    assert L.qz_quantize_nvfp4_grouped(one(3), 3, 0, FAKE, ws_need - 1, NULL) == 7         # workspace
    assert L.qz_quantize_nvfp4_grouped(one(3), 3, 0, NULL, ws_need, NULL) == 7


def test_grouped_w4a16_validation(qz):
    """A group is checked whole before any launch: one bad problem anywhere (here after a
    valid one) rejects the call."""
    L = qz.lib
    P = qz._W4A16Problem
    good = dict(A=0x10000, qweight=0x10000, scale_bf16=0x10000, Y=0x10000, M=4, N=128, K=256)

    def group(*changes):
        arr = (P * len(changes))()
        for i, ch in enumerate(changes):
            arr[i] = P(**{**good, **ch})
        return arr

    many = (P * 257)()
    assert L.qz_gemm_w4a16_grouped(many, 257, NULL, 0, NULL) == 1            # count > 256
    assert L.qz_gemm_w4a16_grouped(group({}, {"M": 65}), 2, NULL, 0, NULL) == 2
    assert L.qz_gemm_w4a16_grouped(group({}, {"K": 200}), 2, NULL, 0, NULL) == 2
    assert L.qz_gemm_w4a16_grouped(group({}, {"N": 96}), 2, NULL, 0, NULL) == 2
    assert L.qz_gemm_w4a16_grouped(group({}, {"N": 0}), 2, NULL, 0, NULL) == 1
    assert L.qz_gemm_w4a16_grouped(group({}, {"Y": 0}), 2, NULL, 0, NULL) == 1
    assert L.qz_gemm_w4a16_grouped(group({}, {"scale_bf16": 0x10008}), 2, NULL, 0, NULL) == 3
    assert L.qz_gemm_w4a16_grouped(group({"M": 0}), 1, NULL, 0, NULL) == 1


def test_fp4_scale_layout_sizes(qz):
    """The prepared scale-factor layout holds whole 128-row blocks of 512-byte atoms (128 rows
    x 4 scales): rows padded up to a multiple of 128, K/16 (NVFP4) or K/32 (MXFP4) scales a
    row. The single-problem FP4 GEMMs' workspace holds both operands' re-laid scales, each
    rounded up to 1 KiB (the limit the allocation-free entry point states)."""
    size = qz.qz_workspace_size
    for rows, K in ((1, 256), (128, 256), (129, 4096), (8192, 4096)):
        padded = -(-rows // 128) * 128
        assert size(qz.OP_PREPARE_FP4_SCALES, rows, K, 1) == padded * (K // 16)
        assert size(qz.OP_PREPARE_FP4_SCALES, rows, K, 0) == padded * (K // 32)
        assert padded * (K // 16) % 512 == 0
    r1k = lambda b: -(-b // 1024) * 1024
    for M, N, K in ((128, 256, 256), (8192, 4096, 4096), (384, 512, 768)):
        want = r1k(M * K // 16) + r1k(N * K // 16)
        assert size(qz.OP_GEMM_NVFP4, M, N, K) == want
        assert size(qz.OP_GEMM_MXFP4, M, N, K) == want
    # the no-alloc scratch (4 MiB) fits M + N = 16384 at K = 4096, as its header states
    assert r1k(8192 * 4096 // 16) + r1k(8192 * 4096 // 16) <= 4 << 20
    assert size(qz.OP_PREPARE_FP4_SCALES, 0, 256, 1) == 0                  # rejected sizes: 0


def test_variant_entry_points_reject_bad_arguments_before_any_launch(qz):
    """The zero-point, KV, weight-only FP4, SmoothQuant/INT8 and fused-output entry points
    validate on the host: null pointers, shapes and alignment are refused before the
    device is even queried."""
    lib = qz.lib
    P = ctypes.c_void_p(0x1000)          # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(0x1002)        # misaligned
    INV, SHAPE, ALIGN, UNSUP = 1, 2, 3, 4
    assert lib.qz_kv_write_fp8_per_head(None, P, 1, 8, 16, 128, P, P, P, P, 0, P, 1 << 20, None) == INV
    assert lib.qz_kv_write_fp8_per_head(P, P, 1, 8, 16, 12, P, P, P, P, 0, P, 1 << 20, None) == SHAPE
    assert lib.qz_kv_write_fp8_per_head(odd, P, 1, 8, 16, 128, P, P, P, P, 0, P, 1 << 20, None) == ALIGN
    assert lib.qz_kv_write_fp8_per_head(P, P, 1, 8, 16, 128, P, P, P, P, 7, P, 1 << 20, None) == INV
    assert lib.qz_kv_write_fp8_channel_zp(P, P, 1, 8, 16, 96, P, P, P, P, P, P, 1 << 20, None) == SHAPE
    assert lib.qz_kv_write_fp8_channel_zp(P, P, 1, 8, 0, 128, P, P, P, P, P, P, 1 << 20, None) == INV
    assert lib.qz_quantize_int4_g128_zp(P, 0, 100, 64, 64, P, P, P, None, None) == SHAPE
    assert lib.qz_quantize_int4_g128_zp(P, 0, 128, 64, 64, P, P, None, None, None) == INV
    assert lib.qz_gemm_w4a16_zp(P, P, P, P, P, 17, 64, 128, None) == SHAPE
    assert lib.qz_gemm_w4a16_zp(P, P, P, odd, P, 1, 64, 128, None) == ALIGN
    assert lib.qz_gemm_w4a16_nvfp4(P, P, P, None, P, 1, 64, 128, None) == INV
    assert lib.qz_gemm_w4a16_nvfp4(P, P, P, P, P, 1, 48, 128, None) == SHAPE
    assert lib.qz_gemm_w4a16_mxfp4(P, P, P, P, 1, 64, 96, None) == SHAPE
    assert lib.qz_col_amax(P, 0, 10, 12, P, P, 1 << 20, None) == SHAPE
    assert lib.qz_smooth_factors(P, P, 16, ctypes.c_float(0.75), P, None) == UNSUP
    assert lib.qz_smooth_factors(None, P, 16, ctypes.c_float(0.5), P, None) == INV
    assert lib.qz_quantize_int8_rows(P, 0, 4, 64, None, 1, P, P, None, None) == INV
    assert lib.qz_quantize_int8_rows(P, 0, 4, 60, None, 0, P, P, None, None) == SHAPE
    assert lib.qz_gemm_int8(P, P, P, P, P, 128, 256, 96, None) == SHAPE
    assert lib.qz_gemm_int8(P, P, P, P, odd, 128, 256, 64, None) == ALIGN
    assert lib.qz_gemm_fp8_block_quant(P, P, P, P, None, None, P, 128, 256, 128, None) == INV
    assert lib.qz_gemm_fp8_block_quant(P, P, P, P, None, P, P, 128, 200, 128, None) == SHAPE


def test_variant_workspace_sizes(qz):
    assert qz.qz_workspace_size(qz.OP_KV_WRITE_FP8_PER_HEAD, 8, 4096 * 128) >= 16 * 4
    assert qz.qz_workspace_size(qz.OP_KV_WRITE_FP8_CHANNEL_ZP, 8, 4096, 128) >= 8 * 2 * 128 * 4
    assert qz.qz_workspace_size(qz.OP_COL_AMAX, 2048, 4096) >= 4096 * 4
    assert qz.qz_workspace_size(qz.OP_KV_WRITE_FP8_PER_HEAD, 0, 0) == 0

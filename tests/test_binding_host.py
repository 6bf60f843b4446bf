"""The Python binding's own checks, on the CPU: the C ABI receives bare pointers, so the
binding must refuse, before anything reaches libqz, tensors whose device, dtype, element
count or layout differ from what the C call will read or write. Every case here fails
in Python; nothing is launched."""
import pytest
import torch

import bit_quantized_linear_quantizers_gb300 as qz


def test_arg_accepts_a_dense_tensor_of_the_right_kind():
    t = torch.zeros((4, 8), dtype=torch.bfloat16)
    assert qz._arg(t, "t", -1, torch.bfloat16, 32) == t.data_ptr()
    assert qz._arg(t, "t", -1, 2) == t.data_ptr()                     # element size only
    assert qz._opt(None, "t", -1, 2) is None


@pytest.mark.parametrize("make, kind, numel, what", [
    (lambda: torch.zeros((4, 8), dtype=torch.float16), torch.bfloat16, None, "bfloat16"),
    (lambda: torch.zeros((4, 8), dtype=torch.float32), 2, None, "2-byte"),
    (lambda: torch.zeros((8, 4), dtype=torch.bfloat16).t(), torch.bfloat16, None, "not contiguous"),
    (lambda: torch.zeros((4, 8), dtype=torch.bfloat16)[:, :4], torch.bfloat16, None, "not contiguous"),
    (lambda: torch.zeros((4, 8), dtype=torch.uint8), 1, 33, "33 elements"),
    (lambda: torch.zeros((2,), dtype=torch.float32), torch.float32, 1, "1 elements"),
])
def test_arg_rejects(make, kind, numel, what):
    with pytest.raises(ValueError, match=what):
        qz._arg(make(), "t", -1, kind, numel)


def test_arg_rejects_another_device():
    with pytest.raises(ValueError, match="on cpu"):
        qz._arg(torch.zeros(4, dtype=torch.uint8), "t", 0, 1)


@pytest.fixture
def on_device0(monkeypatch):
    """The wrappers as they run with cuda:0 current: host tensors are on the wrong device."""
    monkeypatch.setattr(qz, "_device", lambda: 0)


def test_gemm_wrappers_refuse_host_tensors(on_device0):
    M, N, K = 4, 64, 128
    A = torch.zeros((M, K), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="A: .*on cpu"):
        qz.qz_gemm_w4a16(A, torch.zeros((K // 8, N), dtype=torch.int32),
                         torch.zeros((K // 128, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="qA: .*on cpu"):
        qz.qz_gemm_fp8_block(torch.zeros((128, K), dtype=torch.uint8), torch.zeros((128, 1)),
                             torch.zeros((256, K), dtype=torch.uint8), torch.zeros((2, 1)))
    with pytest.raises(ValueError, match="qA: .*on cpu"):
        qz.qz_gemm_nvfp4(torch.zeros((128, 128), dtype=torch.uint8), torch.zeros((128, 16), dtype=torch.uint8),
                         torch.ones(1), torch.zeros((256, 128), dtype=torch.uint8),
                         torch.zeros((256, 16), dtype=torch.uint8), torch.ones(1))
    with pytest.raises(ValueError, match="qA: .*on cpu"):
        qz.qz_gemm_mxfp4(torch.zeros((128, 128), dtype=torch.uint8), torch.zeros((128, 8), dtype=torch.uint8),
                         torch.zeros((256, 128), dtype=torch.uint8), torch.zeros((256, 8), dtype=torch.uint8))
    with pytest.raises(ValueError, match=r"A\[0\]: .*on cpu"):
        qz.qz_gemm_w4a16_grouped([(A, torch.zeros((K // 8, N), dtype=torch.int32),
                                   torch.zeros((K // 128, N), dtype=torch.bfloat16),
                                   torch.zeros((M, N), dtype=torch.bfloat16))])


def test_quantizer_wrappers_refuse_host_tensors(on_device0):
    x = torch.zeros((4, 128), dtype=torch.bfloat16)
    for call in (lambda: qz.qz_quantize_fp8(x, qz.FP8_GROUP_1x128),
                 lambda: qz.qz_quantize_mxfp4(x),
                 lambda: qz.qz_quantize_nvfp4(x),
                 lambda: qz.qz_quantize_int4_g128(torch.zeros((128, 64))),
                 lambda: qz.qz_quantize_nvfp4_grouped([x])):
        with pytest.raises(ValueError, match="on cpu"):
            call()
    kv = torch.zeros((1, 1, 4, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k: .*on cpu"):
        qz.qz_kv_write_fp8(kv, kv)


def test_unknown_fp8_granularity(on_device0, monkeypatch):
    monkeypatch.setattr(qz, "_device", lambda: -1)      # host tensors pass the device check
    with pytest.raises(ValueError, match="granularity"):
        qz.qz_quantize_fp8(torch.zeros((4, 128)), 7)


def test_output_shape_mismatch_is_refused_before_the_call(monkeypatch):
    """Shapes the C call cannot see: a W4A16 weight for another K, a Y of the wrong size,
    a grouped NVFP4 problem whose prepared scales are too short."""
    monkeypatch.setattr(qz, "_device", lambda: -1)
    M, N, K = 4, 64, 256
    A = torch.zeros((M, K), dtype=torch.bfloat16)
    qw = torch.zeros((K // 8, N), dtype=torch.int32)
    sc = torch.zeros((K // 128, N), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="qweight"):
        qz.qz_gemm_w4a16(A, torch.zeros((K // 16, N), dtype=torch.int32), sc)
    with pytest.raises(ValueError, match="scale_bf16"):
        qz.qz_gemm_w4a16(A, qw, torch.zeros((1, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="Y"):
        qz.qz_gemm_w4a16(A, qw, sc, Y=torch.zeros((M, N - 8), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="Y"):
        qz.qz_gemm_w4a16(A, qw, sc, Y=torch.zeros((M, N), dtype=torch.float16))
    qA, sA = torch.zeros((4, 128), dtype=torch.uint8), torch.zeros((4, 16), dtype=torch.uint8)
    qB = torch.zeros((256, 128), dtype=torch.uint8)
    g = torch.ones(1)
    with pytest.raises(ValueError, match=r"sB_prepared\[0\]"):
        qz.qz_gemm_nvfp4_grouped([(qA, sA, g, qB, torch.zeros(100, dtype=torch.uint8), g,
                                   torch.zeros((4, 256), dtype=torch.bfloat16))])


def test_binding_has_the_c_names():
    """Every entry point that include/qz.h declares has a Python function of the same name."""
    import test_abi
    missing = [n for n in test_abi.declared_functions() if not callable(getattr(qz, n, None))]
    assert missing == []


def test_noalloc_wrapper_checks_like_the_others(on_device0):
    with pytest.raises(ValueError, match="qA: .*on cpu"):
        qz.qz_gemm_nvfp4_noalloc(torch.zeros((128, 128), dtype=torch.uint8), torch.zeros((128, 16), dtype=torch.uint8),
                                 torch.ones(1), torch.zeros((256, 128), dtype=torch.uint8),
                                 torch.zeros((256, 16), dtype=torch.uint8), torch.ones(1))

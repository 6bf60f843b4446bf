"""Python binding of libqz, the GB300 (sm_103a) quantizers and quantized GEMMs.

Argument marshalling only: every step of the computation runs in libqz's CUDA
kernels, behind the C ABI declared in include/qz.h. The functions carry the C
names. PyTorch supplies device memory (output tensors) and the current CUDA
stream. There is no CPU path: importing this package fails when libqz.so has
not been built, and every call raises QZError unless libqz returns QZ_OK.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB, build  # noqa: F401  (build() is the in-tree build step)

__all__ = [
    "QZError", "lib", "F32", "BF16", "FP8_PER_TENSOR", "FP8_PER_ROW", "FP8_BLOCK_128x128",
    "FP8_GROUP_1x128", "SCALE_COMPUTE", "SCALE_GIVEN", "qz_workspace_size", "qz_status_string",
    "qz_device_error", "qz_selftest_bounded_wait", "qz_quantize_fp8", "qz_quantize_mxfp4", "qz_quantize_nvfp4",
    "qz_quantize_int4_g128", "qz_kv_write_fp8", "qz_gemm_w4a16", "qz_gemm_w4a16_grouped",
    "qz_gemm_fp8_block", "qz_gemm_nvfp4", "qz_gemm_nvfp4_noalloc", "qz_gemm_mxfp4", "qz_prepare_fp4_scales",
    "qz_gemm_nvfp4_grouped", "qz_quantize_nvfp4_grouped", "Workspace",
    "qz_kv_write_fp8_per_head", "qz_kv_write_fp8_channel_zp", "qz_quantize_int4_g128_zp", "qz_gemm_w4a16_zp",
    "qz_gemm_w4a16_nvfp4", "qz_gemm_w4a16_mxfp4", "qz_col_amax", "qz_smooth_factors", "qz_quantize_int8_rows",
    "qz_gemm_int8", "qz_gemm_fp8_block_quant", "qz_gemm_nvfp4_quant", "qz_gemm_mxfp4_quant", "SMOOTH_NONE",
    "SMOOTH_DIVIDE",
    "SMOOTH_MULTIPLY",
]

F32, BF16 = 0, 1
FP8_PER_TENSOR, FP8_PER_ROW, FP8_BLOCK_128x128, FP8_GROUP_1x128 = 0, 1, 2, 3
SCALE_COMPUTE, SCALE_GIVEN = 0, 1
OP_QUANTIZE_FP8, OP_QUANTIZE_NVFP4, OP_KV_WRITE_FP8 = 0, 1, 2
OP_GEMM_W4A16, OP_GEMM_FP8_BLOCK, OP_GEMM_NVFP4, OP_GEMM_MXFP4 = 3, 4, 5, 6
OP_GEMM_NVFP4_GROUPED, OP_PREPARE_FP4_SCALES, OP_QUANTIZE_NVFP4_GROUPED = 7, 8, 9
OP_KV_WRITE_FP8_PER_HEAD, OP_KV_WRITE_FP8_CHANNEL_ZP, OP_COL_AMAX = 10, 11, 12
SMOOTH_NONE, SMOOTH_DIVIDE, SMOOTH_MULTIPLY = 0, 1, 2

if not os.path.exists(LIB):
    raise ImportError(f"libqz.so is not built ({LIB}); run bit_quantized_linear_quantizers_gb300.build() "
                      "or __graft_entry__.build() first")

lib = ctypes.CDLL(LIB)

_P, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t


class _W4A16Problem(ctypes.Structure):
    _fields_ = [("A", _P), ("qweight", _P), ("scale_bf16", _P), ("Y", _P),
                ("M", _I), ("N", _I), ("K", _I)]


class _Nvfp4Problem(ctypes.Structure):
    _fields_ = [("qA", _P), ("sA", _P), ("gA", _P), ("qB", _P), ("sB_prepared", _P), ("gB", _P),
                ("Y", _P), ("M", _I), ("N", _I), ("K", _I)]


class _Nvfp4Tensor(ctypes.Structure):
    _fields_ = [("x", _P), ("rows", _I64), ("cols", _I64), ("codes", _P), ("scale_e4m3", _P),
                ("global_scale", _P)]


_SIGS = {
    "qz_workspace_size": (_SZ, [_I, _I64, _I64, _I64]),
    "qz_status_string": (ctypes.c_char_p, [_I]),
    "qz_device_error": (_I, []),
    "qz_selftest_bounded_wait": (_I, [ctypes.c_uint32, _P]),
    "qz_quantize_fp8": (_I, [_P, _I, _I64, _I64, _I64, _I, _P, _P, _P, _P, _SZ, _P]),
    "qz_quantize_mxfp4": (_I, [_P, _I, _I64, _I64, _I64, _P, _P, _P, _P]),
    "qz_quantize_nvfp4": (_I, [_P, _I, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qz_quantize_int4_g128": (_I, [_P, _I, _I64, _I64, _I64, _P, _P, _P, _P]),
    "qz_kv_write_fp8": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _SZ, _P]),
    "qz_gemm_w4a16": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "qz_gemm_w4a16_grouped": (_I, [ctypes.POINTER(_W4A16Problem), _I, _P, _SZ, _P]),
    "qz_gemm_fp8_block": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "qz_gemm_nvfp4": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "qz_gemm_mxfp4": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "qz_gemm_nvfp4_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "qz_prepare_fp4_scales": (_I, [_P, _I, _I, _I, _P, _P]),
    "qz_gemm_nvfp4_grouped": (_I, [ctypes.POINTER(_Nvfp4Problem), _I, _P, _SZ, _P]),
    "qz_quantize_nvfp4_grouped": (_I, [ctypes.POINTER(_Nvfp4Tensor), _I, _I, _P, _SZ, _P]),
    "qz_kv_write_fp8_per_head": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _SZ, _P]),
    "qz_kv_write_fp8_channel_zp": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "qz_quantize_int4_g128_zp": (_I, [_P, _I, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "qz_gemm_w4a16_zp": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "qz_gemm_w4a16_nvfp4": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "qz_gemm_w4a16_mxfp4": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "qz_col_amax": (_I, [_P, _I, _I64, _I64, _P, _P, _SZ, _P]),
    "qz_smooth_factors": (_I, [_P, _P, _I64, ctypes.c_float, _P, _P]),
    "qz_quantize_int8_rows": (_I, [_P, _I, _I64, _I64, _P, _I, _P, _P, _P, _P]),
    "qz_gemm_int8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "qz_gemm_fp8_block_quant": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "qz_gemm_nvfp4_quant": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "qz_gemm_mxfp4_quant": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class QZError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.qz_status_string(status).decode()}")


def _check(status: int, where: str):
    if status != 0:
        raise QZError(status, where)


def _ptr(t):
    # plain ints: ctypes converts them for c_void_p parameters (no wrapper object per call)
    return None if t is None else t.data_ptr()


def _device() -> int:
    """The current CUDA device: libqz launches there, so every tensor must live there."""
    return torch.cuda.current_device()


def _arg(t, name, dev, kind, numel=None):
    """Device pointer of a dense tensor on device `dev` whose elements are of dtype `kind`
    (or, for an int, that many bytes), `numel` of them when given. The C ABI sees only
    the pointer, so the layout that it assumes is checked here, before any launch."""
    if (t.get_device() != dev or not t.is_contiguous()
            or (t.dtype is not kind if isinstance(kind, torch.dtype) else t.element_size() != kind)
            or (numel is not None and t.numel() != numel)):
        want = str(kind).replace("torch.", "") if isinstance(kind, torch.dtype) else f"{kind}-byte"
        where = "cpu" if t.get_device() < 0 else f"cuda:{t.get_device()}"
        raise ValueError(f"{name}: expected a contiguous {want} tensor on cuda:{dev}"
                         + ("" if numel is None else f" with {numel} elements")
                         + f", got {t.dtype} {tuple(t.shape)} on {where}"
                         + ("" if t.is_contiguous() else ", not contiguous"))
    return t.data_ptr()


def _opt(t, name, dev, kind, numel=None):
    return None if t is None else _arg(t, name, dev, kind, numel)


def _on(x, name, dev):
    if x.get_device() != dev:
        where = "cpu" if x.get_device() < 0 else f"cuda:{x.get_device()}"
        raise ValueError(f"{name}: expected a tensor on cuda:{dev}, got one on {where}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype == torch.float32:
        return F32
    if x.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"libqz quantizers take float32 or bfloat16 input, got {x.dtype}")


def _rows_cols_ld(x: torch.Tensor):
    if x.dim() != 2 or (x.numel() and x.stride(1) != 1):
        raise ValueError("expected a 2-D tensor with unit stride in the last dimension")
    return x.shape[0], x.shape[1], (x.stride(0) if x.shape[0] > 1 else max(x.shape[1], 1))


_WS_CACHE = {}


def qz_workspace_size(op: int, d0: int, d1: int = 0, d2: int = 0) -> int:
    key = (op, d0, d1, d2)
    n = _WS_CACHE.get(key)
    if n is None:
        n = int(lib.qz_workspace_size(op, d0, d1, d2))
        if len(_WS_CACHE) < 4096:
            _WS_CACHE[key] = n
    return n


def qz_status_string(status: int) -> str:
    return lib.qz_status_string(status).decode()


def qz_device_error() -> int:
    return int(lib.qz_device_error())


def qz_selftest_bounded_wait(polls: int, stream=None):
    """Launch the bounded-wait self-test (a wait that nothing completes gives up after
    `polls` polls and records QZ_ERR_TIMEOUT); read the result with qz_device_error()."""
    _check(lib.qz_selftest_bounded_wait(int(polls), _stream(stream)), "qz_selftest_bounded_wait")


class Workspace:
    """A reusable device scratch buffer (torch-allocated) grown on demand."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device or "cuda")
        return self.buf


def _ws(ws, nbytes, dev):
    if nbytes == 0:
        return None, 0
    if ws is None:
        ws = Workspace(torch.device("cuda", dev))
    buf = ws.get(nbytes) if isinstance(ws, Workspace) else ws
    _on(buf, "ws", dev)
    return buf, buf.numel() * buf.element_size()


# ------------------------------------------------------------- quantizers

def qz_quantize_fp8(x: torch.Tensor, gran: int, codes=None, scales=None, dequant=False, ws=None,
                    stream=None):
    """FP8 E4M3 quantization of a 2-D fp32/bf16 tensor. Returns (codes u8, scales f32,
    dequant f32 or None). `dequant` may be True (allocate) or an output tensor."""
    rows, cols, ld = _rows_cols_ld(x)
    xt, d = _dtype_code(x), _device()
    _on(x, "x", d)
    dev = x.device
    br = min(128, rows) if rows else 1
    shape = {FP8_PER_TENSOR: (1,), FP8_PER_ROW: (rows,),
             FP8_BLOCK_128x128: (rows // br, cols // 128), FP8_GROUP_1x128: (rows, cols // 128)}.get(gran)
    if shape is None:
        raise ValueError(f"unknown FP8 granularity {gran}")
    if codes is None:
        codes = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(shape, dtype=torch.float32, device=dev)
    if dequant is True:
        dequant = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    deq = dequant if isinstance(dequant, torch.Tensor) else None
    n_sc = shape[0] * (shape[1] if len(shape) > 1 else 1)
    args = (_arg(codes, "codes", d, 1, rows * cols), _arg(scales, "scales", d, torch.float32, n_sc),
            _opt(deq, "dequant", d, torch.float32, rows * cols))
    buf, nb = _ws(ws, qz_workspace_size(OP_QUANTIZE_FP8, rows, cols, gran), d)
    _check(lib.qz_quantize_fp8(x.data_ptr(), xt, rows, cols, ld, gran, *args, _ptr(buf), nb, _stream(stream)),
           "qz_quantize_fp8")
    return codes, scales, deq


def qz_quantize_mxfp4(x: torch.Tensor, codes=None, scale_e8m0=None, dequant=False, stream=None):
    """MXFP4 quantization. Returns (codes u8 [R, C/2], e8m0 u8 [R, C/32], dequant|None)."""
    rows, cols, ld = _rows_cols_ld(x)
    xt, d = _dtype_code(x), _device()
    _on(x, "x", d)
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    if scale_e8m0 is None:
        scale_e8m0 = torch.empty((rows, cols // 32), dtype=torch.uint8, device=dev)
    if dequant is True:
        dequant = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    deq = dequant if isinstance(dequant, torch.Tensor) else None
    _check(lib.qz_quantize_mxfp4(x.data_ptr(), xt, rows, cols, ld, _arg(codes, "codes", d, 1, rows * (cols // 2)),
                                 _arg(scale_e8m0, "scale_e8m0", d, 1, rows * (cols // 32)),
                                 _opt(deq, "dequant", d, torch.float32, rows * cols), _stream(stream)),
           "qz_quantize_mxfp4")
    return codes, scale_e8m0, deq


def qz_quantize_nvfp4(x: torch.Tensor, codes=None, scale_e4m3=None, global_scale=None,
                      global_amax_in=None, dequant=False, ws=None, stream=None):
    """NVFP4 quantization. Returns (codes u8 [R, C/2], block scales u8 (E4M3) [R, C/16],
    global scale f32 [1], dequant|None)."""
    rows, cols, ld = _rows_cols_ld(x)
    xt, d = _dtype_code(x), _device()
    _on(x, "x", d)
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    if scale_e4m3 is None:
        scale_e4m3 = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
    if global_scale is None:
        global_scale = torch.empty((1,), dtype=torch.float32, device=dev)
    if dequant is True:
        dequant = torch.empty((rows, cols), dtype=torch.float32, device=dev)
    deq = dequant if isinstance(dequant, torch.Tensor) else None
    args = (_arg(codes, "codes", d, 1, rows * (cols // 2)), _arg(scale_e4m3, "scale_e4m3", d, 1, rows * (cols // 16)),
            _arg(global_scale, "global_scale", d, torch.float32, 1),
            _opt(global_amax_in, "global_amax_in", d, torch.float32, 1),
            _opt(deq, "dequant", d, torch.float32, rows * cols))
    if global_amax_in is None:
        buf, nb = _ws(ws, qz_workspace_size(OP_QUANTIZE_NVFP4, rows, cols), d)
    else:
        buf, nb = None, 0
    _check(lib.qz_quantize_nvfp4(x.data_ptr(), xt, rows, cols, ld, *args, _ptr(buf), nb, _stream(stream)),
           "qz_quantize_nvfp4")
    return codes, scale_e4m3, global_scale, deq


def qz_quantize_nvfp4_grouped(xs, outs=None, ws=None, stream=None):
    """NVFP4 quantization of several contiguous 2-D tensors of one dtype in two launches.
    Returns [(codes, scale_e4m3, global_scale), ...] as qz_quantize_nvfp4 would per tensor;
    `outs` may give those buffers."""
    n = len(xs)
    arr = (_Nvfp4Tensor * n)()
    res = []
    xt = _dtype_code(xs[0]) if n else F32
    d = _device()
    for i, x in enumerate(xs):
        if x.dim() != 2 or not x.is_contiguous():
            raise ValueError("qz_quantize_nvfp4_grouped takes contiguous 2-D tensors")
        if _dtype_code(x) != xt:
            raise TypeError("qz_quantize_nvfp4_grouped takes tensors of one dtype")
        _on(x, f"xs[{i}]", d)
        rows, cols = x.shape
        if outs is not None:
            codes, sc, g = outs[i]
        else:
            codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
            sc = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
            g = torch.empty((1,), dtype=torch.float32, device=x.device)
        arr[i] = _Nvfp4Tensor(x.data_ptr(), rows, cols, _arg(codes, f"codes[{i}]", d, 1, rows * (cols // 2)),
                              _arg(sc, f"scale_e4m3[{i}]", d, 1, rows * (cols // 16)),
                              _arg(g, f"global_scale[{i}]", d, torch.float32, 1))
        res.append((codes, sc, g))
    buf, nb = _ws(ws, qz_workspace_size(OP_QUANTIZE_NVFP4_GROUPED, n) if n else 0, d)
    _check(lib.qz_quantize_nvfp4_grouped(arr, n, xt, _ptr(buf), nb, _stream(stream)),
           "qz_quantize_nvfp4_grouped")
    return res


def qz_quantize_int4_g128(w: torch.Tensor, qweight=None, scale_bf16=None, dequant=False, stream=None):
    """INT4 g128 of a [K, N] weight. Returns (qweight i32 [K/8, N], scale bf16 [K/128, N],
    dequant|None)."""
    K, N, ld = _rows_cols_ld(w)
    wt, d = _dtype_code(w), _device()
    _on(w, "w", d)
    dev = w.device
    if qweight is None:
        qweight = torch.empty((K // 8, N), dtype=torch.int32, device=dev)
    if scale_bf16 is None:
        scale_bf16 = torch.empty((K // 128, N), dtype=torch.bfloat16, device=dev)
    if dequant is True:
        dequant = torch.empty((K, N), dtype=torch.float32, device=dev)
    deq = dequant if isinstance(dequant, torch.Tensor) else None
    _check(lib.qz_quantize_int4_g128(w.data_ptr(), wt, K, N, ld, _arg(qweight, "qweight", d, 4, (K // 8) * N),
                                     _arg(scale_bf16, "scale_bf16", d, 2, (K // 128) * N),
                                     _opt(deq, "dequant", d, torch.float32, K * N), _stream(stream)),
           "qz_quantize_int4_g128")
    return qweight, scale_bf16, deq


def qz_kv_write_fp8(k: torch.Tensor, v: torch.Tensor, k_codes=None, v_codes=None, k_scale=None,
                    v_scale=None, mode: int = SCALE_COMPUTE, ws=None, stream=None):
    """FP8 per-tensor KV write of bf16 [B, H, T, D] tensors. Returns (k_codes, v_codes,
    k_scale, v_scale); in SCALE_GIVEN mode k_scale/v_scale are inputs."""
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16 or k.shape != v.shape or k.dim() != 4:
        raise ValueError("k and v must be bf16 tensors of the same [B, H, T, D] shape")
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("k and v must be contiguous")
    B, H, T, D = k.shape
    d = _device()
    _on(k, "k", d)
    _on(v, "v", d)
    dev = k.device
    if k_codes is None:
        k_codes = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    if v_codes is None:
        v_codes = torch.empty(v.shape, dtype=torch.uint8, device=dev)
    if k_scale is None:
        k_scale = torch.empty((1,), dtype=torch.float32, device=dev)
    if v_scale is None:
        v_scale = torch.empty((1,), dtype=torch.float32, device=dev)
    n = B * H * T * D
    args = (_arg(k_codes, "k_codes", d, 1, n), _arg(v_codes, "v_codes", d, 1, n),
            _arg(k_scale, "k_scale", d, torch.float32, 1), _arg(v_scale, "v_scale", d, torch.float32, 1))
    buf, nb = _ws(ws, qz_workspace_size(OP_KV_WRITE_FP8, n) if mode == SCALE_COMPUTE else 0, d)
    _check(lib.qz_kv_write_fp8(k.data_ptr(), v.data_ptr(), B, H, T, D, *args, mode, _ptr(buf), nb, _stream(stream)),
           "qz_kv_write_fp8")
    return k_codes, v_codes, k_scale, v_scale


# ------------------------------------------------------------------ GEMMs

def qz_gemm_w4a16(A: torch.Tensor, qweight: torch.Tensor, scale_bf16: torch.Tensor, Y=None, ws=None,
                  stream=None):
    """Y[M, N] (bf16) = A[M, K] (bf16) @ dequant(INT4 g128 weight)."""
    M, K = A.shape
    N = qweight.shape[1]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    args = (_arg(A, "A", d, torch.bfloat16), _arg(qweight, "qweight", d, 4, (K // 8) * N),
            _arg(scale_bf16, "scale_bf16", d, 2, (K // 128) * N), _arg(Y, "Y", d, torch.bfloat16, M * N))
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_W4A16, M, N, K), d)
    _check(lib.qz_gemm_w4a16(*args, M, N, K, _ptr(buf), nb, _stream(stream)), "qz_gemm_w4a16")
    return Y


def qz_gemm_w4a16_grouped(problems, ws=None, stream=None):
    """Run independent W4A16 problems [(A, qweight, scale_bf16, Y), ...] in one launch."""
    arr = (_W4A16Problem * len(problems))()
    mmax = kmax = nsum = 0
    d = _device()
    for i, (A, qw, sc, Y) in enumerate(problems):
        M, K = A.shape
        N = qw.shape[1]
        arr[i] = _W4A16Problem(_arg(A, f"A[{i}]", d, torch.bfloat16), _arg(qw, f"qweight[{i}]", d, 4, (K // 8) * N),
                               _arg(sc, f"scale_bf16[{i}]", d, 2, (K // 128) * N),
                               _arg(Y, f"Y[{i}]", d, torch.bfloat16, M * N), M, N, K)
        mmax, kmax, nsum = max(mmax, M), max(kmax, K), nsum + N
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_W4A16, mmax, nsum, kmax), d)
    _check(lib.qz_gemm_w4a16_grouped(arr, len(problems), _ptr(buf), nb, _stream(stream)),
           "qz_gemm_w4a16_grouped")


def qz_gemm_fp8_block(qA, sA, qB, sB, Y=None, ws=None, stream=None):
    """Y[M, N] (bf16) from E4M3 qA [M, K] with 1x128 scales sA and E4M3 qB = B^T [N, K]
    with 128x128 scales sB."""
    M, K = qA.shape
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=qA.device)
    args = (_arg(qA, "qA", d, 1), _arg(sA, "sA", d, torch.float32, M * (K // 128)), _arg(qB, "qB", d, 1, N * K),
            _arg(sB, "sB", d, torch.float32, (N // 128) * (K // 128)), _arg(Y, "Y", d, torch.bfloat16, M * N))
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_FP8_BLOCK, M, N, K), d)
    _check(lib.qz_gemm_fp8_block(*args, M, N, K, _ptr(buf), nb, _stream(stream)), "qz_gemm_fp8_block")
    return Y


def qz_gemm_nvfp4(qA, sA, gA, qB, sB, gB, Y=None, ws=None, stream=None):
    """Y[M, N] (bf16) from NVFP4 A [M, K] and B^T [N, K] (codes, E4M3 block scales, fp32
    tensor scale each)."""
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=qA.device)
    args = (_arg(qA, "qA", d, 1, M * K // 2), _arg(sA, "sA", d, 1, M * (K // 16)), _arg(gA, "gA", d, torch.float32, 1),
            _arg(qB, "qB", d, 1, N * K // 2), _arg(sB, "sB", d, 1, N * (K // 16)), _arg(gB, "gB", d, torch.float32, 1),
            _arg(Y, "Y", d, torch.bfloat16, M * N))
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_NVFP4, M, N, K), d)
    _check(lib.qz_gemm_nvfp4(*args, M, N, K, _ptr(buf), nb, _stream(stream)), "qz_gemm_nvfp4")
    return Y


def qz_gemm_nvfp4_quant(qA, sA, gA, qB, sB, gB, y_amax, y_codes=None, y_scales=None, y_global=None, ws=None,
                        stream=None):
    """NVFP4 GEMM whose output leaves quantized to NVFP4 with the given tensor amax
    (device fp32 scalar). Returns (codes u8 [M, N/2], E4M3 block scales u8 [M, N/16],
    tensor scale fp32 [1]): what qz_quantize_nvfp4 gives for the bf16 output with that
    amax."""
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    d = _device()
    dev = qA.device
    if y_codes is None:
        y_codes = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    if y_scales is None:
        y_scales = torch.empty((M, N // 16), dtype=torch.uint8, device=dev)
    if y_global is None:
        y_global = torch.empty((1,), dtype=torch.float32, device=dev)
    args = (_arg(qA, "qA", d, 1, M * K // 2), _arg(sA, "sA", d, 1, M * (K // 16)), _arg(gA, "gA", d, torch.float32, 1),
            _arg(qB, "qB", d, 1, N * K // 2), _arg(sB, "sB", d, 1, N * (K // 16)), _arg(gB, "gB", d, torch.float32, 1),
            _arg(y_amax, "y_amax", d, torch.float32, 1), _arg(y_codes, "y_codes", d, 1, M * N // 2),
            _arg(y_scales, "y_scales", d, 1, M * N // 16), _arg(y_global, "y_global", d, torch.float32, 1))
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_NVFP4, M, N, K), d)
    _check(lib.qz_gemm_nvfp4_quant(*args, M, N, K, _ptr(buf), nb, _stream(stream)), "qz_gemm_nvfp4_quant")
    return y_codes, y_scales, y_global


def qz_gemm_mxfp4_quant(qA, eA, qB, eB, y_codes=None, y_e8m0=None, ws=None, stream=None):
    """MXFP4 GEMM whose output leaves quantized to MXFP4. Returns (codes u8 [M, N/2], E8M0
    scales u8 [M, N/32]): what qz_quantize_mxfp4 gives for the bf16 output."""
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    d = _device()
    dev = qA.device
    if y_codes is None:
        y_codes = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    if y_e8m0 is None:
        y_e8m0 = torch.empty((M, N // 32), dtype=torch.uint8, device=dev)
    args = (_arg(qA, "qA", d, 1, M * K // 2), _arg(eA, "eA", d, 1, M * (K // 32)),
            _arg(qB, "qB", d, 1, N * K // 2), _arg(eB, "eB", d, 1, N * (K // 32)),
            _arg(y_codes, "y_codes", d, 1, M * N // 2), _arg(y_e8m0, "y_e8m0", d, 1, M * N // 32))
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_MXFP4, M, N, K), d)
    _check(lib.qz_gemm_mxfp4_quant(*args, M, N, K, _ptr(buf), nb, _stream(stream)), "qz_gemm_mxfp4_quant")
    return y_codes, y_e8m0


def qz_gemm_nvfp4_noalloc(qA, sA, gA, qB, sB, gB, Y=None, stream=None):
    """qz_gemm_nvfp4 without a workspace: the re-laid scale factors live in the library's
    fixed device array (see include/qz.h), so calls that may overlap on the GPU must be
    serialised by the caller."""
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=qA.device)
    args = (_arg(qA, "qA", d, 1, M * K // 2), _arg(sA, "sA", d, 1, M * (K // 16)), _arg(gA, "gA", d, torch.float32, 1),
            _arg(qB, "qB", d, 1, N * K // 2), _arg(sB, "sB", d, 1, N * (K // 16)), _arg(gB, "gB", d, torch.float32, 1),
            _arg(Y, "Y", d, torch.bfloat16, M * N))
    _check(lib.qz_gemm_nvfp4_noalloc(*args, M, N, K, _stream(stream)), "qz_gemm_nvfp4_noalloc")
    return Y


def qz_gemm_mxfp4(qA, eA, qB, eB, Y=None, ws=None, stream=None):
    """Y[M, N] (bf16) from MXFP4 A [M, K] and B^T [N, K] (codes, E8M0 block scales)."""
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=qA.device)
    args = (_arg(qA, "qA", d, 1, M * K // 2), _arg(eA, "eA", d, 1, M * (K // 32)), _arg(qB, "qB", d, 1, N * K // 2),
            _arg(eB, "eB", d, 1, N * (K // 32)), _arg(Y, "Y", d, torch.bfloat16, M * N))
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_MXFP4, M, N, K), d)
    _check(lib.qz_gemm_mxfp4(*args, M, N, K, _ptr(buf), nb, _stream(stream)), "qz_gemm_mxfp4")
    return Y


def qz_prepare_fp4_scales(scales, K: int, nv: bool = True, out=None, stream=None):
    """Block scales [rows, K/16] (NVFP4) or [rows, K/32] (MXFP4), row-major uint8, re-laid
    into the tensor cores' scale-factor order (rows padded to a multiple of 128)."""
    rows = scales.shape[0]
    d = _device()
    n_out = qz_workspace_size(OP_PREPARE_FP4_SCALES, rows, K, int(nv))
    if out is None:
        out = torch.empty(n_out, dtype=torch.uint8, device=scales.device)
    _check(lib.qz_prepare_fp4_scales(_arg(scales, "scales", d, 1, rows * (K // (16 if nv else 32))), rows, K,
                                     int(nv), _arg(out, "out", d, 1, n_out), _stream(stream)),
           "qz_prepare_fp4_scales")
    return out


def qz_gemm_nvfp4_grouped(problems, ws=None, stream=None):
    """Run independent NVFP4 problems [(qA, sA, gA, qB, sB_prepared, gB, Y), ...] (decode
    shapes, M <= 128) with one scale re-layout launch and one GEMM launch per 72 problems."""
    arr = (_Nvfp4Problem * len(problems))()
    kmax = 0
    d = _device()
    for i, (qA, sA, gA, qB, sBp, gB, Y) in enumerate(problems):
        M, K = qA.shape[0], qA.shape[1] * 2
        N = qB.shape[0]
        arr[i] = _Nvfp4Problem(_arg(qA, f"qA[{i}]", d, 1, M * K // 2), _arg(sA, f"sA[{i}]", d, 1, M * (K // 16)),
                               _arg(gA, f"gA[{i}]", d, torch.float32, 1), _arg(qB, f"qB[{i}]", d, 1, N * K // 2),
                               _arg(sBp, f"sB_prepared[{i}]", d, 1,
                                    qz_workspace_size(OP_PREPARE_FP4_SCALES, N, K, 1)),
                               _arg(gB, f"gB[{i}]", d, torch.float32, 1),
                               _arg(Y, f"Y[{i}]", d, torch.bfloat16, M * N), M, N, K)
        kmax = max(kmax, K)
    buf, nb = _ws(ws, qz_workspace_size(OP_GEMM_NVFP4_GROUPED, len(problems), kmax), d)
    _check(lib.qz_gemm_nvfp4_grouped(arr, len(problems), _ptr(buf), nb, _stream(stream)),
           "qz_gemm_nvfp4_grouped")


# ------------------------------------------------ variants of the base formats

def _kv_inputs(k, v):
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16 or k.shape != v.shape or k.dim() != 4:
        raise ValueError("k and v must be bf16 tensors of the same [B, H, T, D] shape")
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("k and v must be contiguous")
    d = _device()
    _on(k, "k", d)
    _on(v, "v", d)
    return d


def qz_kv_write_fp8_per_head(k: torch.Tensor, v: torch.Tensor, k_codes=None, v_codes=None, k_scale=None,
                             v_scale=None, mode: int = SCALE_COMPUTE, ws=None, stream=None):
    """FP8 KV write with one scale per (batch, head) of bf16 [B, H, T, D] tensors.
    Returns (k_codes, v_codes, k_scale [B, H], v_scale [B, H]); in SCALE_GIVEN mode the
    scales are inputs."""
    d = _kv_inputs(k, v)
    B, H, T, D = k.shape
    dev = k.device
    k_codes = torch.empty(k.shape, dtype=torch.uint8, device=dev) if k_codes is None else k_codes
    v_codes = torch.empty(v.shape, dtype=torch.uint8, device=dev) if v_codes is None else v_codes
    k_scale = torch.empty((B, H), dtype=torch.float32, device=dev) if k_scale is None else k_scale
    v_scale = torch.empty((B, H), dtype=torch.float32, device=dev) if v_scale is None else v_scale
    n = B * H * T * D
    args = (_arg(k_codes, "k_codes", d, 1, n), _arg(v_codes, "v_codes", d, 1, n),
            _arg(k_scale, "k_scale", d, torch.float32, B * H), _arg(v_scale, "v_scale", d, torch.float32, B * H))
    need = qz_workspace_size(OP_KV_WRITE_FP8_PER_HEAD, B * H, T * D) if mode == SCALE_COMPUTE else 0
    buf, nb = _ws(ws, need, d)
    _check(lib.qz_kv_write_fp8_per_head(k.data_ptr(), v.data_ptr(), B, H, T, D, *args, mode, _ptr(buf), nb,
                                        _stream(stream)), "qz_kv_write_fp8_per_head")
    return k_codes, v_codes, k_scale, v_scale


def qz_kv_write_fp8_channel_zp(k: torch.Tensor, v: torch.Tensor, k_codes=None, v_codes=None, k_scale=None,
                               k_zero=None, v_scale=None, ws=None, stream=None):
    """FP8 KV write with K per channel and a zero point (over the tokens) and V per token.
    Returns (k_codes, v_codes, k_scale [B, H, D], k_zero [B, H, D], v_scale [B, H, T])."""
    d = _kv_inputs(k, v)
    B, H, T, D = k.shape
    dev = k.device
    k_codes = torch.empty(k.shape, dtype=torch.uint8, device=dev) if k_codes is None else k_codes
    v_codes = torch.empty(v.shape, dtype=torch.uint8, device=dev) if v_codes is None else v_codes
    k_scale = torch.empty((B, H, D), dtype=torch.float32, device=dev) if k_scale is None else k_scale
    k_zero = torch.empty((B, H, D), dtype=torch.float32, device=dev) if k_zero is None else k_zero
    v_scale = torch.empty((B, H, T), dtype=torch.float32, device=dev) if v_scale is None else v_scale
    n = B * H * T * D
    args = (_arg(k_codes, "k_codes", d, 1, n), _arg(v_codes, "v_codes", d, 1, n),
            _arg(k_scale, "k_scale", d, torch.float32, B * H * D), _arg(k_zero, "k_zero", d, torch.float32, B * H * D),
            _arg(v_scale, "v_scale", d, torch.float32, B * H * T))
    buf, nb = _ws(ws, qz_workspace_size(OP_KV_WRITE_FP8_CHANNEL_ZP, B * H, T, D), d)
    _check(lib.qz_kv_write_fp8_channel_zp(k.data_ptr(), v.data_ptr(), B, H, T, D, *args, _ptr(buf), nb,
                                          _stream(stream)), "qz_kv_write_fp8_channel_zp")
    return k_codes, v_codes, k_scale, k_zero, v_scale


def qz_quantize_int4_g128_zp(w: torch.Tensor, qweight=None, scale_bf16=None, zero=None, dequant=False, stream=None):
    """INT4 with a zero point (codes 0..15) of a [K, N] weight. Returns (qweight i32 [K/8, N],
    scale bf16 [K/128, N], zero u8 [K/128, N], dequant f32 [K, N] or None)."""
    K, N, ld = _rows_cols_ld(w)
    wt = _dtype_code(w)
    d = _device()
    _on(w, "w", d)
    if qweight is None:
        qweight = torch.empty((K // 8, N), dtype=torch.int32, device=w.device)
    if scale_bf16 is None:
        scale_bf16 = torch.empty((K // 128, N), dtype=torch.bfloat16, device=w.device)
    if zero is None:
        zero = torch.empty((K // 128, N), dtype=torch.uint8, device=w.device)
    deq = torch.empty((K, N), dtype=torch.float32, device=w.device) if dequant else None
    _check(lib.qz_quantize_int4_g128_zp(w.data_ptr(), wt, K, N, ld, _arg(qweight, "qweight", d, 4, (K // 8) * N),
                                        _arg(scale_bf16, "scale_bf16", d, 2, (K // 128) * N),
                                        _arg(zero, "zero", d, 1, (K // 128) * N),
                                        _opt(deq, "dequant", d, torch.float32, K * N), _stream(stream)),
           "qz_quantize_int4_g128_zp")
    return qweight, scale_bf16, zero, deq


def qz_gemm_w4a16_zp(A: torch.Tensor, qweight, scale_bf16, zero, Y=None, stream=None):
    """Y[M, N] (bf16) = A[M, K] (bf16) @ dequant(INT4 weight with zero points), M <= 16."""
    M, K = A.shape
    N = qweight.shape[1]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    args = (_arg(A, "A", d, torch.bfloat16), _arg(qweight, "qweight", d, 4, (K // 8) * N),
            _arg(scale_bf16, "scale_bf16", d, 2, (K // 128) * N), _arg(zero, "zero", d, 1, (K // 128) * N),
            _arg(Y, "Y", d, torch.bfloat16, M * N))
    _check(lib.qz_gemm_w4a16_zp(*args, M, N, K, _stream(stream)), "qz_gemm_w4a16_zp")
    return Y


def qz_gemm_w4a16_nvfp4(A: torch.Tensor, qB, sB, gB, Y=None, stream=None):
    """Weight-only NVFP4: Y[M, N] (bf16) = A[M, K] (bf16) @ dequant(B^T [N, K]), M <= 16."""
    M, K = A.shape
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    args = (_arg(A, "A", d, torch.bfloat16), _arg(qB, "qB", d, 1, N * K // 2), _arg(sB, "sB", d, 1, N * (K // 16)),
            _arg(gB, "gB", d, torch.float32, 1), _arg(Y, "Y", d, torch.bfloat16, M * N))
    _check(lib.qz_gemm_w4a16_nvfp4(*args, M, N, K, _stream(stream)), "qz_gemm_w4a16_nvfp4")
    return Y


def qz_gemm_w4a16_mxfp4(A: torch.Tensor, qB, eB, Y=None, stream=None):
    """Weight-only MXFP4: Y[M, N] (bf16) = A[M, K] (bf16) @ dequant(B^T [N, K]), M <= 16."""
    M, K = A.shape
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    args = (_arg(A, "A", d, torch.bfloat16), _arg(qB, "qB", d, 1, N * K // 2), _arg(eB, "eB", d, 1, N * (K // 32)),
            _arg(Y, "Y", d, torch.bfloat16, M * N))
    _check(lib.qz_gemm_w4a16_mxfp4(*args, M, N, K, _stream(stream)), "qz_gemm_w4a16_mxfp4")
    return Y


def qz_col_amax(x: torch.Tensor, out=None, ws=None, stream=None):
    """max |x[r, c]| over the rows of each column of a contiguous 2-D fp32/bf16 tensor."""
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("qz_col_amax takes a contiguous 2-D tensor")
    rows, cols = x.shape
    d = _device()
    _on(x, "x", d)
    if out is None:
        out = torch.empty((cols,), dtype=torch.float32, device=x.device)
    buf, nb = _ws(ws, qz_workspace_size(OP_COL_AMAX, rows, cols), d)
    _check(lib.qz_col_amax(x.data_ptr(), _dtype_code(x), rows, cols, _arg(out, "out", d, torch.float32, cols),
                           _ptr(buf), nb, _stream(stream)), "qz_col_amax")
    return out


def qz_smooth_factors(x_amax: torch.Tensor, w_amax: torch.Tensor, alpha: float = 0.5, out=None, stream=None):
    """SmoothQuant migration factors s_j = max|X_j|^a / max|W_j|^(1-a), a = 0.5."""
    n = x_amax.numel()
    d = _device()
    if out is None:
        out = torch.empty((n,), dtype=torch.float32, device=x_amax.device)
    _check(lib.qz_smooth_factors(_arg(x_amax, "x_amax", d, torch.float32, n), _arg(w_amax, "w_amax", d, torch.float32, n),
                                 n, float(alpha), _arg(out, "out", d, torch.float32, n), _stream(stream)),
           "qz_smooth_factors")
    return out


def qz_quantize_int8_rows(x: torch.Tensor, factors=None, op: int = SMOOTH_NONE, codes=None, scales=None,
                          dequant=False, stream=None):
    """INT8 per row of a contiguous 2-D fp32/bf16 tensor after the optional per-column
    SmoothQuant factor (SMOOTH_DIVIDE for activations, SMOOTH_MULTIPLY for weights as
    B^T). Returns (codes int8 [R, C], scales f32 [R], dequant f32 or None)."""
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("qz_quantize_int8_rows takes a contiguous 2-D tensor")
    rows, cols = x.shape
    d = _device()
    _on(x, "x", d)
    codes = torch.empty((rows, cols), dtype=torch.int8, device=x.device) if codes is None else codes
    scales = torch.empty((rows,), dtype=torch.float32, device=x.device) if scales is None else scales
    deq = torch.empty((rows, cols), dtype=torch.float32, device=x.device) if dequant else None
    _check(lib.qz_quantize_int8_rows(x.data_ptr(), _dtype_code(x), rows, cols,
                                     _opt(factors, "factors", d, torch.float32, cols), int(op),
                                     _arg(codes, "codes", d, 1, rows * cols), _arg(scales, "scales", d, torch.float32, rows),
                                     _opt(deq, "dequant", d, torch.float32, rows * cols), _stream(stream)),
           "qz_quantize_int8_rows")
    return codes, scales, deq


def qz_gemm_int8(qA, sA, qB, sB, Y=None, stream=None):
    """Y[M, N] (bf16) = diag(sA) (qA qB^T) diag(sB): INT8 A [M, K] and B^T [N, K]."""
    M, K = qA.shape
    N = qB.shape[0]
    d = _device()
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=qA.device)
    args = (_arg(qA, "qA", d, 1, M * K), _arg(sA, "sA", d, torch.float32, M), _arg(qB, "qB", d, 1, N * K),
            _arg(sB, "sB", d, torch.float32, N), _arg(Y, "Y", d, torch.bfloat16, M * N))
    _check(lib.qz_gemm_int8(*args, M, N, K, _stream(stream)), "qz_gemm_int8")
    return Y


def qz_gemm_fp8_block_quant(qA, sA, qB, sB, Y=None, y_codes=None, y_scales=None, want_y: bool = False, stream=None):
    """The FP8 block-scaled GEMM with the output quantized to FP8 1x128 in its epilogue.
    Returns (y_codes u8 [M, N], y_scales f32 [M, N/128], Y bf16 [M, N] or None)."""
    M, K = qA.shape
    N = qB.shape[0]
    d = _device()
    if y_codes is None:
        y_codes = torch.empty((M, N), dtype=torch.uint8, device=qA.device)
    if y_scales is None:
        y_scales = torch.empty((M, N // 128), dtype=torch.float32, device=qA.device)
    if Y is None and want_y:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=qA.device)
    args = (_arg(qA, "qA", d, 1, M * K), _arg(sA, "sA", d, torch.float32, M * (K // 128)), _arg(qB, "qB", d, 1, N * K),
            _arg(sB, "sB", d, torch.float32, (N // 128) * (K // 128)), _opt(Y, "Y", d, torch.bfloat16, M * N),
            _arg(y_codes, "y_codes", d, 1, M * N), _arg(y_scales, "y_scales", d, torch.float32, M * (N // 128)))
    _check(lib.qz_gemm_fp8_block_quant(*args, M, N, K, _stream(stream)), "qz_gemm_fp8_block_quant")
    return y_codes, y_scales, Y

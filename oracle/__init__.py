"""CPU oracle for the quantizers and quantized GEMMs (ctypes over qz_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's
CPU-baseline leg use it. The CUDA library never imports, links or calls it,
and it shares no code with the CUDA path.

Every wrapper takes and returns numpy arrays. bf16 data travels as uint16 bit
patterns. The C file states, for each function, the passage of the pages it
follows and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qz_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libqz_oracle.so")
_lock = threading.Lock()
_lib = None

FP8_PER_TENSOR, FP8_PER_ROW, FP8_BLOCK_128x128, FP8_GROUP_1x128 = 0, 1, 2, 3


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile qz_oracle.c (or another copy of it, `src`, into `out`) with gcc:
    single-threaded, no FMA contraction."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sigs = {
            "or_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "or_e4m3_encode": (ctypes.c_uint8, [F]),
            "or_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "or_e2m1_encode": (ctypes.c_uint8, [F]),
            "or_bf16_to_f32": (F, [ctypes.c_uint16]),
            "or_f32_to_bf16": (ctypes.c_uint16, [F]),
            "or_int_quant_one": (I, [F, F, I, I, P]),
            "or_amax": (F, [P, I, I64, I64, I64]),
            "or_quant_fp8": (I, [P, I, I64, I64, I64, I, P, P, P]),
            "or_quant_fp8_given": (None, [P, I, I64, F, P, P]),
            "or_kv_write_fp8": (None, [P, P, I64, P, P, P, P, P, P]),
            "or_quant_mxfp4": (I, [P, I, I64, I64, I64, P, P, P]),
            "or_quant_nvfp4": (I, [P, I, I64, I64, I64, P, P, P, P, P]),
            "or_quant_int4_g128": (I, [P, I, I64, I64, I64, P, P, P]),
            "or_gemm_w4a16": (None, [P, P, P, I64, I64, I64, P, P, I64, P, P]),
            "or_gemm_fp8_block": (None, [P, P, P, P, I64, I64, I64, P, P, I64, P, P]),
            "or_gemm_nvfp4": (None, [P, P, F, P, P, F, I64, I64, I64, P, P, I64, P, P]),
            "or_gemm_mxfp4": (None, [P, P, P, P, I64, I64, I64, P, P, I64, P, P]),
            "or_kv_write_fp8_per_head": (None, [P, P, I64, I64, P, P, P, P, P, P]),
            "or_kv_fp8_per_head_given": (None, [P, I64, I64, P, P, P]),
            "or_kv_k_channel_zp": (None, [P, I64, I64, I64, P, P, P, P]),
            "or_quant_int4_g128_zp": (I, [P, I, I64, I64, I64, P, P, P, P]),
            "or_gemm_w4a16_zp": (None, [P, P, P, P, I64, I64, I64, P, P, I64, P, P]),
            "or_gemm_w4a16_nvfp4": (None, [P, P, P, F, I64, I64, I64, P, P, I64, P, P]),
            "or_gemm_w4a16_mxfp4": (None, [P, P, P, I64, I64, I64, P, P, I64, P, P]),
            "or_col_amax": (None, [P, I, I64, I64, P]),
            "or_smooth_factors": (None, [P, P, I64, P]),
            "or_quant_int8_rows": (I, [P, I, I64, I64, P, I, P, P, P]),
            "or_gemm_int8": (None, [P, P, P, P, I64, I64, I64, P, P, I64, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _src(x):
    """(contiguous array, is_bf16) for fp32 arrays or uint16 bf16 bit patterns."""
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), 1
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), 0
    raise TypeError(f"oracle input must be float32 or bf16 bits (uint16), got {x.dtype}")


# ----------------------------------------------------------------- codecs

def e4m3_decode(code: int) -> float:
    return _load().or_e4m3_decode(int(code))


def e4m3_encode(y: float) -> int:
    return int(_load().or_e4m3_encode(float(y)))


def e2m1_decode(code: int) -> float:
    return _load().or_e2m1_decode(int(code))


def e2m1_encode(y: float) -> int:
    return int(_load().or_e2m1_encode(float(y)))


def f32_to_bf16(f: float) -> int:
    return int(_load().or_f32_to_bf16(float(f)))


def bf16_to_f32(b: int) -> float:
    return float(_load().or_bf16_to_f32(int(b)))


def e4m3_encode_array(y: np.ndarray) -> np.ndarray:
    """Element-wise E4M3 encode of an fp32 array (per-tensor FP8 with scale 1, no clamp
    needed below 448): uses the given-scale path with scale 1.0."""
    y = np.ascontiguousarray(y, dtype=np.float32).ravel()
    codes = np.empty(y.size, np.uint8)
    _load().or_quant_fp8_given(_ptr(y), 0, y.size, 1.0, _ptr(codes), None)
    return codes


def int_quant_one(x: float, s: float, qmin: int, qmax: int):
    """(q, dequant) of one value: q = clamp(rint(x / s), qmin, qmax), x^ = q * s."""
    d = ctypes.c_float()
    q = _load().or_int_quant_one(float(x), float(s), int(qmin), int(qmax), ctypes.byref(d))
    return int(q), float(d.value)


# ------------------------------------------------------------- quantizers

def amax(x: np.ndarray) -> float:
    x2, bf = _src(x)
    rows, cols = x2.shape
    return float(_load().or_amax(_ptr(x2), bf, rows, cols, cols))


def quant_fp8(x: np.ndarray, gran: int, want_deq: bool = True):
    """FP8 E4M3 fake-quant of a 2-D array. Returns (codes u8 [R,C], scales f32, deq f32|None).
    Scale shapes: tensor (1,), row (R,), 128x128 (R/br, C/128), 1x128 (R, C/128)."""
    x2, bf = _src(x)
    rows, cols = x2.shape
    if gran == FP8_PER_TENSOR:
        sshape = (1,)
    elif gran == FP8_PER_ROW:
        sshape = (rows,)
    elif gran == FP8_BLOCK_128x128:
        sshape = (rows // min(128, rows), cols // 128)
    elif gran == FP8_GROUP_1x128:
        sshape = (rows, cols // 128)
    else:
        raise ValueError(gran)
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty(sshape, np.float32)
    deq = np.empty((rows, cols), np.float32) if want_deq else None
    rc = _load().or_quant_fp8(_ptr(x2), bf, rows, cols, cols, gran, _ptr(codes), _ptr(scales), _ptr(deq))
    if rc != 0:
        raise ValueError(f"oracle rejects shape {x2.shape} for FP8 granularity {gran}")
    return codes, scales, deq


def quant_fp8_given(x: np.ndarray, scale: float, want_deq: bool = True):
    x2, bf = _src(x)
    x1 = x2.ravel()
    codes = np.empty(x1.size, np.uint8)
    deq = np.empty(x1.size, np.float32) if want_deq else None
    _load().or_quant_fp8_given(_ptr(x1), bf, x1.size, float(scale), _ptr(codes), _ptr(deq))
    return codes.reshape(x.shape), (deq.reshape(x.shape) if want_deq else None)


def kv_write_fp8(k: np.ndarray, v: np.ndarray, want_deq: bool = False):
    """FP8 per-tensor KV write of bf16 bit arrays. Returns (k_codes, v_codes, k_scale,
    v_scale, k_deq, v_deq)."""
    assert k.dtype == np.uint16 and v.dtype == np.uint16 and k.shape == v.shape
    k1, v1 = np.ascontiguousarray(k).ravel(), np.ascontiguousarray(v).ravel()
    kc, vc = np.empty(k1.size, np.uint8), np.empty(v1.size, np.uint8)
    ks, vs = np.empty(1, np.float32), np.empty(1, np.float32)
    kd = np.empty(k1.size, np.float32) if want_deq else None
    vd = np.empty(v1.size, np.float32) if want_deq else None
    _load().or_kv_write_fp8(_ptr(k1), _ptr(v1), k1.size, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                            _ptr(kd), _ptr(vd))
    shp = k.shape
    return (kc.reshape(shp), vc.reshape(shp), float(ks[0]), float(vs[0]),
            kd.reshape(shp) if want_deq else None, vd.reshape(shp) if want_deq else None)


def quant_mxfp4(x: np.ndarray, want_deq: bool = True):
    """Returns (codes u8 [R, C/2], e8m0 u8 [R, C/32], deq f32|None)."""
    x2, bf = _src(x)
    rows, cols = x2.shape
    codes = np.empty((rows, cols // 2), np.uint8)
    e8 = np.empty((rows, cols // 32), np.uint8)
    deq = np.empty((rows, cols), np.float32) if want_deq else None
    rc = _load().or_quant_mxfp4(_ptr(x2), bf, rows, cols, cols, _ptr(codes), _ptr(e8), _ptr(deq))
    if rc != 0:
        raise ValueError(f"oracle rejects shape {x2.shape} for MXFP4")
    return codes, e8, deq


def quant_nvfp4(x: np.ndarray, amax_in: float | None = None, want_deq: bool = True):
    """Returns (codes u8 [R, C/2], block scales e4m3 u8 [R, C/16], g f32, deq f32|None)."""
    x2, bf = _src(x)
    rows, cols = x2.shape
    codes = np.empty((rows, cols // 2), np.uint8)
    sb = np.empty((rows, cols // 16), np.uint8)
    g = np.empty(1, np.float32)
    deq = np.empty((rows, cols), np.float32) if want_deq else None
    am = None if amax_in is None else np.array([amax_in], np.float32)
    rc = _load().or_quant_nvfp4(_ptr(x2), bf, rows, cols, cols, _ptr(am), _ptr(codes), _ptr(sb),
                                _ptr(g), _ptr(deq))
    if rc != 0:
        raise ValueError(f"oracle rejects shape {x2.shape} for NVFP4")
    return codes, sb, float(g[0]), deq


def quant_int4_g128(w: np.ndarray, want_deq: bool = True):
    """INT4 g128 of a [K, N] weight. Returns (qweight i32 [K/8, N], scale bf16 bits [K/128, N],
    deq f32 [K, N]|None)."""
    w2, bf = _src(w)
    K, N = w2.shape
    qw = np.empty((K // 8, N), np.int32)
    sc = np.empty((K // 128, N), np.uint16)
    deq = np.empty((K, N), np.float32) if want_deq else None
    rc = _load().or_quant_int4_g128(_ptr(w2), bf, K, N, N, _ptr(qw), _ptr(sc), _ptr(deq))
    if rc != 0:
        raise ValueError(f"oracle rejects shape {w2.shape} for INT4 g128")
    return qw, sc, deq


# ------------------------------------------------------------------ GEMMs

def _points(M, N, ii, jj):
    if ii is None:
        ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ii = np.ascontiguousarray(np.asarray(ii, dtype=np.int64).ravel())
    jj = np.ascontiguousarray(np.asarray(jj, dtype=np.int64).ravel())
    return ii, jj


def _run_gemm(fn, args, M, N, ii, jj, full):
    ii, jj = _points(M, N, ii, jj)
    y = np.empty(ii.size, np.float64)
    b = np.empty(ii.size, np.float64)
    fn(*args, ii.ctypes.data_as(ctypes.c_void_p), jj.ctypes.data_as(ctypes.c_void_p), ii.size,
       _ptr(y), _ptr(b))
    if full:
        return y.reshape(M, N), b.reshape(M, N)
    return y, b


def gemm_w4a16(A_bf16, qweight, scale_bf16, ii=None, jj=None):
    """y, bound (double) of Y = A @ dequant(W) at the points (ii, jj), or all points."""
    A = np.ascontiguousarray(A_bf16, dtype=np.uint16)
    qw = np.ascontiguousarray(qweight, dtype=np.int32)
    sc = np.ascontiguousarray(scale_bf16, dtype=np.uint16)
    M, K = A.shape
    N = qw.shape[1]
    return _run_gemm(_load().or_gemm_w4a16, (_ptr(A), _ptr(qw), _ptr(sc), M, N, K), M, N, ii, jj,
                     ii is None)


def gemm_fp8_block(qA, sA, qB, sB, ii=None, jj=None):
    qA, qB = np.ascontiguousarray(qA, np.uint8), np.ascontiguousarray(qB, np.uint8)
    sA, sB = np.ascontiguousarray(sA, np.float32), np.ascontiguousarray(sB, np.float32)
    M, K = qA.shape
    N = qB.shape[0]
    return _run_gemm(_load().or_gemm_fp8_block, (_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB), M, N, K),
                     M, N, ii, jj, ii is None)


def gemm_nvfp4(qA, sA, gA, qB, sB, gB, ii=None, jj=None):
    qA, qB = np.ascontiguousarray(qA, np.uint8), np.ascontiguousarray(qB, np.uint8)
    sA, sB = np.ascontiguousarray(sA, np.uint8), np.ascontiguousarray(sB, np.uint8)
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    return _run_gemm(_load().or_gemm_nvfp4,
                     (_ptr(qA), _ptr(sA), float(gA), _ptr(qB), _ptr(sB), float(gB), M, N, K),
                     M, N, ii, jj, ii is None)


def gemm_mxfp4(qA, eA, qB, eB, ii=None, jj=None):
    qA, qB = np.ascontiguousarray(qA, np.uint8), np.ascontiguousarray(qB, np.uint8)
    eA, eB = np.ascontiguousarray(eA, np.uint8), np.ascontiguousarray(eB, np.uint8)
    M, K = qA.shape[0], qA.shape[1] * 2
    N = qB.shape[0]
    return _run_gemm(_load().or_gemm_mxfp4, (_ptr(qA), _ptr(eA), _ptr(qB), _ptr(eB), M, N, K),
                     M, N, ii, jj, ii is None)



# ------------------------------------------------------------ next rows

def kv_write_fp8_per_head(k: np.ndarray, v: np.ndarray, want_deq: bool = False):
    """FP8 KV write with one scale per (batch, head) of bf16 bit arrays [B, H, T, D].
    Returns (k_codes, v_codes, k_scales [B, H], v_scales [B, H], k_deq, v_deq)."""
    assert k.dtype == np.uint16 and v.dtype == np.uint16 and k.shape == v.shape and k.ndim == 4
    B, H, T, D = k.shape
    k1, v1 = np.ascontiguousarray(k), np.ascontiguousarray(v)
    kc, vc = np.empty(k.shape, np.uint8), np.empty(k.shape, np.uint8)
    ks, vs = np.empty((B, H), np.float32), np.empty((B, H), np.float32)
    kd = np.empty(k.shape, np.float32) if want_deq else None
    vd = np.empty(k.shape, np.float32) if want_deq else None
    _load().or_kv_write_fp8_per_head(_ptr(k1), _ptr(v1), B * H, T * D, _ptr(kc), _ptr(vc), _ptr(ks),
                                     _ptr(vs), _ptr(kd), _ptr(vd))
    return kc, vc, ks, vs, kd, vd


def kv_fp8_per_head_given(x: np.ndarray, scales: np.ndarray, want_deq: bool = False):
    """Per-head FP8 codes of bf16 bits [B, H, T, D] with given scales [B, H]."""
    assert x.dtype == np.uint16 and x.ndim == 4
    B, H, T, D = x.shape
    x1 = np.ascontiguousarray(x)
    sc = np.ascontiguousarray(scales, np.float32).reshape(B * H)
    codes = np.empty(x.shape, np.uint8)
    deq = np.empty(x.shape, np.float32) if want_deq else None
    _load().or_kv_fp8_per_head_given(_ptr(x1), B * H, T * D, _ptr(sc), _ptr(codes), _ptr(deq))
    return codes, deq


def kv_k_channel_zp(k: np.ndarray, want_deq: bool = False):
    """K per channel with a zero point (FP8 residual) of bf16 bits [B, H, T, D].
    Returns (codes [B, H, T, D], scale [B, H, D], zero [B, H, D], deq|None)."""
    assert k.dtype == np.uint16 and k.ndim == 4
    B, H, T, D = k.shape
    k1 = np.ascontiguousarray(k)
    codes = np.empty(k.shape, np.uint8)
    sc, zp = np.empty((B, H, D), np.float32), np.empty((B, H, D), np.float32)
    deq = np.empty(k.shape, np.float32) if want_deq else None
    _load().or_kv_k_channel_zp(_ptr(k1), B * H, T, D, _ptr(codes), _ptr(sc), _ptr(zp), _ptr(deq))
    return codes, sc, zp, deq


def quant_int4_g128_zp(w: np.ndarray, want_deq: bool = True):
    """Asymmetric INT4 g128 of a [K, N] weight. Returns (qweight i32 [K/8, N] (codes
    0..15), scale bf16 bits [K/128, N], zero u8 [K/128, N], deq f32 [K, N]|None)."""
    w2, bf = _src(w)
    K, N = w2.shape
    qw = np.empty((K // 8, N), np.int32)
    sc = np.empty((K // 128, N), np.uint16)
    zp = np.empty((K // 128, N), np.uint8)
    deq = np.empty((K, N), np.float32) if want_deq else None
    rc = _load().or_quant_int4_g128_zp(_ptr(w2), bf, K, N, N, _ptr(qw), _ptr(sc), _ptr(zp), _ptr(deq))
    if rc != 0:
        raise ValueError(f"oracle rejects shape {w2.shape} for INT4 g128 with zero points")
    return qw, sc, zp, deq


def gemm_w4a16_zp(A_bf16, qweight, scale_bf16, zero, ii=None, jj=None):
    A = np.ascontiguousarray(A_bf16, dtype=np.uint16)
    qw = np.ascontiguousarray(qweight, dtype=np.int32)
    sc = np.ascontiguousarray(scale_bf16, dtype=np.uint16)
    zp = np.ascontiguousarray(zero, dtype=np.uint8)
    M, K = A.shape
    N = qw.shape[1]
    return _run_gemm(_load().or_gemm_w4a16_zp, (_ptr(A), _ptr(qw), _ptr(sc), _ptr(zp), M, N, K), M, N,
                     ii, jj, ii is None)


def gemm_w4a16_nvfp4(A_bf16, qB, sB, gB, ii=None, jj=None):
    """Weight-only NVFP4: bf16 A [M, K] times B^T [N, K] given as NVFP4 codes and scales."""
    A = np.ascontiguousarray(A_bf16, dtype=np.uint16)
    qB, sB = np.ascontiguousarray(qB, np.uint8), np.ascontiguousarray(sB, np.uint8)
    M, K = A.shape
    N = qB.shape[0]
    return _run_gemm(_load().or_gemm_w4a16_nvfp4, (_ptr(A), _ptr(qB), _ptr(sB), float(gB), M, N, K), M, N,
                     ii, jj, ii is None)


def gemm_w4a16_mxfp4(A_bf16, qB, eB, ii=None, jj=None):
    """Weight-only MXFP4: bf16 A [M, K] times B^T [N, K] given as MXFP4 codes and E8M0 scales."""
    A = np.ascontiguousarray(A_bf16, dtype=np.uint16)
    qB, eB = np.ascontiguousarray(qB, np.uint8), np.ascontiguousarray(eB, np.uint8)
    M, K = A.shape
    N = qB.shape[0]
    return _run_gemm(_load().or_gemm_w4a16_mxfp4, (_ptr(A), _ptr(qB), _ptr(eB), M, N, K), M, N,
                     ii, jj, ii is None)


def col_amax(x: np.ndarray) -> np.ndarray:
    """max |x| over the rows of each column of a 2-D fp32 or bf16-bits array."""
    x2, bf = _src(x)
    rows, cols = x2.shape
    out = np.empty(cols, np.float32)
    _load().or_col_amax(_ptr(x2), bf, rows, cols, _ptr(out))
    return out


def smooth_factors(xmax: np.ndarray, wmax: np.ndarray) -> np.ndarray:
    """SmoothQuant migration factors with alpha = 0.5 from per-channel amaxes."""
    xm = np.ascontiguousarray(xmax, np.float32)
    wm = np.ascontiguousarray(wmax, np.float32)
    assert xm.shape == wm.shape and xm.ndim == 1
    s = np.empty(xm.size, np.float32)
    _load().or_smooth_factors(_ptr(xm), _ptr(wm), xm.size, _ptr(s))
    return s


INT8_PLAIN, INT8_DIVIDE, INT8_MULTIPLY = 0, 1, 2


def quant_int8_rows(x: np.ndarray, factors: np.ndarray | None = None, smooth: int = INT8_PLAIN,
                    want_deq: bool = True):
    """INT8 per row (token or output channel) after an optional per-column smoothing
    factor (INT8_DIVIDE for activations, INT8_MULTIPLY for weights as B^T).
    Returns (codes i8 [R, C], scales f32 [R], deq f32|None)."""
    x2, bf = _src(x)
    rows, cols = x2.shape
    f = None if factors is None else np.ascontiguousarray(factors, np.float32)
    codes = np.empty((rows, cols), np.int8)
    scales = np.empty(rows, np.float32)
    deq = np.empty((rows, cols), np.float32) if want_deq else None
    rc = _load().or_quant_int8_rows(_ptr(x2), bf, rows, cols, _ptr(f), int(smooth), _ptr(codes), _ptr(scales),
                                    _ptr(deq))
    if rc != 0:
        raise ValueError("oracle rejects the INT8 arguments")
    return codes, scales, deq


def gemm_int8(qA, sA, qB, sB, ii=None, jj=None):
    """y, bound of Y = diag(sA) (qA qB^T) diag(sB) with int8 qA [M, K], qB [N, K]."""
    qA, qB = np.ascontiguousarray(qA, np.int8), np.ascontiguousarray(qB, np.int8)
    sA, sB = np.ascontiguousarray(sA, np.float32), np.ascontiguousarray(sB, np.float32)
    M, K = qA.shape
    N = qB.shape[0]
    return _run_gemm(_load().or_gemm_int8, (_ptr(qA), _ptr(sA), _ptr(qB), _ptr(sB), M, N, K), M, N, ii, jj,
                     ii is None)

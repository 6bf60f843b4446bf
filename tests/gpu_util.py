"""Helpers shared by the GPU parity tests: host <-> device transfers of the
seeded inputs and bit-level comparisons. No quantization arithmetic here."""
import numpy as np
import torch


def dev_f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def dev_u8(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.uint8)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> numpy, keeping bit patterns (bf16 -> uint16)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits32(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, np.float32).view(np.uint32)


def assert_same_bytes(gpu: np.ndarray, ref: np.ndarray, what: str):
    gpu, ref = np.asarray(gpu), np.asarray(ref)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if gpu.dtype == np.float32:
        gpu, ref = bits32(gpu), bits32(ref)
    bad = np.argwhere(gpu != ref)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                          f"gpu {gpu[tuple(bad[0])]!r} ref {ref[tuple(bad[0])]!r}"


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def half_ulp_bf16(y_ref: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at the exact value: the error of rounding it to the bf16 output
    (8 significant bits: ulp = 2^(floor(log2|y|) - 7))."""
    y = np.abs(np.asarray(y_ref, np.float64))
    _, e = np.frexp(y)                     # y = m * 2^e, m in [0.5, 1)
    return np.where(y > 0, np.ldexp(1.0, e - 9), 0.0)


def gemm_tolerance(y_ref: np.ndarray, bound: np.ndarray, rel: float = 1e-3) -> np.ndarray:
    """Acceptance bound of a bf16-output GEMM against the exact FP64 reference:
    rel * sum_k |a*b| (the accumulation error allowed) plus half a bf16 ulp of the
    exact result (the rounding of the output to bf16, which alone exceeds the first
    term wherever |y| approaches sum_k |a*b|)."""
    return rel * np.asarray(bound, np.float64) + half_ulp_bf16(y_ref)


# Audit of the half-ulp term: per GEMM check, how many elements pass only because of it
# (|y - y_ref| above rel * sum|ab| but within the full tolerance). Printed in the pytest
# terminal summary, so every GPU run records how much the output-rounding term is used.
HALF_ULP_TALLY = []        # (what, elements checked, elements passing only through the half ulp)


def check_gemm(y_bits: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what: str, rel: float = 1e-3):
    """Assert a bf16 GEMM output against the FP64 reference: every element within
    rel * sum_k |a*b| + half a bf16 ulp of the exact value; tally the elements that
    need the half-ulp term."""
    y = bf16_bits_to_f64(y_bits)
    err = np.abs(y - np.asarray(y_ref, np.float64))
    strict = err <= rel * np.asarray(bound, np.float64)
    ok = err <= gemm_tolerance(y_ref, bound, rel)
    HALF_ULP_TALLY.append((what, int(ok.size), int(np.count_nonzero(ok & ~strict))))
    bad = np.argwhere(~ok)
    assert ok.all(), f"{what}: {len(bad)} outside {rel}*sum|ab| + half a bf16 ulp; first {bad[:3].tolist()}"

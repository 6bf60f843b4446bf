"""GPU parity of the quantizers and the KV write against the CPU oracle.

Codes, scales and dequantized values must match the oracle bit for bit (the
codes are integer decisions taken in fp32 on both sides). Inputs: the seeded
workloads (full size where the oracle finishes in seconds, sampled units of
the full-size tensors otherwise), ragged and tiny shapes, and hand-built edge
values (zeros, signed zeros, exact rounding midpoints, huge outliers)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import assert_same_bytes, dev_bf16, dev_f32, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def to_dev(x):
    return dev_bf16(x) if x.dtype == np.uint16 else dev_f32(x)


GRANS = [oracle.FP8_PER_TENSOR, oracle.FP8_PER_ROW, oracle.FP8_BLOCK_128x128, oracle.FP8_GROUP_1x128]


def check_fp8(qz, x, gran, what):
    c, s, d = qz.qz_quantize_fp8(to_dev(x), gran, dequant=True)
    rc, rs, rd = oracle.quant_fp8(x, gran)
    torch.cuda.synchronize()
    assert_same_bytes(host(c), rc, f"{what} codes")
    assert_same_bytes(host(s).reshape(rs.shape), rs, f"{what} scales")
    assert_same_bytes(host(d), rd, f"{what} dequant")


def edge_tensor(rows, cols, seed=0):
    """N(0,1) data salted with zeros, signed zeros, huge outliers and values that sit
    exactly on E4M3/E2M1 rounding midpoints for unit scales."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    flat = x.ravel()
    n = flat.size
    idx = rng.choice(n, size=min(n, 64), replace=False)
    specials = np.float32([0.0, -0.0, 1e-30, -1e-30, 0.75, -1.75, 3.5, 1.0625, 1e4, -2.5e3, 5.0, 0.25])
    flat[idx] = np.resize(specials, idx.size)
    return x


# ----------------------------------------------------------------- FP8

@pytest.mark.parametrize("gran", GRANS)
def test_fp8_config1_roundtrip(qz, gran):
    """The 1024 x 1024 fp32 weight with 8 outlier columns x50, every granularity, full size."""
    check_fp8(qz, syn.quant_roundtrip_input(seed=0), gran, f"config1 gran{gran}")


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (1, 128), (64, 256), (384, 1024)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fp8_shapes_and_dtypes(qz, gran, shape, dtype):
    x = edge_tensor(*shape, seed=shape[0] * 7 + shape[1])
    if dtype == "bf16":
        x = syn.to_bf16_bits(x)
    check_fp8(qz, x, gran, f"{dtype} {shape} gran{gran}")


@pytest.mark.parametrize("gran", [oracle.FP8_PER_TENSOR, oracle.FP8_PER_ROW])
@pytest.mark.parametrize("shape", [(3, 5), (7, 129), (33, 1000), (1, 1)])
def test_fp8_ragged_scalar_path(qz, gran, shape):
    """Row lengths that are not a multiple of 8 take the scalar path."""
    check_fp8(qz, edge_tensor(*shape, seed=sum(shape)), gran, f"ragged {shape} gran{gran}")


def test_fp8_strided_rows(qz):
    """A leading dimension larger than the row length (a column slice of a wider tensor)."""
    base = edge_tensor(96, 512, seed=3)
    for gran in GRANS:
        xs = to_dev(base)[:, 128:384]
        c, s, d = qz.qz_quantize_fp8(xs, gran, dequant=True)
        rc, rs, rd = oracle.quant_fp8(np.ascontiguousarray(base[:, 128:384]), gran)
        assert_same_bytes(host(c), rc, f"strided codes {gran}")
        assert_same_bytes(host(s).reshape(rs.shape), rs, f"strided scales {gran}")
        assert_same_bytes(host(d), rd, f"strided dequant {gran}")


def test_fp8_all_zero_and_constant(qz):
    check_fp8(qz, np.zeros((16, 256), np.float32), oracle.FP8_PER_TENSOR, "zeros")
    check_fp8(qz, np.zeros((16, 256), np.float32), oracle.FP8_GROUP_1x128, "zeros group")
    check_fp8(qz, np.full((16, 256), -3.0, np.float32), oracle.FP8_BLOCK_128x128, "constant")


def test_fp8_config3_full_size_sampled(qz):
    """Config-3 sizes in the bench's launch configuration: A bf16 2048x4096 -> 1x128,
    B^T bf16 14336x4096 -> 128x128. Sampled rows/blocks are checked one by one."""
    a, bt = syn.fp8_block_gemm_inputs(seed=0)
    ca, sa, _ = qz.qz_quantize_fp8(dev_bf16(a), qz.FP8_GROUP_1x128)
    cb, sb, _ = qz.qz_quantize_fp8(dev_bf16(bt), qz.FP8_BLOCK_128x128)
    ca, sa, cb, sb = host(ca), host(sa), host(cb), host(sb)
    rng = np.random.default_rng(0)
    for r in rng.choice(a.shape[0], 24, replace=False):
        rc, rs, _ = oracle.quant_fp8(a[r:r + 1], oracle.FP8_GROUP_1x128, want_deq=False)
        assert_same_bytes(ca[r:r + 1], rc, f"A row {r} codes")
        assert_same_bytes(sa[r:r + 1], rs, f"A row {r} scales")
    for _ in range(12):
        bi, bj = rng.integers(0, bt.shape[0] // 128), rng.integers(0, bt.shape[1] // 128)
        blk = bt[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
        rc, rs, _ = oracle.quant_fp8(blk, oracle.FP8_BLOCK_128x128, want_deq=False)
        assert_same_bytes(cb[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128], rc, f"B block {bi},{bj}")
        assert_same_bytes(sb[bi:bi + 1, bj:bj + 1], rs, f"B block scale {bi},{bj}")


@pytest.mark.parametrize("shape,dtype", [((2048, 4096), "bf16"), ((1000, 4224), "f32"), ((3001, 1280), "bf16"),
                                         ((8192, 4096), "bf16")])
def test_fp8_group_large_contiguous(qz, shape, dtype):
    """FP8 1x128 on large contiguous tensors: the bench's A (2048 x 4096 bf16), group
    counts that leave a ragged last grid-stride step, fp32 input, and a 67 MB tensor.
    The format is row-local, so rows are compared bit for bit (codes, scales,
    dequant): the first two, the last two and 60 at random."""
    rows, cols = shape
    x = edge_tensor(rows, cols, seed=rows)
    x = syn.to_bf16_bits(x) if dtype == "bf16" else x
    c, s, d = qz.qz_quantize_fp8(to_dev(x), oracle.FP8_GROUP_1x128, dequant=True)
    c, s, d = host(c), host(s), host(d)
    assert qz.qz_device_error() == 0
    pick = {0, 1, rows - 2, rows - 1} | set(np.random.default_rng(rows).choice(rows, 60, replace=False).tolist())
    pick = np.array(sorted(pick))
    rc, rs, rd = oracle.quant_fp8(x[pick], oracle.FP8_GROUP_1x128)
    assert_same_bytes(c[pick], rc, f"large {shape} {dtype} codes")
    assert_same_bytes(s[pick], rs, f"large {shape} {dtype} scales")
    assert_same_bytes(d[pick], rd, f"large {shape} {dtype} dequant")


# ------------------------------------------------------------- MXFP4

def check_mx(qz, x, what):
    c, e, d = qz.qz_quantize_mxfp4(to_dev(x), dequant=True)
    rc, re_, rd = oracle.quant_mxfp4(x)
    assert_same_bytes(host(c), rc, f"{what} codes")
    assert_same_bytes(host(e), re_, f"{what} e8m0")
    assert_same_bytes(host(d), rd, f"{what} dequant")


def check_nv(qz, x, what, amax_in=None):
    amax_dev = None if amax_in is None else torch.tensor([amax_in], dtype=torch.float32, device="cuda")
    c, s, g, d = qz.qz_quantize_nvfp4(to_dev(x), global_amax_in=amax_dev, dequant=True)
    rc, rs, rg, rd = oracle.quant_nvfp4(x, amax_in=amax_in)
    assert_same_bytes(host(g), np.float32([rg]), f"{what} global scale")
    assert_same_bytes(host(s), rs, f"{what} block scales")
    assert_same_bytes(host(c), rc, f"{what} codes")
    assert_same_bytes(host(d), rd, f"{what} dequant")


def test_mxfp4_config1(qz):
    check_mx(qz, syn.quant_roundtrip_input(seed=0), "config1 mxfp4")


def test_nvfp4_config1(qz):
    check_nv(qz, syn.quant_roundtrip_input(seed=0), "config1 nvfp4")


@pytest.mark.parametrize("shape", [(1, 32), (5, 64), (128, 96), (33, 4096)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fp4_shapes(qz, shape, dtype):
    x = edge_tensor(*shape, seed=shape[0] + 3 * shape[1])
    if dtype == "bf16":
        x = syn.to_bf16_bits(x)
    check_mx(qz, x, f"mx {dtype} {shape}")
    check_nv(qz, x, f"nv {dtype} {shape}")


def test_fp4_midpoints_and_zero_signs(qz):
    """Values placed exactly on E2M1 midpoints for the block's scale: ties go down."""
    x = np.zeros((4, 64), np.float32)
    # each 32-block has amax 6 * 2^k so the MX scale is 2^k (exact ratios)
    x[0, :8] = np.float32([6, 0.75, 1.75, 3.5, -0.75, -1.75, -3.5, 5.0])
    x[1, :8] = np.float32([12, 1.5, 3.5, 7.0, 0.5, -0.5, -0.0, -1e-9])
    x[2, :4] = np.float32([-6, 2.5, 1.25, 0.25])
    x[3, :] = -0.0
    check_mx(qz, x, "mx midpoints")
    check_nv(qz, x, "nv midpoints")


def test_fp4_ulp_above_midpoints(qz):
    """Quotients exactly on each E2M1 midpoint and one fp32 ulp above it, with unit scales
    (NVFP4: given tensor amax 2688 -> g = 1, block amax 6 -> block scale 1; MXFP4: block amax
    6 -> scale 2^0), so y = x: ties go down, one ulp above a midpoint goes up."""
    mids = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    above = np.nextafter(mids, np.float32(np.inf), dtype=np.float32)
    below = np.nextafter(mids, np.float32(0), dtype=np.float32)
    vals = np.concatenate([mids, above, below, -mids, -above])          # 35 values
    x = np.zeros((3, 32), np.float32)
    flat = np.concatenate([vals, np.float32([0.0, -0.0, 6.0, -6.0, 3.0, 1e-30, -1e-30])])
    for r in range(3):
        row = flat[r * 14:(r + 1) * 14] if r < 2 else flat[28:]
        x[r, 0] = 6.0                                                   # each 16- and 32-block's max
        x[r, 16] = 6.0
        x[r, 1:1 + min(15, len(row))] = row[:15]
        x[r, 17:17 + max(0, min(15, len(row) - 15))] = row[15:30]
    check_nv(qz, x, "nv ulp above midpoints", amax_in=2688.0)
    check_mx(qz, x, "mx ulp above midpoints")
    check_nv(qz, syn.to_bf16_bits(x), "nv bf16 midpoints", amax_in=2688.0)


def test_fp4_tiny_values_beside_huge_ones(qz):
    """Blocks whose amax is huge hold tiny values (down to bf16 subnormals) of both signs,
    zeros of both signs and values one step either side of midpoints: the quotients of the
    tiny ones underflow to fp32 subnormals or to zero, where the sign of a zero code and
    the step toward zero must still follow the oracle (fp32 and bf16 inputs)."""
    rng = np.random.default_rng(21)
    x = np.zeros((8, 64), np.float32)
    tiny = np.float32([1e-39, -1e-39, 9.2e-41, -9.2e-41, 1e-45, -1e-45, 2.0 ** -133, -(2.0 ** -133),
                       1e-30, -1e-30, 0.0, -0.0, 3e-38, -3e-38])
    for r in range(8):
        big = np.float32(2.0 ** (r * 16 - 20)) * np.float32(1.5 + r / 8)
        for b in range(2):
            row = x[r, b * 32:(b + 1) * 32]
            row[0] = big if (r + b) % 2 == 0 else -big
            row[1:1 + len(tiny)] = tiny
            row[1 + len(tiny):] = rng.standard_normal(31 - len(tiny)).astype(np.float32) * big * np.float32(1e-3)
    check_mx(qz, x, "mx tiny beside huge")
    xb = syn.to_bf16_bits(x)
    check_mx(qz, xb, "mx bf16 tiny beside huge")
    check_nv(qz, x, "nv tiny beside huge")
    check_nv(qz, xb, "nv bf16 tiny beside huge")


def test_nvfp4_given_amax(qz):
    x = edge_tensor(64, 256, seed=8)
    check_nv(qz, x, "nv given amax", amax_in=float(np.abs(x).max()) * 2.0)


def test_nvfp4_block_scale_rounds_to_zero(qz):
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1000.0
    x[0, 16:] = 1e-7
    check_nv(qz, x, "nv zero block scale")


def test_fp4_config4_full_size_sampled(qz):
    """Config-4 sizes: A bf16 8192x4096 and B^T bf16 4096x4096, NVFP4 and MXFP4, in the
    bench's launch configuration; rows sampled, NVFP4 with the oracle's tensor amax."""
    a, bt = syn.fp4_gemm_inputs(seed=0)
    rng = np.random.default_rng(1)
    for name, x in (("A", a), ("Bt", bt)):
        c, s, g, _ = qz.qz_quantize_nvfp4(dev_bf16(x))
        mc, me, _ = qz.qz_quantize_mxfp4(dev_bf16(x))
        c, s, g, mc, me = host(c), host(s), host(g), host(mc), host(me)
        amax = oracle.amax(x)
        rows = rng.choice(x.shape[0], 16, replace=False)
        for r in rows:
            rc, rs, rg, _ = oracle.quant_nvfp4(x[r:r + 1], amax_in=amax, want_deq=False)
            assert_same_bytes(g, np.float32([rg]), f"{name} g")
            assert_same_bytes(c[r:r + 1], rc, f"{name} nv codes row {r}")
            assert_same_bytes(s[r:r + 1], rs, f"{name} nv scales row {r}")
            rc, re_, _ = oracle.quant_mxfp4(x[r:r + 1], want_deq=False)
            assert_same_bytes(mc[r:r + 1], rc, f"{name} mx codes row {r}")
            assert_same_bytes(me[r:r + 1], re_, f"{name} mx scales row {r}")


def check_nv_grouped(qz, xs, what):
    outs = qz.qz_quantize_nvfp4_grouped([to_dev(x) for x in xs])
    torch.cuda.synchronize()
    for i, (x, (c, s, g)) in enumerate(zip(xs, outs)):
        rc, rs, rg, _ = oracle.quant_nvfp4(x, want_deq=False)
        assert_same_bytes(host(g), np.float32([rg]), f"{what} tensor {i} global scale")
        assert_same_bytes(host(s), rs, f"{what} tensor {i} block scales")
        assert_same_bytes(host(c), rc, f"{what} tensor {i} codes")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nvfp4_grouped_mixed_tensors(qz, dtype):
    """Tensors of unrelated sizes in one call (some a single 16-element block, so one warp
    spans several tensors); each must equal its own single-tensor quantization."""
    shapes = [(1, 16), (1, 1024), (3, 4096), (2, 48), (17, 3072), (1, 32), (5, 64), (128, 96), (1, 16)]
    xs = [edge_tensor(r, c, seed=11 * i + r) for i, (r, c) in enumerate(shapes)]
    xs[3] *= np.float32(1e-30)                               # tiny amax: the 1e-12 floors decide
    if dtype == "bf16":
        xs = [syn.to_bf16_bits(x) for x in xs]
    check_nv_grouped(qz, xs, f"grouped {dtype}")


def test_nvfp4_grouped_maximum_count(qz):
    """256 tensors (the most one call takes), all-zero ones among them."""
    rng = np.random.default_rng(5)
    xs = []
    for i in range(256):
        x = (rng.standard_normal((1 + i % 3, 16 * (1 + i % 7))) * (1 + i)).astype(np.float32)
        if i % 50 == 0:
            x[:] = 0.0
        xs.append(syn.to_bf16_bits(x))
    check_nv_grouped(qz, xs, "grouped 256")


def test_nvfp4_grouped_decode_activations(qz):
    """The activations of one Qwen3-0.6B decode layer at 16 tokens (q/k/v/o, gate/up, down
    inputs), matching per-tensor qz_quantize_nvfp4 calls in the same launch configuration."""
    rng = np.random.default_rng(9)
    shapes = [(16, 1024)] * 3 + [(16, 2048)] + [(16, 1024)] * 2 + [(16, 3072)]
    xs = [syn.to_bf16_bits(rng.standard_normal(s).astype(np.float32) * 3) for s in shapes]
    outs = qz.qz_quantize_nvfp4_grouped([dev_bf16(x) for x in xs])
    for x, (c, s, g) in zip(xs, outs):
        c1, s1, g1, _ = qz.qz_quantize_nvfp4(dev_bf16(x))
        torch.cuda.synchronize()
        assert_same_bytes(host(c), host(c1), "codes vs single call")
        assert_same_bytes(host(s), host(s1), "scales vs single call")
        assert_same_bytes(host(g), host(g1), "global scale vs single call")
    check_nv_grouped(qz, xs[:2], "decode layer sample")


# -------------------------------------------------------------- INT4 g128

@pytest.mark.parametrize("shape", [(128, 64), (384, 192), (1024, 1024)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_int4_g128_shapes(qz, shape, dtype):
    rng = np.random.default_rng(shape[0] + shape[1])
    w = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    w.ravel()[rng.choice(w.size, 16, replace=False)] = np.float32([0.0, -0.0, 0.5, -0.7] * 4)
    if dtype == "bf16":
        w = syn.to_bf16_bits(w)
    qw, sc, d = qz.qz_quantize_int4_g128(to_dev(w), dequant=True)
    rq, rs, rd = oracle.quant_int4_g128(w)
    assert_same_bytes(host(qw), rq, "qweight")
    assert_same_bytes(host(sc), rs, "scales")
    assert_same_bytes(host(d), rd, "dequant")


def test_int4_config2_weight_sampled(qz):
    """The config-2 weight 4096 x 14336 fp32, column slices checked one by one."""
    _, w = syn.w4a16_decode_inputs(M=1, seed=0)
    qw, sc, _ = qz.qz_quantize_int4_g128(dev_f32(w))
    qw, sc = host(qw), host(sc)
    rng = np.random.default_rng(2)
    for j in rng.choice(w.shape[1] // 64, 6, replace=False):
        sl = slice(j * 64, j * 64 + 64)
        rq, rs, _ = oracle.quant_int4_g128(np.ascontiguousarray(w[:, sl]), want_deq=False)
        assert_same_bytes(qw[:, sl], rq, f"qweight cols {j * 64}")
        assert_same_bytes(sc[:, sl], rs, f"scales cols {j * 64}")


# ------------------------------------------------------------ KV write

def test_kv_write_config5_full(qz):
    """FP8 per-tensor KV write of K (N(0,1) + per-channel bias N(0,4)) and V, bf16
    [1, 8, 4096, 128], full size."""
    k, v = syn.kv_cache_inputs(seed=0)
    kc, vc, ks, vs = qz.qz_kv_write_fp8(dev_bf16(k), dev_bf16(v))
    rkc, rvc, rks, rvs, _, _ = oracle.kv_write_fp8(k, v)
    assert_same_bytes(host(ks), np.float32([rks]), "k scale")
    assert_same_bytes(host(vs), np.float32([rvs]), "v scale")
    assert_same_bytes(host(kc), rkc, "k codes")
    assert_same_bytes(host(vc), rvc, "v codes")


@pytest.mark.parametrize("shape", [(1, 1, 1, 8), (1, 3, 100, 8), (2, 8, 1000, 64), (1, 8, 8192, 128)])
def test_kv_write_shapes(qz, shape):
    """Slices that leave some CTAs empty, a single 16-byte word, and a size past the
    one-launch limit (the two-launch path)."""
    B, H, T, D = shape
    rng = np.random.default_rng(T + D)
    k = syn.to_bf16_bits((rng.standard_normal(shape) * 3).astype(np.float32))
    v = syn.to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    kc, vc, ks, vs = qz.qz_kv_write_fp8(dev_bf16(k), dev_bf16(v))
    rkc, rvc, rks, rvs, _, _ = oracle.kv_write_fp8(k, v)
    assert_same_bytes(host(ks), np.float32([rks]), "k scale")
    assert_same_bytes(host(vs), np.float32([rvs]), "v scale")
    assert_same_bytes(host(kc).ravel(), rkc.ravel(), "k codes")
    assert_same_bytes(host(vc).ravel(), rvc.ravel(), "v codes")


def test_kv_write_workspace_reuse_and_graph_replay(qz):
    """One workspace across calls with different data, then a captured call replayed
    on new data: each result must be that data's own (no stale meeting records)."""
    shape = (1, 8, 512, 128)
    ws = qz.Workspace()
    kd = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    vd = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    kc = torch.empty(shape, dtype=torch.uint8, device="cuda")
    vc = torch.empty(shape, dtype=torch.uint8, device="cuda")
    ks = torch.empty(1, dtype=torch.float32, device="cuda")
    vs = torch.empty(1, dtype=torch.float32, device="cuda")

    def data(seed):
        rng = np.random.default_rng(seed)
        scale = 1.0 + seed
        return (syn.to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32)),
                syn.to_bf16_bits((rng.standard_normal(shape) * 0.5 * scale).astype(np.float32)))

    def check(k, v, what):
        torch.cuda.synchronize()
        rkc, rvc, rks, rvs, _, _ = oracle.kv_write_fp8(k, v)
        assert_same_bytes(host(ks), np.float32([rks]), f"{what} k scale")
        assert_same_bytes(host(vs), np.float32([rvs]), f"{what} v scale")
        assert_same_bytes(host(kc).ravel(), rkc.ravel(), f"{what} k codes")
        assert_same_bytes(host(vc).ravel(), rvc.ravel(), f"{what} v codes")

    def load(k, v):
        kd.copy_(dev_bf16(k))
        vd.copy_(dev_bf16(v))

    for seed in range(3):
        k, v = data(seed)
        load(k, v)
        qz.qz_kv_write_fp8(kd, vd, k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs, ws=ws)
        check(k, v, f"call {seed}")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qz.qz_kv_write_fp8(kd, vd, k_codes=kc, v_codes=vc, k_scale=ks, v_scale=vs, ws=ws, stream=s)
    for seed in range(3, 6):
        k, v = data(seed)
        load(k, v)
        torch.cuda.synchronize()
        g.replay()
        check(k, v, f"replay {seed}")
    assert qz.qz_device_error() == 0


def test_kv_write_given_scale(qz):
    k, v = syn.kv_cache_inputs(seed=1, T=64)
    ks = torch.tensor([0.05], dtype=torch.float32, device="cuda")
    vs = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    kc, vc, _, _ = qz.qz_kv_write_fp8(dev_bf16(k), dev_bf16(v), k_scale=ks, v_scale=vs, mode=qz.SCALE_GIVEN)
    rk, _ = oracle.quant_fp8_given(k, 0.05, want_deq=False)
    rv, _ = oracle.quant_fp8_given(v, 0.01, want_deq=False)
    assert_same_bytes(host(kc), rk, "k codes given")
    assert_same_bytes(host(vc), rv, "v codes given")
    assert host(ks)[0] == np.float32(0.05) and host(vs)[0] == np.float32(0.01)


def test_repeated_calls_share_workspace(qz):
    """Per-tensor partial maxima live in the caller's workspace; back-to-back calls on
    different tensors with one workspace stay independent."""
    ws = qz.Workspace()
    x1 = edge_tensor(64, 256, seed=10)
    x2 = edge_tensor(64, 256, seed=11) * np.float32(1e-3)
    o1 = qz.qz_quantize_fp8(dev_f32(x1), qz.FP8_PER_TENSOR, ws=ws)
    o2 = qz.qz_quantize_fp8(dev_f32(x2), qz.FP8_PER_TENSOR, ws=ws)
    for (c, s, _), x in ((o1, x1), (o2, x2)):
        rc, rs, _ = oracle.quant_fp8(x, oracle.FP8_PER_TENSOR, want_deq=False)
        assert_same_bytes(host(c), rc, "codes")
        assert_same_bytes(host(s), rs, "scale")

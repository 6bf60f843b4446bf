"""GPU parity of the quantizers on a tensor of more than 2^31 elements.

One bf16 [524544, 4096] tensor (2,148,532,224 elements; 4.3 GB), built on the
device from a seeded 256-row block: tile t (rows 256 t .. 256 t + 255) is the
block times 2^((t mod 7) - 3), except the last tile, which starts exactly at
element 2^31 and is the block times 2^4, so the tensor's amax lies past the
32-bit boundary. Outputs are pre-filled with a sentinel. Checked against the
oracle, bit for bit, on rows on both sides of the boundary: the row-local
formats on those rows, the 128 x 128 blocks and INT4 groups that hold them, and
the per-tensor formats (FP8 per tensor, NVFP4, the KV write) on a subset that
includes the row holding the tensor's maximum, which fixes the same per-tensor
scale. The block-scaled GEMMs (FP8, NVFP4, MXFP4, INT8) run at M x N = 65664 x
32768 (2,151,677,952 outputs), sampled on rows on both sides of output 2^31."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import assert_same_bytes, check_gemm, host

pytestmark = pytest.mark.gpu

P, COLS = 256, 4096
TILES = 2049
ROWS = P * TILES                                   # 524544 rows
BOUNDARY_ROW = (1 << 31) // COLS                    # 524288: first row past element 2^31
assert ROWS * COLS > (1 << 31) and BOUNDARY_ROW == P * (TILES - 1)


def tile_exp(t):
    return 4 if t == TILES - 1 else (t % 7) - 3


def base_block():
    rng = np.random.default_rng(2024)
    return syn.to_bf16_bits(rng.standard_normal((P, COLS)).astype(np.float32))


def host_rows(base_f32, rows):
    """The tensor's rows, built on the host from the block (exact: power-of-two factors)."""
    rows = np.asarray(rows)
    f = np.array([np.ldexp(np.float32(1), tile_exp(int(r) // P)) for r in rows], np.float32)
    return base_f32[rows % P] * f[:, None]


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


@pytest.fixture(scope="module")
def big():
    bits = base_block()
    base_f32 = (bits.astype(np.uint32) << 16).view(np.float32)
    x = torch.empty((ROWS, COLS), dtype=torch.bfloat16, device="cuda")
    tiles = x.view(TILES, P, COLS)
    tiles.copy_(torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16).expand(TILES, P, COLS))
    f = torch.tensor([2.0 ** tile_exp(t) for t in range(TILES)], dtype=torch.float32, device="cuda")
    tiles.mul_(f.view(TILES, 1, 1).to(torch.bfloat16))
    torch.cuda.synchronize()
    yield x, base_f32
    del x, tiles
    torch.cuda.empty_cache()


# rows on both sides of element 2^31, and the row holding the tensor's maximum
SAMPLE = [0, 1, 77_777, BOUNDARY_ROW - 1, BOUNDARY_ROW, BOUNDARY_ROW + 129, ROWS - 1]


def max_row(base_f32):
    return BOUNDARY_ROW + int(np.argmax(np.abs(base_f32).max(axis=1)))


def sentinel(shape, dtype=torch.uint8):
    return torch.full(shape, -91 if dtype == torch.int8 else 0xA5, dtype=dtype, device="cuda")   # byte 0xA5


@pytest.mark.parametrize("gran", [oracle.FP8_PER_ROW, oracle.FP8_GROUP_1x128])
def test_fp8_row_local_past_2_31(qz, big, gran):
    x, base = big
    ns = COLS // 128 if gran == oracle.FP8_GROUP_1x128 else 1
    codes, scales, _ = qz.qz_quantize_fp8(x, gran, codes=sentinel((ROWS, COLS)),
                                         scales=torch.full((ROWS, ns) if ns > 1 else (ROWS,), -1.0,
                                                           device="cuda"))
    torch.cuda.synchronize()
    rows = np.array(SAMPLE)
    rc, rs, _ = oracle.quant_fp8(host_rows(base, rows), gran, want_deq=False)
    idx = torch.from_numpy(rows).cuda()
    assert_same_bytes(host(codes[idx]), rc, f"fp8 gran {gran} codes")
    assert_same_bytes(host(scales[idx]).reshape(rs.shape), rs, f"fp8 gran {gran} scales")


def test_fp8_block_past_2_31(qz, big):
    x, base = big
    codes, scales, _ = qz.qz_quantize_fp8(x, oracle.FP8_BLOCK_128x128, codes=sentinel((ROWS, COLS)))
    torch.cuda.synchronize()
    for rb in sorted({r // 128 for r in SAMPLE}):
        rows = np.arange(rb * 128, rb * 128 + 128)
        rc, rs, _ = oracle.quant_fp8(host_rows(base, rows), oracle.FP8_BLOCK_128x128, want_deq=False)
        assert_same_bytes(host(codes[rb * 128:rb * 128 + 128]), rc, f"fp8 128x128 codes, row block {rb}")
        assert_same_bytes(host(scales.view(ROWS // 128, COLS // 128)[rb:rb + 1]), rs,
                          f"fp8 128x128 scales, row block {rb}")


def test_fp8_per_tensor_past_2_31(qz, big):
    x, base = big
    codes, scale, _ = qz.qz_quantize_fp8(x, oracle.FP8_PER_TENSOR, codes=sentinel((ROWS, COLS)))
    torch.cuda.synchronize()
    rows = np.array(SAMPLE + [max_row(base)])
    rc, rs, _ = oracle.quant_fp8(host_rows(base, rows), oracle.FP8_PER_TENSOR, want_deq=False)
    assert_same_bytes(host(scale), rs, "fp8 per-tensor scale (amax past 2^31)")
    assert_same_bytes(host(codes[torch.from_numpy(rows).cuda()]), rc, "fp8 per-tensor codes")


def test_mxfp4_past_2_31(qz, big):
    x, base = big
    codes, e8, _ = qz.qz_quantize_mxfp4(x, codes=sentinel((ROWS, COLS // 2)),
                                        scale_e8m0=sentinel((ROWS, COLS // 32)))
    torch.cuda.synchronize()
    rows = np.array(SAMPLE)
    rc, re8, _ = oracle.quant_mxfp4(host_rows(base, rows), want_deq=False)
    idx = torch.from_numpy(rows).cuda()
    assert_same_bytes(host(codes[idx]), rc, "mxfp4 codes")
    assert_same_bytes(host(e8[idx]), re8, "mxfp4 scales")


def test_nvfp4_past_2_31(qz, big):
    x, base = big
    codes, sb, g, _ = qz.qz_quantize_nvfp4(x, codes=sentinel((ROWS, COLS // 2)),
                                           scale_e4m3=sentinel((ROWS, COLS // 16)))
    torch.cuda.synchronize()
    rows = np.array(SAMPLE + [max_row(base)])
    rc, rsb, rg, _ = oracle.quant_nvfp4(host_rows(base, rows), want_deq=False)
    idx = torch.from_numpy(rows).cuda()
    assert_same_bytes(host(g).reshape(np.shape(rg)), np.asarray(rg, np.float32), "nvfp4 global scale")
    assert_same_bytes(host(codes[idx]), rc, "nvfp4 codes")
    assert_same_bytes(host(sb[idx]), rsb, "nvfp4 block scales")


def test_int4_g128_past_2_31(qz, big):
    """The tensor as an INT4 weight [K = 524544, N = 4096]: groups of 128 along K."""
    x, base = big
    qw, sc, _ = qz.qz_quantize_int4_g128(x, qweight=sentinel((ROWS // 8, COLS), torch.int32),
                                         scale_bf16=sentinel((ROWS // 128, COLS), torch.int16).view(torch.bfloat16))
    torch.cuda.synchronize()
    for g in sorted({r // 128 for r in SAMPLE}):
        rows = np.arange(g * 128, g * 128 + 128)
        rq, rs, _ = oracle.quant_int4_g128(host_rows(base, rows), want_deq=False)
        assert_same_bytes(host(qw[g * 16:g * 16 + 16]), rq, f"int4 codes, group {g}")
        assert_same_bytes(host(sc[g:g + 1]).view(np.uint16), rs, f"int4 scales, group {g}")


def test_int8_rows_past_2_31(qz, big):
    x, base = big
    q, s, _ = qz.qz_quantize_int8_rows(x, codes=sentinel((ROWS, COLS), torch.int8),
                                       scales=torch.full((ROWS,), -1.0, device="cuda"))
    torch.cuda.synchronize()
    rows = np.array(SAMPLE)
    rq, rs, _ = oracle.quant_int8_rows(host_rows(base, rows), want_deq=False)
    idx = torch.from_numpy(rows).cuda()
    assert_same_bytes(host(q[idx]).view(np.uint8), rq.view(np.uint8), "int8 codes")
    assert_same_bytes(host(s[idx]), rs, "int8 scales")


def test_kv_write_past_2_31(qz, big):
    """K and V both the whole tensor as [1, 1, 524544, 4096]: each is one per-tensor FP8
    quantization of 2,148,532,224 elements."""
    x, base = big
    kv = x.view(1, 1, ROWS, COLS)
    kc, vc, ks, vs = qz.qz_kv_write_fp8(kv, kv, k_codes=sentinel(kv.shape), v_codes=sentinel(kv.shape))
    torch.cuda.synchronize()
    rows = np.array(SAMPLE + [max_row(base)])
    sub = syn.to_bf16_bits(host_rows(base, rows))                 # exact: the values are bf16
    rkc, rvc, rks, rvs, _, _ = oracle.kv_write_fp8(sub, sub)
    idx = torch.from_numpy(rows).cuda()
    assert_same_bytes(host(ks), np.float32([rks]), "k scale (amax past 2^31)")
    assert_same_bytes(host(vs), np.float32([rvs]), "v scale")
    assert_same_bytes(host(kc[0, 0][idx]), rkc, "k codes")
    assert_same_bytes(host(vc[0, 0][idx]), rvc, "v codes")


# ---------------------------------------------------- GEMM outputs past 2^31

GM, GN = 65664, 32768                              # M x N = 2,151,677,952 outputs
GROWS = [0, 1, 65535, 65536, GM - 1]               # row 65536 starts at output 2^31
GCOLS = [0, 255, 256, 16384, GN - 1]


def gemm_samples(seed):
    rng = np.random.default_rng(seed)
    ii, jj = np.meshgrid(GROWS, GCOLS, indexing="ij")
    ii = np.concatenate([ii.ravel(), rng.integers(0, GM, 1000), rng.integers(65536, GM, 500)])
    jj = np.concatenate([jj.ravel(), rng.integers(0, GN, 1500)])
    return ii, jj


def gemm_operands(K, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((GM, K)).astype(np.float32)
    a[:, rng.choice(K, 2, replace=False)] *= np.float32(20)
    bt = (rng.standard_normal((GN, K)) * 0.02).astype(np.float32)
    return syn.to_bf16_bits(a), syn.to_bf16_bits(bt)


def gather(Y, ii, jj):
    return host(Y[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()])


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_fp8_block_gemm_output_past_2_31(qz):
    a, bt = gemm_operands(128, seed=1)
    qa, sa, _ = oracle.quant_fp8(a, oracle.FP8_GROUP_1x128, want_deq=False)
    qb, sb, _ = oracle.quant_fp8(bt, oracle.FP8_BLOCK_128x128, want_deq=False)
    Y = qz.qz_gemm_fp8_block(dev(qa), dev(sa), dev(qb), dev(sb))
    torch.cuda.synchronize()
    ii, jj = gemm_samples(1)
    y_ref, bound = oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)
    check_gemm(gather(Y, ii, jj), y_ref, bound, "fp8 block GEMM, outputs past 2^31", 1e-3)


@pytest.mark.parametrize("fmt", ["nv", "mx"])
def test_fp4_gemm_output_past_2_31(qz, fmt):
    a, bt = gemm_operands(256, seed=2)
    if fmt == "nv":
        ca, sa, ga, _ = oracle.quant_nvfp4(a, want_deq=False)
        cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
        ops = (ca, sa, ga, cb, sb, gb)
        Y = qz.qz_gemm_nvfp4(dev(ca), dev(sa), dev(np.float32([ga])), dev(cb), dev(sb), dev(np.float32([gb])))
        ref = oracle.gemm_nvfp4
    else:
        ca, ea, _ = oracle.quant_mxfp4(a, want_deq=False)
        cb, eb, _ = oracle.quant_mxfp4(bt, want_deq=False)
        ops = (ca, ea, cb, eb)
        Y = qz.qz_gemm_mxfp4(dev(ca), dev(ea), dev(cb), dev(eb))
        ref = oracle.gemm_mxfp4
    torch.cuda.synchronize()
    ii, jj = gemm_samples(2)
    y_ref, bound = ref(*ops, ii, jj)
    check_gemm(gather(Y, ii, jj), y_ref, bound, f"{fmt}fp4 GEMM, outputs past 2^31", 1e-3)


def test_int8_gemm_output_past_2_31(qz):
    a, bt = gemm_operands(64, seed=3)
    qa, sa, _ = oracle.quant_int8_rows(a, want_deq=False)
    qb, sb, _ = oracle.quant_int8_rows(bt, want_deq=False)
    Y = qz.qz_gemm_int8(dev(qa), dev(sa), dev(qb), dev(sb))
    torch.cuda.synchronize()
    ii, jj = gemm_samples(3)
    y_ref, bound = oracle.gemm_int8(qa, sa, qb, sb, ii, jj)
    check_gemm(gather(Y, ii, jj), y_ref, bound, "int8 GEMM, outputs past 2^31", 1e-3)

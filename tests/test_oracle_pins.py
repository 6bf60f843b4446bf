"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself:
values the pages print (tests/golden/), library routines (torch's fp32 ->
float8_e4m3fn and fp32 -> bfloat16 casts, numpy matmul), closed forms,
invariants and brute force on tiny inputs. A plausible mistake in the oracle
(a wrong grid value, tie direction, scale formula, index or transposed
operand) fails at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f32(v):
    return np.float32(v)


def f32_neighbours(values, n_ulp):
    """Every fp32 within n_ulp ulps of each value (positive finite inputs)."""
    bits = np.asarray(values, np.float32).view(np.int32).astype(np.int64)
    offs = np.arange(-n_ulp, n_ulp + 1, dtype=np.int64)
    allb = (bits[:, None] + offs[None, :]).ravel()
    allb = allb[(allb > 0) & (allb < 0x7F800000)]
    return np.unique(allb.astype(np.int32)).view(np.float32)


# ------------------------------------------------------------------- E4M3

def test_e4m3_format_facts():
    g = {r[0]: r[1:] for r in read_golden("format_grids.txt")}
    vals = [oracle.e4m3_decode(c) for c in range(256)]
    finite = [v for v in vals if not np.isnan(v)]
    assert len(vals) == int(g["e4m3_patterns"][0])
    assert max(finite) == float(g["e4m3_max"][0]) == oracle.e4m3_decode(0x7E)
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))
    assert sum(np.isnan(v) for v in vals) == 2          # one NaN pattern per sign, no inf
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6         # smallest normal
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9         # smallest subnormal
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0xFE) == -448.0


def test_e4m3_decode_encode_identity_all_codes():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if np.isnan(v):
            continue
        assert oracle.e4m3_encode(f32(v)) == c, hex(c)


def _e4m3_sweep_values():
    pos = np.array([oracle.e4m3_decode(c) for c in range(0x7F)], np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    pts = np.concatenate([pos[1:], mids, [2.0 ** -10, 3 * 2.0 ** -11]])
    near = f32_neighbours(pts.astype(np.float32), 40)
    rng = np.random.default_rng(1234)
    rnd = np.exp(rng.uniform(np.log(1e-6), np.log(448.0), 400_000)).astype(np.float32)
    v = np.concatenate([near, rnd, np.float32([0.0, 448.0, 2.0 ** -20])])
    v = v[v <= 448.0]
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_cast():
    """Library pin: torch's fp32 -> float8_e4m3fn cast (round to nearest even) on a
    sweep of every fp32 within 40 ulps of each E4M3 value and rounding midpoint, plus
    random magnitudes, both signs, all within the +-448 range."""
    y = _e4m3_sweep_values()
    ours = oracle.e4m3_encode_array(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(y[i]), hex(ours[i]), hex(ref[i])) for i in bad[:8]]


def test_e4m3_saturates_like_clamp():
    # Beyond 448 the oracle saturates (the pages clamp to +-448 before the cast).
    assert oracle.e4m3_encode(f32(460.0)) == 0x7E
    assert oracle.e4m3_encode(f32(-1000.0)) == 0xFE
    assert oracle.e4m3_encode(f32(-0.0)) == 0x80
    assert oracle.e4m3_encode(f32(-1e-6)) == 0x80


# ------------------------------------------------------------------- E2M1

def test_e2m1_format_facts():
    g = {r[0]: r[1:] for r in read_golden("format_grids.txt")}
    grid = [float(v) for v in g["e2m1_values"]]
    assert [oracle.e2m1_decode(c) for c in range(8)] == grid
    assert [oracle.e2m1_decode(c | 8) for c in range(8)] == [-v for v in grid]
    assert len({(c, oracle.e2m1_decode(c)) for c in range(16)}) == int(g["e2m1_patterns"][0])
    for i, v in enumerate(grid):
        assert oracle.e2m1_encode(f32(v)) == i
        if v > 0:
            assert oracle.e2m1_encode(f32(-v)) == i | 8


def test_e2m1_ties_go_to_smaller_magnitude():
    # Midpoints between grid neighbours: the argmin's first index is the lower one.
    for lo in range(7):
        mid = (E2M1_GRID[lo] + E2M1_GRID[lo + 1]) / 2
        assert oracle.e2m1_encode(f32(mid)) == lo, mid
        assert oracle.e2m1_encode(np.nextafter(f32(mid), f32(np.inf))) == lo + 1, mid
        assert oracle.e2m1_encode(np.nextafter(f32(mid), f32(0))) == lo, mid
        assert oracle.e2m1_encode(f32(-mid)) == (lo | 8), mid


def test_e2m1_matches_torch_argmin_pipeline():
    """Library pin: torch.argmin over fp32 distances to the grid (first index on ties),
    on every fp32 within 64 ulps of each grid point and midpoint, plus a uniform
    sweep of [-6, 6]."""
    pts = np.concatenate([E2M1_GRID[1:], (E2M1_GRID[:-1] + E2M1_GRID[1:]) / 2])
    near = f32_neighbours(pts.astype(np.float32), 64)
    y = np.concatenate([near, np.linspace(0, 6, 200_001, dtype=np.float32)])
    y = np.concatenate([y, -y[y > 0]])
    t = torch.from_numpy(y)
    idx = (t.abs().unsqueeze(-1) - torch.tensor(E2M1_GRID, dtype=torch.float32)).abs().argmin(-1)
    ref = idx.numpy().astype(np.uint8) | np.where(y < 0, 8, 0).astype(np.uint8)
    ours = np.array([oracle.e2m1_encode(v) for v in y], np.uint8)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(y[i]), ours[i], ref[i]) for i in bad[:8]]


def test_e2m1_sign_of_zero():
    assert oracle.e2m1_encode(f32(-0.0)) == 0          # sign(-0.0) == 0
    assert oracle.e2m1_encode(f32(-1e-3)) == 8         # negative, rounds to magnitude 0
    assert np.signbit(oracle.e2m1_decode(8))


# ------------------------------------------------------------------- bf16

def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * np.float32(100.0),
        # exact ties: low 16 bits == 0x8000
        ((rng.integers(0x3F000000, 0x43000000, 2000, dtype=np.int64) & ~0xFFFF) | 0x8000)
        .astype(np.int32).view(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.f32_to_bf16(v) for v in x], np.uint16)
    assert np.array_equal(ours, ref)
    assert all(oracle.bf16_to_f32(b) == np.float32(v) for b, v in [(0x3F80, 1.0), (0xC000, -2.0)])


# ------------------------------------------------------- worked example

def test_int_quant_worked_example():
    for x, s, q, xh in read_golden("worked_example_int.txt"):
        got_q, got_xh = oracle.int_quant_one(f32(float(x)), f32(float(s)), -8, 7)
        assert got_q == int(q)
        assert abs(got_xh - float(xh)) < 1e-6
        assert abs(abs(float(x) - got_xh) - 0.04) < 1e-6


def test_int_quant_round_half_even_and_clip():
    assert oracle.int_quant_one(f32(2.5), f32(1.0), -8, 7)[0] == 2
    assert oracle.int_quant_one(f32(3.5), f32(1.0), -8, 7)[0] == 4
    assert oracle.int_quant_one(f32(-2.5), f32(1.0), -8, 7)[0] == -2
    assert oracle.int_quant_one(f32(9.0), f32(1.0), -8, 7)[0] == 7
    assert oracle.int_quant_one(f32(-9.0), f32(1.0), -8, 7)[0] == -8


# ------------------------------------------------------------ storage

def test_storage_costs():
    g = {r[0]: float(r[2]) for r in read_golden("storage_costs.txt")}
    rng = np.random.default_rng(3)
    w = rng.standard_normal((256, 64)).astype(np.float32)
    qw, sc, _ = oracle.quant_int4_g128(w, want_deq=False)
    per_weight = (qw.nbytes + sc.nbytes) / w.size
    assert per_weight == 0.5 + 2 / 128
    assert round(per_weight, 3) == g["int4_g128"]
    x = rng.standard_normal((8, 256)).astype(np.float32)
    c, e, _ = oracle.quant_mxfp4(x, want_deq=False)
    assert 8 * (c.nbytes + e.nbytes) / x.size == g["mxfp4"]
    c, s, gg, _ = oracle.quant_nvfp4(x, want_deq=False)
    assert 8 * (c.nbytes + s.nbytes) / x.size == g["nvfp4"]
    assert np.float32(gg).nbytes * 8 == 32     # one FP32 scale per tensor


# ------------------------------------------------------- quantizer invariants

def _outlier_tensor(rows=256, cols=512, seed=11):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(0.02)
    x[:, rng.choice(cols, 4, replace=False)] *= np.float32(50)
    return x


def _fp4_codes_mod_zero_sign(packed):
    lo, hi = packed & 0xF, packed >> 4
    lo = np.where((lo & 7) == 0, 0, lo)
    hi = np.where((hi & 7) == 0, 0, hi)
    return lo | (hi << 4)


def _grid_half_gap(grid_pos, a):
    """Half the gap of the grid interval holding |y| = a (a within the grid)."""
    i = np.clip(np.searchsorted(grid_pos, a, side="right") - 1, 0, len(grid_pos) - 2)
    return (grid_pos[i + 1] - grid_pos[i]) / 2


E4M3_POS = np.array([oracle.e4m3_decode(c) for c in range(0x7F)], np.float64)


@pytest.mark.parametrize("gran", [0, 1, 2, 3])
def test_fp8_invariants(gran):
    x = _outlier_tensor()
    codes, scales, deq = oracle.quant_fp8(x, gran)
    # error bound: half a grid step of y, times the scale (+ the fp32 roundings)
    expand = {0: lambda s: np.full(x.shape, s[0]),
              1: lambda s: np.repeat(s[:, None], x.shape[1], 1),
              2: lambda s: np.kron(s, np.ones((128, 128), np.float32)),
              3: lambda s: np.repeat(s, 128, 1)}[gran]
    s_full = expand(scales).astype(np.float64)
    y = np.abs(x.astype(np.float64) / s_full)
    hg = _grid_half_gap(E4M3_POS, np.minimum(y, 448.0))
    err = np.abs(x.astype(np.float64) - deq.astype(np.float64))
    assert np.all(err <= hg * s_full * (1 + 2.0 ** -20) + 2.0 ** -24 * np.abs(x))
    # each unit's amax element maps to +-448
    if gran == 0:
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert codes[i] & 0x7F == 0x7E
        assert scales[0] == np.float32(np.abs(x).max() / np.float32(448))
    # idempotence: quantizing the dequantized tensor gives the same codes and scales
    c2, s2, d2 = oracle.quant_fp8(deq, gran)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales) and np.array_equal(d2, deq)


def test_fp8_block_over_one_row_equals_group():
    x = _outlier_tensor(rows=1, cols=1024)
    a = oracle.quant_fp8(x, oracle.FP8_BLOCK_128x128)
    b = oracle.quant_fp8(x, oracle.FP8_GROUP_1x128)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))


def test_fp8_block_extent_is_min_128_rows():
    x = _outlier_tensor(rows=64, cols=256)
    codes, scales, _ = oracle.quant_fp8(x, oracle.FP8_BLOCK_128x128)
    assert scales.shape == (1, 2)
    assert scales[0, 1] == np.float32(np.abs(x[:, 128:]).max() / np.float32(448))
    with pytest.raises(ValueError):
        oracle.quant_fp8(_outlier_tensor(rows=200, cols=256), oracle.FP8_BLOCK_128x128)


def test_fp8_unit_scale_reduces_to_plain_cast():
    """With amax = 448 the per-tensor scale is 1 and FP8 is a plain E4M3 cast (torch)."""
    rng = np.random.default_rng(5)
    x = rng.uniform(-448, 448, (64, 64)).astype(np.float32)
    x[3, 7] = 448.0
    codes, scales, deq = oracle.quant_fp8(x, oracle.FP8_PER_TENSOR)
    assert scales[0] == 1.0
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn)
    assert np.array_equal(codes, ref.view(torch.uint8).numpy())
    assert np.array_equal(deq, ref.float().numpy())


def test_fp8_all_zero_tensor_uses_clamp_floor():
    x = np.zeros((4, 128), np.float32)
    codes, scales, deq = oracle.quant_fp8(x, oracle.FP8_PER_TENSOR)
    assert scales[0] == np.float32(np.float32(1e-12) / np.float32(448))
    assert not codes.any() and not deq.any()


def test_fp4_all_zero_blocks_use_clamp_floor():
    # The page clamps every amax to at least 1e-12 before taking a scale. MXFP4: an all-zero
    # block gets E = floor(log2(fp32(1e-12))) - 2 = -42, E8M0 code 85. NVFP4: an all-zero
    # tensor gets g = fp32(1e-12) / 2688 and block scale E4M3(0) = 0.
    x = np.zeros((2, 64), np.float32)
    x[1, 32:] = 1.0                                                   # one non-zero block
    codes, e8, deq = oracle.quant_mxfp4(x)
    e_floor = int(np.floor(np.log2(np.float64(np.float32(1e-12))))) - 2
    assert e_floor == -42
    assert e8[0, 0] == e8[0, 1] == e8[1, 0] == e_floor + 127 and e8[1, 1] == 0 - 2 + 127
    assert not codes[0].any() and not deq[0].any()
    z = np.zeros((1, 32), np.float32)
    c, sb, g, d = oracle.quant_nvfp4(z)
    assert g == np.float32(np.float32(1e-12) / np.float32(2688.0))
    assert not sb.any() and not c.any() and not d.any()


def test_mxfp4_invariants():
    x = _outlier_tensor()
    codes, e8, deq = oracle.quant_mxfp4(x)
    s = np.ldexp(1.0, e8.astype(np.int64) - 127)                     # [R, C/32]
    amax = np.abs(x.reshape(x.shape[0], -1, 32)).max(-1).astype(np.float64)
    r = amax / s
    assert np.all((r >= 4) & (r < 8))                                  # block max lands in [4, 8)
    # error: half a grid step for unclipped, |x| - 6s for clipped elements
    sf = np.repeat(s, 32, 1)
    y = np.abs(x / sf)
    err = np.abs(x.astype(np.float64) - deq)
    unclipped = y <= 6
    hg = _grid_half_gap(E2M1_GRID, np.minimum(y, 6.0))
    assert np.all(err[unclipped] <= (hg * sf)[unclipped] * (1 + 2.0 ** -20))
    assert np.all(err[~unclipped] < 2 * sf[~unclipped])
    # dequant is exact, so quantize(dequant) is the identity on scales, values and codes
    # (up to the sign of zero: -0.0 re-encodes as +0 because sign(-0.0) == 0)
    c2, e2, d2 = oracle.quant_mxfp4(deq)
    assert np.array_equal(e2, e8) and np.array_equal(d2, deq)
    assert np.array_equal(_fp4_codes_mod_zero_sign(c2), _fp4_codes_mod_zero_sign(codes))


def test_mxfp4_exponent_is_exact_below_power_of_two():
    # amax just below 2^5: floor(log2) is 4, so the scale is 2^2 and the code 6 * 4 = 24 < 32
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = np.nextafter(np.float32(32.0), np.float32(0))
    _, e8, _ = oracle.quant_mxfp4(x)
    assert int(e8[0, 0]) - 127 == 4 - 2


def test_nvfp4_invariants():
    x = _outlier_tensor()
    codes, sb, g, deq = oracle.quant_nvfp4(x)
    amax = np.abs(x).max()
    assert g == np.float32(amax / np.float32(2688.0))
    assert np.all((sb & 0x7F) <= 0x7E) and not np.any(sb & 0x80)     # all block scales <= 448
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sb[r, c // 16] == 0x7E                                      # the amax block gets 448
    # error bound with the effective scale max(b, 1e-12) * g
    b = np.array([oracle.e4m3_decode(v) for v in range(256)])[sb]
    seff = (np.maximum(b, np.float32(1e-12)).astype(np.float32) * np.float32(g)).astype(np.float64)
    sf = np.repeat(seff, 16, 1)
    y = np.abs(x / sf)
    err = np.abs(x.astype(np.float64) - deq)
    unclipped = y <= 6
    hg = _grid_half_gap(E2M1_GRID, np.minimum(y, 6.0))
    assert np.all(err[unclipped] <= (hg * sf)[unclipped] * (1 + 2.0 ** -20) + 2.0 ** -24 * np.abs(x[unclipped]))
    # each block's largest |x| encodes to magnitude 6 (E2M1 index 7): the block scale is
    # amax16 / 6 / g rounded to E4M3, within 1/16 relative wherever that E4M3 value is normal
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(x.shape[0], -1, 16)
    top = np.abs(x).reshape(x.shape[0], -1, 16).argmax(axis=2)
    top_idx = np.take_along_axis(nib, top[..., None], axis=2)[..., 0] & 0x7
    normal = b >= 2.0 ** -6
    assert normal.sum() > normal.size // 2 and np.all(top_idx[normal] == 7)
    # given amax reproduces the computed path
    c2, s2, g2, d2 = oracle.quant_nvfp4(x, amax_in=float(amax))
    assert np.array_equal(c2, codes) and np.array_equal(s2, sb) and g2 == g


def test_nvfp4_block_scale_rounding_to_zero_keeps_codes_of_page():
    # A block far below the tensor amax: its E4M3 block scale rounds to 0, the
    # effective scale is 1e-12 * g, and every non-zero value clips to +-6.
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1000.0
    x[0, 16:] = 1e-7
    codes, sb, g, deq = oracle.quant_nvfp4(x)
    assert sb[0, 1] == 0
    assert all((codes[0, 8 + i] & 0xF) == 0x7 and (codes[0, 8 + i] >> 4) == 0x7 for i in range(8))
    # and dequantizes to 6 * (1e-12 * g) in fp32, not to 0 (the floor applies before the product)
    s_eff = np.float32(np.float32(1e-12) * np.float32(g))
    assert np.all(deq[0, 16:] == np.float32(6.0) * s_eff) and s_eff > 0


def test_int4_g128_invariants():
    rng = np.random.default_rng(9)
    w = rng.standard_normal((512, 96)).astype(np.float32) * np.float32(0.02)
    qw, sc, deq = oracle.quant_int4_g128(w)
    q = ((qw.view(np.uint32)[:, None, :] >> (4 * np.arange(8, dtype=np.uint32))[None, :, None]) & 0xF)
    q = q.reshape(512, 96).astype(np.int64)
    q[q >= 8] -= 16
    s = np.array([[oracle.bf16_to_f32(v) for v in row] for row in sc], np.float64)
    sf = np.repeat(s, 128, 0)
    assert np.array_equal(q * sf, deq.astype(np.float64))              # dequant = q * s exactly
    assert q.min() >= -8 and q.max() <= 7
    amax = np.abs(w.reshape(4, 128, 96)).max(1)
    assert np.array_equal(sc, np.array([[oracle.f32_to_bf16(v) for v in row]
                                        for row in (amax / np.float32(7)).astype(np.float32)], np.uint16))
    err = np.abs(w - deq)
    assert np.all(err <= 0.5 * sf * (1 + 2.0 ** -20) + 2.0 ** -24 * np.abs(w) + 0.02 * sf * (np.abs(w / sf) > 7))
    qw2, sc2, d2 = oracle.quant_int4_g128(deq)
    assert np.array_equal(qw2, qw) and np.array_equal(sc2, sc)


def test_kv_write_is_per_tensor_on_k_and_v():
    rng = np.random.default_rng(2)
    k = (rng.standard_normal((1, 2, 16, 64)) + 5).astype(np.float32)
    v = rng.standard_normal((1, 2, 16, 64)).astype(np.float32)
    kb = torch.from_numpy(k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vb = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kc, vc, ks, vs, kd, vd = oracle.kv_write_fp8(kb, vb, want_deq=True)
    kf = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).float().numpy()
    vf = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert ks == np.float32(np.abs(kf).max() / np.float32(448))
    assert vs == np.float32(np.abs(vf).max() / np.float32(448))
    assert kc.ravel()[np.argmax(np.abs(kf))] & 0x7F == 0x7E
    assert vc.ravel()[np.argmax(np.abs(vf))] & 0x7F == 0x7E
    # the given-scale mode with the computed scale reproduces the codes
    c2, _ = oracle.quant_fp8_given(kb, ks)
    assert np.array_equal(c2, kc)


# ----------------------------------------------------------------- GEMMs

def _int_fp8_codes(rng, shape):
    vals = rng.integers(-8, 9, shape)
    codes = np.array([oracle.e4m3_encode(f32(v)) for v in vals.ravel()], np.uint8).reshape(shape)
    return vals, codes


def test_gemm_fp8_block_integer_case_is_exact_matmul():
    rng = np.random.default_rng(21)
    M, N, K = 3, 5, 256                          # non-square: a transposed operand fails
    a, qa = _int_fp8_codes(rng, (M, K))
    b, qb = _int_fp8_codes(rng, (N, K))
    y, bound = oracle.gemm_fp8_block(qa, np.ones((M, 2), np.float32), qb, np.ones((1, 2), np.float32))
    assert np.array_equal(y, (a @ b.T).astype(np.float64))
    assert np.array_equal(bound, (np.abs(a) @ np.abs(b).T).astype(np.float64))


def _fp4_pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def test_gemm_fp4_integer_case_is_exact_matmul():
    rng = np.random.default_rng(22)
    M, N, K = 4, 6, 64
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    va = np.vectorize(oracle.e2m1_decode)(ca)
    vb = np.vectorize(oracle.e2m1_decode)(cb)
    ref = va @ vb.T
    one_e4m3 = np.full((M, K // 16), 0x38, np.uint8)
    y, _ = oracle.gemm_nvfp4(_fp4_pack(ca), one_e4m3, 1.0, _fp4_pack(cb),
                             np.full((N, K // 16), 0x38, np.uint8), 1.0)
    assert np.array_equal(y, ref)
    y, _ = oracle.gemm_mxfp4(_fp4_pack(ca), np.full((M, K // 32), 127, np.uint8), _fp4_pack(cb),
                             np.full((N, K // 32), 127, np.uint8))
    assert np.array_equal(y, ref)


def test_gemm_w4a16_integer_case_is_exact_matmul():
    rng = np.random.default_rng(23)
    M, N, K = 3, 8, 256
    q = rng.integers(-8, 8, (K, N))
    qw = np.zeros((K // 8, N), np.uint32)
    for k in range(K):
        qw[k // 8] |= (q[k].astype(np.uint32) & 0xF) << np.uint32(4 * (k % 8))
    a = rng.integers(-4, 5, (M, K))
    A = np.array([[oracle.f32_to_bf16(f32(v)) for v in row] for row in a], np.uint16)
    sc = np.full((K // 128, N), 0x3F80, np.uint16)                      # bf16 1.0
    y, bound = oracle.gemm_w4a16(A, qw.view(np.int32), sc)
    assert np.array_equal(y, (a @ q).astype(np.float64))
    assert np.array_equal(bound, (np.abs(a) @ np.abs(q)).astype(np.float64))


def test_gemm_scale_indexing_matches_quantizer_dequant():
    """The GEMM references read the scales at the right (row, block) indices: they
    agree with numpy's matmul of the quantizers' own dequantized outputs."""
    rng = np.random.default_rng(24)
    M, N, K = 48, 256, 512
    A = (rng.standard_normal((M, K)) * rng.uniform(0.1, 10, (M, 1))).astype(np.float32)
    Bt = (rng.standard_normal((N, K)) * rng.uniform(0.1, 10, (1, K))).astype(np.float32)

    qa, sa, da = oracle.quant_fp8(A, oracle.FP8_GROUP_1x128)
    qb, sb, db = oracle.quant_fp8(Bt, oracle.FP8_BLOCK_128x128)
    y, bound = oracle.gemm_fp8_block(qa, sa, qb, sb)
    assert np.all(np.abs(y - da.astype(np.float64) @ db.astype(np.float64).T) <= 2.0 ** -22 * bound)

    ca, ea, da = oracle.quant_mxfp4(A)
    cb, eb, db = oracle.quant_mxfp4(Bt)
    y, bound = oracle.gemm_mxfp4(ca, ea, cb, eb)
    assert np.all(np.abs(y - da.astype(np.float64) @ db.astype(np.float64).T) <= 2.0 ** -40 * bound)

    ca, sa4, ga, da = oracle.quant_nvfp4(A)
    cb, sb4, gb, db = oracle.quant_nvfp4(Bt)
    y, bound = oracle.gemm_nvfp4(ca, sa4, ga, cb, sb4, gb)
    assert np.all(np.abs(y - da.astype(np.float64) @ db.astype(np.float64).T) <= 2.0 ** -21 * bound)

    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    Ab = np.array([[oracle.f32_to_bf16(v) for v in row] for row in A], np.uint16)
    qw, sc, dw = oracle.quant_int4_g128(W)
    y, bound = oracle.gemm_w4a16(Ab, qw, sc)
    af = (Ab.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.abs(y - af @ dw.astype(np.float64)) <= 2.0 ** -40 * bound)


def test_gemm_sampled_points_match_full():
    rng = np.random.default_rng(25)
    A = rng.standard_normal((16, 256)).astype(np.float32)
    B = rng.standard_normal((128, 256)).astype(np.float32)
    qa, sa, _ = oracle.quant_fp8(A, oracle.FP8_GROUP_1x128)
    qb, sb, _ = oracle.quant_fp8(B, oracle.FP8_BLOCK_128x128)
    yf, bf = oracle.gemm_fp8_block(qa, sa, qb, sb)
    ii, jj = rng.integers(0, 16, 50), rng.integers(0, 128, 50)
    ys, bs = oracle.gemm_fp8_block(qa, sa, qb, sb, ii, jj)
    assert np.array_equal(ys, yf[ii, jj]) and np.array_equal(bs, bf[ii, jj])


# ------------------------------------------------------ next rows: KV variants

def _kv_small(seed, B=2, H=3, T=16, D=64, bias_std=4.0):
    import synthetic as syn
    return syn.kv_cache_inputs(seed=seed, B=B, H=H, T=T, D=D, bias_std=bias_std)


def test_kv_per_head_reduces_to_per_tensor_per_head():
    """Each head's slice quantized alone by the per-tensor FP8 steps (pinned above) gives
    exactly the per-head result; the largest element of every head maps to +-448."""
    k, v = _kv_small(3)
    kc, vc, ks, vs, kd, vd = oracle.kv_write_fp8_per_head(k, v, want_deq=True)
    B, H, T, D = k.shape
    for b in range(B):
        for h in range(H):
            for x, c, s in ((k, kc, ks), (v, vc, vs)):
                rc, rs, _ = oracle.quant_fp8(x[b, h], oracle.FP8_PER_TENSOR, want_deq=False)
                assert np.array_equal(c[b, h], rc) and np.float32(s[b, h]) == rs[0]
                xf = (x[b, h].astype(np.uint32) << 16).view(np.float32)
                i = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
                assert c[b, h][i] & 0x7F == 0x7E


def test_kv_per_head_power_of_two_head_scaling():
    """Scaling one head by 2^3 multiplies only that head's scale by 8; all codes stay."""
    import synthetic as syn
    k, v = _kv_small(4)
    kf = (k.astype(np.uint32) << 16).view(np.float32).copy()
    kf[1, 2] *= np.float32(8.0)
    k2 = syn.to_bf16_bits(kf)
    a = oracle.kv_write_fp8_per_head(k, v)
    b = oracle.kv_write_fp8_per_head(k2, v)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ratio = b[2] / a[2]
    assert ratio[1, 2] == 8.0 and np.all(np.delete(ratio.ravel(), 1 * 3 + 2) == 1.0)


def test_kv_per_head_given_matches_per_tensor_given():
    k, _ = _kv_small(5)
    scales = np.array([[0.01, 0.02, 0.5], [1.0, 0.003, 0.25]], np.float32)
    codes, _ = oracle.kv_fp8_per_head_given(k, scales)
    for b in range(2):
        for h in range(3):
            rc, _ = oracle.quant_fp8_given(k[b, h], float(scales[b, h]), want_deq=False)
            assert np.array_equal(codes[b, h], rc)


def test_k_channel_zero_point_extremes_map_to_full_range():
    """Per channel the residual is centred: the channel's largest and smallest values map
    to +448 and -448 (codes 0x7E and 0xFE), whatever the channel's constant bias."""
    k, _ = _kv_small(6, T=32)
    codes, sc, zp, _ = oracle.kv_k_channel_zp(k)
    kf = (k.astype(np.uint32) << 16).view(np.float32)
    B, H, T, D = k.shape
    for b in range(B):
        for h in range(H):
            for d in range(D):
                col = kf[b, h, :, d]
                if col.max() == col.min():
                    continue
                assert codes[b, h, np.argmax(col), d] == 0x7E
                assert codes[b, h, np.argmin(col), d] == 0xFE


def test_k_channel_zero_point_unit_scale_reduces_to_plain_cast():
    """Channels spanning exactly [-448, 448]: zero point 0 and scale 1, so the codes are
    the plain E4M3 cast of the values (torch's float8_e4m3fn)."""
    import synthetic as syn
    rng = np.random.default_rng(19)
    x = rng.uniform(-448, 448, (1, 2, 40, 16)).astype(np.float32)
    x[:, :, 3, :] = 448.0
    x[:, :, 17, :] = -448.0
    xb = syn.to_bf16_bits(x)
    codes, sc, zp, _ = oracle.kv_k_channel_zp(xb)
    assert np.all(sc == 1.0) and np.all(zp == 0.0)
    xf = torch.from_numpy((xb.astype(np.uint32) << 16).view(np.float32))
    assert np.array_equal(codes, xf.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_k_channel_zero_point_is_translation_invariant():
    """Adding an exactly representable constant to every value of a channel moves its
    zero point by that constant and leaves codes and scales unchanged (values on a
    grid where every sum involved is exact in fp32 and bf16)."""
    import synthetic as syn
    rng = np.random.default_rng(7)
    i = rng.integers(-16, 17, (1, 2, 24, 8)).astype(np.float32) / 16.0      # steps of 1/16 in [-1, 1]
    c0, s0, z0, _ = oracle.kv_k_channel_zp(syn.to_bf16_bits(i))
    c4, s4, z4, _ = oracle.kv_k_channel_zp(syn.to_bf16_bits(i + np.float32(4.0)))
    assert np.array_equal(c0, c4) and np.array_equal(s0, s4)
    assert np.array_equal(z4 - z0, np.full_like(z0, 4.0))


def test_k_channel_zero_point_error_tracks_the_variation():
    """The dequantized K is within half an E4M3 step of the residual (plus the final
    rounding), so its error scales with each channel's variation, not its bias: on K
    with a per-channel bias of std 4 it is far below the per-tensor error."""
    import synthetic as syn
    k, _ = _kv_small(8, T=64)
    kf32 = (k.astype(np.uint32) << 16).view(np.float32).copy()
    kf32[:, :, 0, :8] += np.float32(6.0)               # some channels peak at the first token,
    kf32[:, :, -1, 8:16] -= np.float32(6.0)            # some bottom out at the last
    k = syn.to_bf16_bits(kf32)
    codes, sc, zp, deq = oracle.kv_k_channel_zp(k, want_deq=True)
    kf = (k.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = np.abs(kf - zp[:, :, None, :])
    s = sc[:, :, None, :].astype(np.float64)
    bound = 2.0 ** -4 * r + 2.0 ** -10 * s + 2.0 ** -22 * (np.abs(kf) + np.abs(zp[:, :, None, :]))
    assert np.all(np.abs(deq - kf) <= bound)
    _, _, _, _, kd_t, _ = oracle.kv_write_fp8(k, k, want_deq=True)
    assert np.mean(np.abs(deq - kf)) < 0.5 * np.mean(np.abs(kd_t - kf))


# ------------------------------------------------- next rows: INT4 zero point

def test_int4_zp_worked_example():
    """A group spanning [-0.75, 3.0] in steps of 0.25: s = 3.75 / 15 = 0.25 exactly,
    z = 3, and each value x maps to x / 0.25 + 3."""
    vals = np.tile(np.arange(-3, 13, dtype=np.float32) * np.float32(0.25), 8)      # 128 values
    w = vals.reshape(128, 1).repeat(64, axis=1)
    qw, sc, zp, deq = oracle.quant_int4_g128_zp(w)
    assert np.all(sc == 0x3E80) and np.all(zp == 3)                                 # bf16 0.25
    codes = (qw.view(np.uint32)[:, :, None] >> (4 * np.arange(8))[None, None, :]) & 0xF
    codes = codes.transpose(0, 2, 1).reshape(128, 64)
    assert np.array_equal(codes[:, 0], (vals / np.float32(0.25) + 3).astype(np.int64))
    assert np.array_equal(deq, w)


def test_int4_zp_invariants():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((512, 96)) * 0.02).astype(np.float32)
    w[:, 5] = np.abs(w[:, 5])                          # an all-positive column: z = 0
    w[:, 6] = np.float32(1.0) + np.abs(w[:, 6])        # all values far above 0: the range still starts at 0
    w[:128, 7] = 0.0                                   # an all-zero group
    qw, sc, zp, deq = oracle.quant_int4_g128_zp(w)
    s = (sc.astype(np.uint32) << 16).view(np.float32)
    codes = ((qw.view(np.uint32)[:, :, None] >> (4 * np.arange(8))[None, None, :]) & 0xF)
    codes = codes.transpose(0, 2, 1).reshape(512, 96)
    assert np.all(zp <= 15)
    assert np.all(zp[:, 5] == 0) and np.all(zp[:, 6] == 0) and zp[0, 7] == 0 and np.all(codes[:128, 7] == 0)
    srep = np.repeat(s, 128, axis=0)
    assert np.all(np.abs(deq.astype(np.float64) - w) <= 0.55 * srep)
    for g in range(4):
        grp, cg, z = w[g * 128:(g + 1) * 128], codes[g * 128:(g + 1) * 128], zp[g]
        for n in range(96):
            if grp[:, n].min() < 0:
                assert cg[np.argmin(grp[:, n]), n] == 0          # the minimum sits on code 0
            if grp[:, n].max() > 0:
                assert cg[np.argmax(grp[:, n]), n] >= 14         # the maximum on the top codes
    # quantizing the dequantized weight again reproduces codes, scales and zero points
    # in every group whose codes reach both ends of the range
    qw2, sc2, zp2, _ = oracle.quant_int4_g128_zp(deq)
    full = np.zeros((4, 96), bool)
    for g in range(4):
        cg = codes[g * 128:(g + 1) * 128]
        full[g] = (cg.min(axis=0) == 0) & (cg.max(axis=0) == 15)
    assert full.sum() > 50
    assert np.array_equal(sc2[full], sc[full]) and np.array_equal(zp2[full], zp[full])
    codes2 = ((qw2.view(np.uint32)[:, :, None] >> (4 * np.arange(8))[None, None, :]) & 0xF)
    codes2 = codes2.transpose(0, 2, 1).reshape(512, 96)
    fullk = np.repeat(full, 128, axis=0)
    assert np.array_equal(codes2[fullk], codes[fullk])


def test_gemm_w4a16_zp_integer_case_is_exact_matmul():
    """Unit scales, integer activations: the reference equals the integer matmul
    A (q - z) exactly (numpy, int64)."""
    import synthetic as syn
    rng = np.random.default_rng(12)
    M, K, N = 5, 256, 24
    A = rng.integers(-20, 21, (M, K)).astype(np.float32)
    q = rng.integers(0, 16, (K, N)).astype(np.int64)
    z = rng.integers(0, 16, (K // 128, N)).astype(np.uint8)
    qw = np.zeros((K // 8, N), np.uint32)
    for k in range(K):
        qw[k // 8] |= (q[k].astype(np.uint32) << np.uint32(4 * (k % 8)))
    sc = np.full((K // 128, N), 0x3F80, np.uint16)
    y, bound = oracle.gemm_w4a16_zp(syn.to_bf16_bits(A), qw.view(np.int32), sc, z)
    deq = q - np.repeat(z.astype(np.int64), 128, axis=0)
    ref = A.astype(np.int64) @ deq
    assert np.array_equal(y, ref.astype(np.float64))
    assert np.array_equal(bound, (np.abs(A.astype(np.int64))[:, :, None] * np.abs(deq)[None]).sum(1))


# --------------------------------------------- next rows: weight-only FP4 GEMM

def test_gemm_w4a16_fp4_equals_matmul_of_decoded_weights():
    """Weight-only NVFP4 and MXFP4 references against a numpy matmul of the weights
    decoded element by element with the (pinned) E2M1 / E4M3 decoders."""
    import synthetic as syn
    rng = np.random.default_rng(13)
    M, N, K = 3, 20, 128
    A = syn.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    Af = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qB = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    codes = np.stack([qB & 0xF, qB >> 4], axis=-1).reshape(N, K)
    e2 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    sB = rng.integers(0x10, 0x70, (N, K // 16)).astype(np.uint8)
    e4 = np.array([oracle.e4m3_decode(c) for c in range(256)])
    gB = 0.375
    W = e2[codes] * np.repeat(e4[sB], 16, axis=1) * gB
    y, bound = oracle.gemm_w4a16_nvfp4(A, qB, sB, gB)
    np.testing.assert_allclose(y, Af @ W.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bound, np.abs(Af) @ np.abs(W).T, rtol=1e-12)
    eB = rng.integers(110, 140, (N, K // 32)).astype(np.uint8)
    W = e2[codes] * np.repeat(np.ldexp(1.0, eB.astype(np.int64) - 127), 32, axis=1)
    y, bound = oracle.gemm_w4a16_mxfp4(A, qB, eB)
    np.testing.assert_allclose(y, Af @ W.T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------- next rows: SmoothQuant + INT8

def test_col_amax_matches_numpy():
    import synthetic as syn
    rng = np.random.default_rng(14)
    x = rng.standard_normal((37, 50)).astype(np.float32)
    assert np.array_equal(oracle.col_amax(x), np.abs(x).max(axis=0))
    b = syn.to_bf16_bits(x)
    assert np.array_equal(oracle.col_amax(b), np.abs((b.astype(np.uint32) << 16).view(np.float32)).max(axis=0))


def test_smooth_factors_closed_forms():
    """alpha = 0.5: equal amaxes give 1, a ratio of 4 gives 2 (exactly), a zero amax
    takes the 1e-12 floor, and s^2 = ax / aw to a few fp32 ulps."""
    xm = np.array([3.0, 12.0, 0.5, 0.0, 7.0], np.float32)
    wm = np.array([3.0, 3.0, 2.0, 4.0, 0.0], np.float32)
    s = oracle.smooth_factors(xm, wm)
    assert s[0] == 1.0 and s[1] == 2.0 and s[2] == 0.5
    assert s[3] == np.float32(np.sqrt(np.float32(1e-12))) / np.float32(2.0)
    rng = np.random.default_rng(15)
    xm = rng.uniform(0.01, 100, 1000).astype(np.float32)
    wm = rng.uniform(0.001, 1, 1000).astype(np.float32)
    s = oracle.smooth_factors(xm, wm).astype(np.float64)
    np.testing.assert_allclose(s * s, xm.astype(np.float64) / wm, rtol=4e-7)


def test_int8_rows_worked_example():
    """amax 127 gives s = 1, so q = rint(x) with halves to even, and -127 at the minimum."""
    x = np.array([[2.5, 3.5, -2.5, 127.0, -127.0, 0.4, -0.6, 126.5]], np.float32)
    q, s, deq = oracle.quant_int8_rows(x)
    assert s[0] == 1.0
    assert q.tolist() == [[2, 4, -2, 127, -127, 0, -1, 126]]


def test_int8_rows_invariants_and_smoothing():
    rng = np.random.default_rng(16)
    x = rng.standard_normal((20, 256)).astype(np.float32)
    x[:, 9] *= np.float32(40.0)
    q, s, deq = oracle.quant_int8_rows(x)
    assert np.all(np.abs(q).max(axis=1) == 127)
    assert np.all(np.abs(deq.astype(np.float64) - x) <= 0.5 * s[:, None] * (1 + 2.0 ** -20))
    ones = np.ones(256, np.float32)
    for mode in (oracle.INT8_DIVIDE, oracle.INT8_MULTIPLY):
        q1, s1, _ = oracle.quant_int8_rows(x, ones, mode)
        assert np.array_equal(q1, q) and np.array_equal(s1, s)
    four = np.full(256, 4.0, np.float32)
    qm, sm, _ = oracle.quant_int8_rows(x, four, oracle.INT8_MULTIPLY)
    qd, sd, _ = oracle.quant_int8_rows(x, four, oracle.INT8_DIVIDE)
    assert np.array_equal(qm, q) and np.array_equal(sm, 4 * s)
    assert np.array_equal(qd, q) and np.array_equal(sd, s / 4)


def test_smoothquant_int8_pipeline_preserves_the_product():
    """X / s and W^T * s quantized per token and per output channel: the INT8 GEMM
    reference stays close to X W (the migration leaves the product unchanged), and
    closer than without smoothing on activations with outlier channels."""
    rng = np.random.default_rng(17)
    M, K, N = 32, 256, 48
    X = rng.standard_normal((M, K)).astype(np.float32)
    X[:, rng.choice(K, 3, replace=False)] *= np.float32(60.0)
    Wt = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)       # B^T [N, K]
    s = oracle.smooth_factors(oracle.col_amax(X), oracle.col_amax(Wt))
    qa, sa, _ = oracle.quant_int8_rows(X, s, oracle.INT8_DIVIDE)
    qb, sb, _ = oracle.quant_int8_rows(Wt, s, oracle.INT8_MULTIPLY)
    y, _ = oracle.gemm_int8(qa, sa, qb, sb)
    exact = X.astype(np.float64) @ Wt.T.astype(np.float64)
    err_smooth = np.abs(y - exact).mean()
    qa0, sa0, _ = oracle.quant_int8_rows(X)
    qb0, sb0, _ = oracle.quant_int8_rows(Wt)
    y0, _ = oracle.gemm_int8(qa0, sa0, qb0, sb0)
    err_plain = np.abs(y0 - exact).mean()
    assert err_smooth < 0.05 * np.abs(exact).mean()
    assert err_smooth < 0.7 * err_plain


def test_gemm_int8_is_scaled_integer_matmul():
    rng = np.random.default_rng(18)
    M, N, K = 9, 14, 384
    qa = rng.integers(-128, 128, (M, K)).astype(np.int8)
    qb = rng.integers(-128, 128, (N, K)).astype(np.int8)
    sa = rng.uniform(0.001, 1, M).astype(np.float32)
    sb = rng.uniform(0.001, 1, N).astype(np.float32)
    y, bound = oracle.gemm_int8(qa, sa, qb, sb)
    acc = qa.astype(np.int64) @ qb.T.astype(np.int64)
    sc = sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
    np.testing.assert_allclose(y, acc * sc, rtol=1e-15)
    np.testing.assert_allclose(bound, (np.abs(qa.astype(np.int64)) @ np.abs(qb.T.astype(np.int64))) * sc,
                               rtol=1e-15)

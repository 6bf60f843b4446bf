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

"""The seeded synthetic inputs follow the stated recipe (CPU): shapes, dtypes, the
distributions (N(0, 0.02) weights, N(0, 1) activations), the number and scale of the
outlier channels, the Qwen3-0.6B linear set, the K-cache's per-channel bias, and
determinism per seed. The generators draw numbers only; nothing here quantizes."""
import numpy as np

import synthetic as syn


def _std_ok(x, want, rel=0.05):
    return abs(float(np.std(x)) - want) <= rel * want


def test_seeded_and_distinct():
    a = syn.quant_roundtrip_input(seed=3)
    assert np.array_equal(a, syn.quant_roundtrip_input(seed=3))
    assert not np.array_equal(a, syn.quant_roundtrip_input(seed=4))


def test_quant_roundtrip_input_outlier_columns():
    x = syn.quant_roundtrip_input(seed=0)
    assert x.shape == (1024, 1024) and x.dtype == np.float32
    col_std = x.std(axis=0)
    out = np.flatnonzero(col_std > 0.2)
    assert len(out) == 8                                         # 8 seeded columns
    assert np.all(np.abs(col_std[out] / 1.0 - 1) < 0.1)           # x50 of N(0, 0.02)
    rest = np.delete(x, out, axis=1)
    assert _std_ok(rest, 0.02) and abs(float(rest.mean())) < 1e-3


def test_w4a16_inputs_recipe():
    M, K, N = 16, 4096, 512
    a_bits, w = syn.w4a16_decode_inputs(M, seed=0, K=K, N=N)
    a = syn.bf16_bits_to_f32(a_bits)
    assert a_bits.shape == (M, K) and a_bits.dtype == np.uint16
    assert w.shape == (K, N) and w.dtype == np.float32 and _std_ok(w, 0.02)
    # round(1% of K) = 41 channels x20, the same channels in every row
    big = np.abs(a) > 8.0
    chans = np.flatnonzero(big.any(axis=0))
    assert len(chans) == 41
    assert np.all(np.abs(a[:, chans]).mean(axis=0) > 5.0)
    rest = np.delete(a, chans, axis=1)
    assert _std_ok(rest, 1.0) and np.abs(rest).max() < 6.5


def test_fp8_and_fp4_gemm_inputs_recipe():
    a_bits, bt_bits = syn.fp8_block_gemm_inputs(seed=1, M=256, K=1024, N=384)
    assert a_bits.shape == (256, 1024) and bt_bits.shape == (384, 1024)
    a, bt = syn.bf16_bits_to_f32(a_bits), syn.bf16_bits_to_f32(bt_bits)
    assert len(np.flatnonzero(np.abs(a).max(axis=0) > 8.0)) == round(0.01 * 1024)
    assert _std_ok(bt, 0.02)
    a_bits, bt_bits = syn.fp4_gemm_inputs(seed=2, M=256, K=4096, N=256)
    a = syn.bf16_bits_to_f32(a_bits)
    chans = np.flatnonzero(np.abs(a).max(axis=0) > 8.0)
    assert len(chans) == 20                                       # 0.5% of 4096, x30
    assert np.all(np.abs(a[:, chans]).mean(axis=0) > 8.0)
    assert bt_bits.shape == (256, 4096) and _std_ok(syn.bf16_bits_to_f32(bt_bits), 0.02)


def test_qwen3_linear_set():
    got = list(syn.qwen3_decode_linears(layers=2, tokens=4, seed=0))
    assert len(got) == 2 * 7
    shapes = [(name, w.shape) for _, name, _, w in got[:7]]
    assert shapes == [("q_proj", (1024, 2048)), ("k_proj", (1024, 1024)), ("v_proj", (1024, 1024)),
                      ("o_proj", (2048, 1024)), ("gate_proj", (1024, 3072)), ("up_proj", (1024, 3072)),
                      ("down_proj", (3072, 1024))]
    # 28 layers x 7 linears = 196 GEMMs, 440,401,920 weights in all
    assert 28 * sum(K * N for _, K, N in syn.QWEN3_LINEARS) == 440_401_920
    for layer, name, a_bits, w in got:
        assert a_bits.shape == (4, w.shape[0]) and _std_ok(w, 0.02)
    # every (layer, projection) draws its own weights
    assert not np.array_equal(got[1][3], got[2][3])
    assert not np.array_equal(got[0][3], got[7][3])


def test_kv_cache_bias_structure():
    k_bits, v_bits = syn.kv_cache_inputs(seed=0, T=512)
    k = syn.bf16_bits_to_f32(k_bits).astype(np.float64)
    v = syn.bf16_bits_to_f32(v_bits).astype(np.float64)
    assert k.shape == v.shape == (1, 8, 512, 128)
    chan_mean = k.mean(axis=2)                                   # over tokens: the bias
    resid = k - chan_mean[:, :, None, :]
    assert abs(chan_mean.std() - 4.0) < 0.4                       # bias ~ N(0, 4) per (h, d)
    assert abs(resid.std() - 1.0) < 0.05                          # N(0, 1) around it
    assert abs(v.std() - 1.0) < 0.05 and abs(v.mean()) < 0.01


def test_bf16_bits_round_trip():
    x = np.array([0.0, -0.0, 1.0, -2.5, 3.140625, 65280.0, 1e-30], np.float32)
    b = syn.to_bf16_bits(x)
    back = syn.bf16_bits_to_f32(b)
    assert np.array_equal(syn.to_bf16_bits(back), b)
    assert np.array_equal(back[:6], x[:6])                       # bf16-representable values stay

"""Pins for the CPU oracle: the pages' printed numbers, closed forms, invariants
and brute force on tiny inputs.  Each test would fail under a plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand)."""
import itertools
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import native
from tests.conftest import golden_numbers

G = golden_numbers()
L = native.lib()


# ---------------------------------------------------------------- accounting
def test_entry_sizes_match_pages():
    assert oracle.entry_bytes(512, 16) == G["main_entry_bytes"]
    assert oracle.entry_bytes(128, 32) == G["index_entry_bytes"]
    assert 512 / 2 == G["main_entry_code_bytes"] and 512 / 16 == G["main_entry_scale_bytes"]


def test_890_bytes_per_token_arithmetic():
    ratios = [2, 2, 2, 1]
    assert sum(1 / m for m in ratios) == G["sum_inverse_ratio"]
    assert oracle.global_bytes_per_token(ratios) == G["global_bytes_per_token"]
    assert 288 * 2.5 == G["main_subtotal"] and 68 * 2.5 == G["index_subtotal"]
    assert abs(G["global_bytes_per_token"] * 1e6 / 1e9 - G["resident_gb_at_1m"]) < 1e-12


def test_v4flash_chain_arithmetic():
    assert oracle.v4flash_bytes_per_token() == G["v4flash_bytes_per_token"]
    assert 448 + 64 * 2 + 8 == G["v4flash_main_entry"]
    step1 = 4 * (G["v4flash_main_entry"] + 68) / 4
    assert step1 == G["after_cross_layer_reuse"]
    step2 = step1 * 2.5
    assert step2 == G["after_relaxed_ratio"]
    step3 = step2 * (288 + 68) / (G["v4flash_main_entry"] + 68)
    assert step3 == G["after_fp4_main"]
    assert round(G["v4flash_bytes_per_token"] / step3, 2) == 3.95


def test_cache_write_emits_890_bytes_per_token():
    """Four source layers (three at m=2, one at m=1) over the same tokens write
    exactly 890 bytes per token through the oracle's own cache write."""
    g = synth.rng(11)
    T = 16
    x = synth.latents(g, T)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    total = 0
    for m in (2, 2, 2, 1):
        main, codes, scales = oracle.compress_quantize(x, m, w0, w1, W)
        total += main.nbytes + codes.nbytes + scales.nbytes
    assert main.shape[1] == 288 and codes.shape[1] + scales.shape[1] == 68
    assert total / T == G["global_bytes_per_token"]


# ---------------------------------------------------------------- formats
def test_e2m1_grid_and_round_trip():
    vals = oracle.e2m1_values()
    assert vals.max() == G["e2m1_max"]
    np.testing.assert_array_equal(vals[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for code in range(16):
        assert L.oracle_e2m1_decode(code) == vals[code] or (code == 8 and vals[code] == 0)
        if code != 8:
            assert L.oracle_e2m1_encode(vals[code]) == code
    assert L.oracle_e2m1_encode(-0.0) == 8


@pytest.mark.parametrize("x,expect", [
    (0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
    (5.0, 4.0), (0.2499, 0.0), (0.2501, 0.5), (5.0001, 6.0), (7.0, 6.0), (1e30, 6.0),
])
def test_e2m1_ties_to_even_and_saturation(x, expect):
    vals = oracle.e2m1_values()
    assert vals[L.oracle_e2m1_encode(x)] == expect
    assert vals[L.oracle_e2m1_encode(-x)] == -expect


def test_e2m1_small_negative_keeps_sign():
    assert L.oracle_e2m1_encode(-0.1) == 8


def test_e4m3_round_trip_all_finite_codes():
    vals = oracle.e4m3_values()
    assert np.nanmax(vals) == G["e4m3_max"]
    for code in range(0x7F):
        assert L.oracle_e4m3_decode(code) == vals[code]
        if code:
            assert L.oracle_e4m3_encode(vals[code]) == code


def test_e4m3_rounding_and_saturation():
    vals = oracle.e4m3_values()
    assert vals[L.oracle_e4m3_encode(500.0)] == 448.0
    assert vals[L.oracle_e4m3_encode(1e9)] == 448.0
    assert vals[L.oracle_e4m3_encode(2.0 ** -10)] == 0.0          # tie 0 | 2^-9 -> even (0)
    assert vals[L.oracle_e4m3_encode(3 * 2.0 ** -10)] == 2.0 ** -8  # tie 2^-9 | 2^-8 -> even code 2
    assert vals[L.oracle_e4m3_encode(1.0625)] == 1.0               # tie 1.0 | 1.125 -> even
    assert vals[L.oracle_e4m3_encode(1.1875)] == 1.25              # tie 1.125 | 1.25 -> even
    # brute force: the encoder picks a nearest representable value
    for x in np.linspace(0.001, 440, 2001).astype(np.float32):
        got = vals[L.oracle_e4m3_encode(float(x))]
        assert abs(got - x) == np.nanmin(np.abs(vals[:0x7F] - x))


def _group(y):
    y = np.ascontiguousarray(y, np.float32)
    codes = np.zeros(8, np.uint8)
    scale = np.zeros(1, np.uint8)
    L.oracle_fp4_group_quantize(native.ptr(y), native.ptr(codes), native.ptr(scale))
    return codes, int(scale[0])


def test_main_fp4_round_trip_every_scale_and_code():
    """Every E2M1 code times every positive finite E4M3 scale survives a round
    trip when the group's maximum is 6*s (so amax/6 is exactly s)."""
    e2m1 = oracle.e2m1_values()
    e4m3 = oracle.e4m3_values()
    for s_code in range(1, 0x7F):
        s = e4m3[s_code]
        codes_in = np.array([7] + list(range(16)[:15]), np.uint8)   # one element at 6*s
        y = (e2m1[codes_in] * s).astype(np.float32)
        assert np.all(y.astype(np.float64) == e2m1[codes_in] * s)    # exact in binary32
        codes, scale = _group(y)
        assert scale == s_code
        got = np.stack([codes & 15, codes >> 4], -1).ravel()
        want = codes_in.copy()
        want[(e2m1[codes_in] == 0)] = codes_in[(e2m1[codes_in] == 0)]
        np.testing.assert_array_equal(e2m1[got] * s, e2m1[codes_in] * s)


def test_main_fp4_saturation_2688():
    y = np.zeros(16, np.float32)
    y[0] = G["fp4_max_magnitude"]
    y[1] = -G["fp4_max_magnitude"]
    y[2] = 5000.0
    codes, scale = _group(y)
    assert oracle.e4m3_values()[scale] == 448.0
    deq = oracle.dequant_main(np.concatenate([np.tile(codes, 32), np.full(32, scale, np.uint8)]))
    assert deq[0] == 2688.0 and deq[1] == -2688.0 and deq[2] == 2688.0
    assert 6 * 448 == G["fp4_max_magnitude"]


def test_main_fp4_zero_and_tiny_group():
    codes, scale = _group(np.zeros(16, np.float32))
    assert scale == 0 and not codes.any()
    codes, scale = _group(np.full(16, -1e-6, np.float32))   # amax/6 rounds to E4M3 zero
    assert scale == 0 and not codes.any()


def _mx(v):
    v = np.ascontiguousarray(v, np.float32)
    codes = np.zeros(16, np.uint8)
    scale = np.zeros(1, np.uint8)
    L.oracle_mxfp4_block_quantize(native.ptr(v), native.ptr(codes), native.ptr(scale))
    return codes, int(scale[0])


@pytest.mark.parametrize("X", [-20, -3, 0, 1, 7, 40])
def test_mxfp4_grid_round_trip(X):
    e2m1 = oracle.e2m1_values()
    g = np.random.default_rng(X + 100)
    codes_in = g.integers(0, 16, 32).astype(np.uint8)
    codes_in[5] = 7                                           # amax = 6 * 2^X
    v = (e2m1[codes_in] * 2.0 ** X).astype(np.float32)
    codes, scale = _mx(v)
    assert scale == X + 127                                   # floor(log2(6*2^X)) - 2 = X
    got = np.stack([codes & 15, codes >> 4], -1).ravel()
    np.testing.assert_array_equal(e2m1[got], e2m1[codes_in])


def test_mxfp4_scale_rule_and_zero_block():
    codes, scale = _mx(np.zeros(32))
    assert scale == 0 and not codes.any()
    v = np.zeros(32, np.float32)
    v[3] = 7.9                                               # floor(log2 7.9) = 2 -> X = 0
    codes, scale = _mx(v)
    assert scale == 127 and oracle.e2m1_values()[(codes[1] >> 4)] == 6.0   # 7.9 saturates to 6
    v[3] = 8.0                                               # X = 1
    assert _mx(v)[1] == 128


# ---------------------------------------------------------------- cache-write stages
def _stages(x0, x1, m, w0, w1, pos, W=None):
    cs = oracle.rope_table(pos + 1)
    if W is None:
        W = np.zeros((128, 512), np.uint16)
    return oracle.entry_stages(x0, x1, m, w0, w1, cs[pos], W)


def test_compressor_equal_unit_weights_is_exact_mean():
    g = synth.rng(1)
    x0, x1 = synth.latents(g, 2)
    for w in (1.0, 2.0, 0.25):
        ones = np.full(512, w, np.float32)
        c, *_ = _stages(x0, x1, 2, ones, ones, 0)
        mean = ((synth.bf16_bits_to_f32(x0).astype(np.float64)
                 + synth.bf16_bits_to_f32(x1)) / 2).astype(np.float32)
        np.testing.assert_array_equal(c, mean)


def test_compressor_equal_weights_is_mean_within_three_roundings():
    """Equal non-power-of-two weights give the plain mean up to the three binary32
    roundings of w*x1, the fused multiply-add and the division."""
    g = synth.rng(2)
    x0, x1 = synth.latents(g, 2)
    w = np.full(512, 0.7310586, np.float32)
    c, *_ = _stages(x0, x1, 2, w, w, 0)
    a = synth.bf16_bits_to_f32(x0).astype(np.float64)
    b = synth.bf16_bits_to_f32(x1).astype(np.float64)
    mean = (a + b) / 2
    bound = 2.0 ** -24 * (np.abs(b) / 2 + (np.abs(a) + np.abs(b)) / 2 + np.abs(mean)) * 1.01
    assert np.all(np.abs(c - mean) <= bound)
    assert np.mean(c == mean.astype(np.float32)) > 0.5


def test_compressor_weights_order_and_m1_identity():
    g = synth.rng(3)
    x0, x1 = synth.latents(g, 2)
    w0 = np.full(512, 1.0, np.float32)
    w1 = np.full(512, 0.0, np.float32)
    c, *_ = _stages(x0, x1, 2, w0, w1, 0)        # w1 = 0 -> c is exactly the first token
    np.testing.assert_array_equal(c, synth.bf16_bits_to_f32(x0))
    c, *_ = _stages(x0, x1, 2, w1, w0, 0)        # w0 = 0 -> the second token
    np.testing.assert_array_equal(c, synth.bf16_bits_to_f32(x1))
    c, *_ = _stages(x0, None, 1, w0, w0, 0)
    np.testing.assert_array_equal(c, synth.bf16_bits_to_f32(x0))


def test_rmsnorm_unit_rms_and_constant_vector():
    g = synth.rng(4)
    x0 = synth.latents(g, 1)[0]
    w = np.ones(512, np.float32)
    c, yn, *_ = _stages(x0, None, 1, w, w, 0)
    ss = np.sum(yn.astype(np.float64) ** 2)
    assert abs(ss - 512) < 512 * 1e-5 * (1 + 512 * 1e-6)
    np.testing.assert_allclose(yn, c.astype(np.float64) / np.sqrt(np.mean(c.astype(np.float64) ** 2) + 1e-6),
                               rtol=2e-6)
    const = synth.f32_to_bf16_bits(np.full(512, 2.0, np.float32))
    _, yn, *_ = _stages(const, None, 1, w, w, 0)
    np.testing.assert_allclose(yn, 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-7)


def test_rope_identity_at_zero_norm_preserved_and_frequencies():
    g = synth.rng(5)
    x0 = synth.latents(g, 1)[0]
    w = np.ones(512, np.float32)
    _, yn, yr, _ = _stages(x0, None, 1, w, w, 0)
    np.testing.assert_array_equal(yr, yn)                      # position 0 is the identity
    cs = oracle.rope_table(1 << 12)
    ang = np.arctan2(cs[..., 1].astype(np.float64), cs[..., 0])
    # pair 0 turns by exactly 1 radian per position (theta^0)
    np.testing.assert_allclose(np.cos(ang[:, 0]), np.cos(np.arange(1 << 12)), atol=1e-6)
    # frequency ratio between consecutive pairs is theta^(-1/32) with theta = 160000
    f = ang[1, :]                                              # position 1: angle = frequency
    np.testing.assert_allclose(f[1:] / f[:-1], 160000.0 ** (-1 / 32), rtol=1e-6)
    # angle is linear in position: position 3 = 3 * position 1 (mod 2 pi)
    d = np.angle(np.exp(1j * (ang[3] - 3 * ang[1])))
    assert np.max(np.abs(d)) < 1e-6
    for pos in (1, 77, 4095):
        _, yn, yr, _ = _stages(x0, None, 1, w, w, pos)
        np.testing.assert_array_equal(yr[:448], yn[:448])          # NoPE part untouched
        a = yn[448:].astype(np.float64).reshape(32, 2)
        b = yr[448:].astype(np.float64).reshape(32, 2)
        np.testing.assert_allclose(np.hypot(b[:, 0], b[:, 1]), np.hypot(a[:, 0], a[:, 1]), rtol=1e-6)
        # interleaved pairs rotate counter-clockwise: (y0, y1) -> (y0 c - y1 s, y0 s + y1 c)
        c_, s_ = cs[pos, :, 0].astype(np.float64), cs[pos, :, 1].astype(np.float64)
        np.testing.assert_allclose(b[:, 0], a[:, 0] * c_ - a[:, 1] * s_, atol=1e-5)
        np.testing.assert_allclose(b[:, 1], a[:, 0] * s_ + a[:, 1] * c_, atol=1e-5)


def test_projection_one_hot_selects_column_and_is_linear():
    g = synth.rng(6)
    W = synth.index_projection(g)
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    for ch in (0, 17, 448, 511):
        y = np.zeros(512, np.float32)
        y[ch] = 1.0
        k = np.zeros(128, np.float32)
        L.oracle_project(native.ptr(y), native.ptr(W), native.ptr(k))
        np.testing.assert_array_equal(k, Wf[:, ch].astype(np.float32))
    y = g.standard_normal(512).astype(np.float32)
    k = np.zeros(128, np.float32)
    L.oracle_project(native.ptr(y), native.ptr(W), native.ptr(k))
    np.testing.assert_allclose(k, Wf @ y.astype(np.float64), rtol=1e-4, atol=1e-5)


def test_cache_write_entry_matches_stage_composition():
    """The bytes of a written entry equal the stage functions composed by hand,
    and decode back to the rotated latent within FP4 error."""
    g = synth.rng(7)
    x = synth.latents(g, 8)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    main, codes, scales = oracle.compress_quantize(x, 2, w0, w1, W, entry0=5)
    cs = oracle.rope_table(16)
    for j in range(4):
        _, _, yr, k = oracle.entry_stages(x[2 * j], x[2 * j + 1], 2, w0, w1, cs[5 + j], W)
        ent = np.zeros(288, np.uint8)
        L.oracle_main_entry(native.ptr(yr), native.ptr(ent))
        np.testing.assert_array_equal(main[j], ent)
        c2, s2 = oracle.mxfp4_quantize(k[None])
        np.testing.assert_array_equal(codes[j], c2[0])
        np.testing.assert_array_equal(scales[j], s2[0])
        deq = oracle.dequant_main(main[j])
        # widest E2M1 gap is 4 -> 6 (error <= 1 scale); the scale is amax/6 rounded
        # to E4M3, so saturation adds at most 0.4 scale: |err| <= s per group
        s_dec = oracle.e4m3_values()[main[j, 256:]]
        assert np.all(np.abs(deq - yr).reshape(32, 16).max(1) <= s_dec)
        assert np.all(s_dec <= np.abs(yr.astype(np.float64)).reshape(32, 16).max(1) / 6 * 17 / 16)
        # MXFP4: amax / 2^X in [4, 8): gap error <= 2^X, saturation (6, 8) <= 2 * 2^X
        kd = oracle.dequant_index(codes[j], scales[j])
        two_x = np.ldexp(1.0, scales[j].astype(int) - 127)
        assert np.all(np.abs(kd - k).reshape(4, 32).max(1) <= 2 * two_x)


# ---------------------------------------------------------------- indexer
def _tiny_cache(seed, n):
    g = synth.rng(seed)
    x = synth.latents(g, n)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    return g, oracle.compress_quantize(x, 1, w0, w1, W)


def test_index_score_brute_force():
    g, (main, codes, scales) = _tiny_cache(8, 24)
    q = synth.index_queries(g)
    w = synth.head_weights(g)
    got = oracle.index_scores(q, w, codes, scales)
    qd = oracle.quantize_index_query(q)
    kd = oracle.dequant_index(codes, scales)
    for j in range(24):
        s = 0.0
        for h in range(32):
            dot = sum(float(qd[h, d]) * float(kd[j, d]) for d in range(128))
            s += float(w[h]) * max(0.0, dot)
        assert abs(got[j] - s) <= 1e-12 * max(1.0, abs(s))


def test_index_score_closed_form_one_head():
    _, (main, codes, scales) = _tiny_cache(9, 4)
    kd = oracle.dequant_index(codes, scales)
    for d in (0, 31, 32, 127):
        q = np.zeros((32, 128), np.float32)
        q[3, d] = 1.0                                          # exact in MXFP4 (code 2, X = -2)
        qb = synth.f32_to_bf16_bits(q)
        w = np.zeros(32, np.float32)
        w[3] = 2.5
        s = oracle.index_scores(qb, w, codes, scales)
        np.testing.assert_array_equal(s, 2.5 * np.maximum(kd[:, d], 0))
        w[3] = -1.0                                            # a negative head weight flips the sign
        s = oracle.index_scores(qb, w, codes, scales)
        np.testing.assert_array_equal(s, -np.maximum(kd[:, d], 0))


def _brute_block_topm(scores, nv, M):
    nb = -(-nv // 8)
    g = []
    for r in range(nb):
        vals = [scores[j] for j in range(8 * r, min(8 * r + 8, nv))]
        g.append(max(vals))
    g[(nv - 1) // 8] = math.inf
    ranked = sorted(range(nb), key=lambda r: (-g[r], r))
    chosen = sorted(ranked[:M])
    return chosen + [-1] * (M - len(chosen))


def test_block_topm_brute_force_forced_block_and_padding():
    g = np.random.default_rng(10)
    for nv, M in [(1, 4), (7, 1), (8, 2), (9, 1), (61, 3), (64, 8), (100, 20), (173, 5)]:
        scores = g.standard_normal(nv + 5)
        scores[3] = scores[11] if nv > 11 else scores[3]       # a tie
        got = oracle.block_topm(scores, nv, M)
        assert list(got) == _brute_block_topm(scores, nv, M)
        assert (nv - 1) // 8 in got                             # newest block always kept


def test_block_topm_last_block_padded_with_minus_inf():
    # last (partial) block holds only -5 among visible entries; padding must not lift it
    s = np.array([1, 1, 1, 1, 1, 1, 1, 1, -5, 9, 9], float)
    got = oracle.block_topm(s, 9, 2)
    assert list(got) == [0, 1]
    got = oracle.block_topm(np.array([3.0] * 16 + [-1.0] * 3), 19, 1)
    assert list(got) == [2]                                     # forced newest block wins


def test_select_topk_brute_force_ties_to_lower_index():
    g = np.random.default_rng(12)
    s = np.round(g.standard_normal(50), 1)                      # many ties
    for K in (1, 5, 17, 50, 64):
        got = oracle.select_topk(s, np.arange(50), K)
        ranked = sorted(range(50), key=lambda j: (-s[j], j))[:K]
        assert list(got[got >= 0]) == sorted(ranked)
        assert np.all(got[min(K, 50):] == -1)
    dom = np.array([3, 9, 10, 40])
    got = oracle.select_topk(s, dom, 2)
    assert set(got) <= set(dom)


def test_hsi_equals_exhaustive_when_pool_covers_all_blocks():
    g, (main, codes, scales) = _tiny_cache(13, 200)
    q = synth.index_queries(g)
    w = synth.head_weights(g)
    s = oracle.index_scores(q, w, codes, scales)
    nv = 197
    blocks = oracle.block_topm(s, nv, 25)                       # ceil(197/8) = 25 -> all
    assert np.all(blocks == np.arange(25))
    pool = oracle.pool_entries(blocks, nv)
    np.testing.assert_array_equal(pool, np.arange(nv))
    np.testing.assert_array_equal(oracle.select_topk(s, pool, 16),
                                  oracle.select_topk(s, np.arange(nv), 16))


def test_full_topk_inside_pool_when_M_exceeds_K():
    """Any block holding a top-K entry has block max >= the K-th score, so with
    M >= K+1 blocks (one slot taken by the forced block) the pool holds the whole
    Full top-K."""
    g = np.random.default_rng(14)
    for trial in range(50):
        nv = int(g.integers(40, 400))
        K = int(g.integers(1, 12))
        M = K + 1
        s = np.round(g.standard_normal(nv), 1)
        pool = oracle.pool_entries(oracle.block_topm(s, nv, M), nv)
        top = oracle.select_topk(s, np.arange(nv), K)
        assert set(top[top >= 0]) <= set(pool)


def test_hisa_summary_of_identical_keys_is_the_key():
    """The mean of copies of one key is that key (exactly, in binary32), and an
    MXFP4 key quantises back to its own values: the summary of such a block
    has the entry's values and scales (a negative-zero code comes back as +0,
    the sum starting from +0), for a partial block of 3 copies as well."""
    g, (main, codes, scales) = _tiny_cache(21, 40)
    rep_c = np.repeat(codes[[5, 17, 30]], 8, axis=0)[:19]      # blocks of 8, 8 and 3 copies
    rep_s = np.repeat(scales[[5, 17, 30]], 8, axis=0)[:19]
    sc, ss = oracle.block_summary(rep_c, rep_s, 19)
    np.testing.assert_array_equal(ss, scales[[5, 17, 30]])
    np.testing.assert_array_equal(oracle.dequant_index(sc, ss), oracle.dequant_index(codes[[5, 17, 30]],
                                                                                     scales[[5, 17, 30]]))


def test_hisa_summary_is_the_mean_within_mxfp4_rounding():
    """Dequantised summary = the block's mean key up to MXFP4 rounding: per
    32-wide group with scale 2^X, X = floor(log2 amax) - 2, the E2M1 grid's
    largest spacing is 2 * 2^X and values in [6, 8) * 2^X saturate to 6, so the
    error is at most 2 * 2^X; opposite keys give a zero block (zero codes, zero
    scale byte)."""
    g, (main, codes, scales) = _tiny_cache(22, 61)
    sc, ss = oracle.block_summary(codes, scales, 61)
    assert sc.shape == (8, 64)
    kd = oracle.dequant_index(codes, scales)
    got = oracle.dequant_index(sc, ss)
    for r in range(8):
        rows = kd[8 * r:min(8 * r + 8, 61)]
        mean = rows.sum(axis=0) / len(rows)
        for grp in range(4):
            m = mean[32 * grp:32 * grp + 32]
            amax = np.abs(m).max()
            bound = 2.0 ** (math.floor(math.log2(amax)) - 1) if amax > 0 else 0.0
            assert np.all(np.abs(got[r, 32 * grp:32 * grp + 32] - m) <= bound)
    neg_c, neg_s = oracle.mxfp4_quantize(-kd[3].astype(np.float32))
    pc = np.stack([codes[3], neg_c])
    ps = np.stack([scales[3], neg_s])
    zc, zs = oracle.block_summary(pc, ps, 2)
    assert not zc.any() and not zs.any()


def test_hisa_with_every_block_equals_exhaustive_topk():
    """With M at least the number of visible blocks HISA keeps every block, and
    its second stage (top-K over the pool) is the exhaustive top-K."""
    g, (main, codes, scales) = _tiny_cache(23, 203)
    q = synth.index_queries(g)
    w = synth.head_weights(g)
    sc, ss = oracle.block_summary(codes, scales, 203)
    nv = 199
    blocks = oracle.hisa_blocks(q, w, sc, ss, nv, 30)
    np.testing.assert_array_equal(blocks[:25], np.arange(25))
    assert np.all(blocks[25:] == -1)
    s = oracle.index_scores(q, w, codes, scales)
    pool = oracle.pool_entries(blocks, nv)
    np.testing.assert_array_equal(oracle.select_topk(s, pool, 16), oracle.select_topk(s, np.arange(nv), 16))


def test_hisa_summary_of_a_block_depends_only_on_its_entries():
    """Appending entries changes only the newest block's summary (so a decode
    step recomputes one block), and a block's summary is unchanged when the
    entries of other blocks change."""
    g, (main, codes, scales) = _tiny_cache(25, 70)
    sc_a, ss_a = oracle.block_summary(codes, scales, 66)      # blocks 0..8, block 8 holds 2 entries
    sc_b, ss_b = oracle.block_summary(codes, scales, 70)      # block 8 now holds 6
    np.testing.assert_array_equal(sc_a[:8], sc_b[:8])
    np.testing.assert_array_equal(ss_a[:8], ss_b[:8])
    assert not (np.array_equal(sc_a[8], sc_b[8]) and np.array_equal(ss_a[8], ss_b[8]))
    c2 = codes.copy()
    c2[8:16] = codes[40:48]                                    # block 1 replaced by block 5's entries
    s2 = scales.copy()
    s2[8:16] = scales[40:48]
    sc_c, ss_c = oracle.block_summary(c2, s2, 70)
    np.testing.assert_array_equal(sc_c[[0, 2, 3, 4, 5, 6, 7, 8]], sc_b[[0, 2, 3, 4, 5, 6, 7, 8]])
    np.testing.assert_array_equal(oracle.dequant_index(sc_c[1:2], ss_c[1:2]),
                                  oracle.dequant_index(sc_b[5:6], ss_b[5:6]))


def test_hisa_blocks_rank_by_the_mean_key_score():
    """Brute force on a small cache: the chosen blocks are the M highest scores
    of the block mean keys (ties to the lower block), none forced."""
    g, (main, codes, scales) = _tiny_cache(24, 120)
    q = synth.index_queries(g)
    w = synth.head_weights(g)
    sc, ss = oracle.block_summary(codes, scales, 120)
    qd = oracle.quantize_index_query(q)
    kd = oracle.dequant_index(sc, ss)
    score = [sum(float(w[h]) * max(0.0, float(qd[h] @ kd[r])) for h in range(32)) for r in range(15)]
    want = sorted(sorted(range(15), key=lambda r: (-score[r], r))[:4])
    got = oracle.hisa_blocks(q, w, sc, ss, 120, 4)
    assert list(got) == want


# ---------------------------------------------------------------- attention
def _attn_inputs(seed, n_entries=40, S=160):
    g, (main, codes, scales) = _tiny_cache(seed, n_entries)
    q = synth.main_queries(g)
    swa = synth.swa_rows(g, S)
    return g, main, q, swa


def test_attention_brute_force():
    g, main, q, swa = _attn_inputs(15, 12, 20)
    sel = np.array([3, -1, 0, 11, 7], np.int32)
    t, base = 9, 0
    qq = q.copy()
    out = oracle.attention(qq, sel, main, swa, base, t, 1 / math.sqrt(512))
    V = [oracle.dequant_main(main[j]) for j in (3, 0, 11, 7)]
    V += [oracle.bf16_to_f64(swa[p]) for p in range(0, 10)]
    qd = oracle.bf16_to_f64(qq)
    for h in (0, 31, 63):
        logits = [sum(qd[h, d] * v[d] for d in range(512)) / math.sqrt(512) for v in V]
        mx = max(logits)
        e = [math.exp(x - mx) for x in logits]
        tot = sum(e)
        want = [sum(e[i] * V[i][d] for i in range(len(V))) / tot for d in range(512)]
        np.testing.assert_allclose(out[h], want, rtol=1e-10, atol=1e-12)


def test_attention_window_bounds_and_convex_hull():
    g, main, q, swa = _attn_inputs(16, 30, 400)
    sel = np.arange(0, 30, 3).astype(np.int32)
    t, base = 300, 100
    out = oracle.attention(q, sel, main, swa, base, t, 1 / math.sqrt(512))
    V = np.concatenate([oracle.dequant_main(main[sel]),
                        oracle.bf16_to_f64(swa[np.arange(t - 127, t + 1) - base])])
    assert len(oracle.window_positions(t)) == 128
    assert np.all(out >= V.min(0) - 1e-12) and np.all(out <= V.max(0) + 1e-12)
    # window of an early query is clipped at position 0
    assert list(oracle.window_positions(5)) == list(range(6))


def test_attention_single_and_identical_keys():
    g, main, q, swa = _attn_inputs(17, 8, 4)
    # only the window's one row (t = 0) and no selection: output = that row
    out = oracle.attention(q, np.full(4, -1, np.int32), main, swa, 0, 0, 0.05)
    np.testing.assert_allclose(out, np.broadcast_to(oracle.bf16_to_f64(swa[0]), out.shape), rtol=1e-12)
    # the same entry selected many times and a window row equal to it: output = that vector
    v = oracle.dequant_main(main[2])
    swa2 = swa.copy()
    swa2[0] = synth.f32_to_bf16_bits(v.astype(np.float32))     # FP4 values are exact in bf16
    out = oracle.attention(q, np.full(5, 2, np.int32), main, swa2, 0, 0, 0.05)
    np.testing.assert_allclose(out, np.broadcast_to(v, out.shape), rtol=1e-12)


# ---------------------------------------------------------------- FP8 window
def test_swa_fp8_keeps_every_e4m3_value():
    """Every finite E4M3 value is a bf16 value; quantising it returns its own
    code (both zeros included)."""
    vals = oracle.e4m3_values()
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    bits = synth.f32_to_bf16_bits(vals[codes].astype(np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(bits).astype(np.float64), vals[codes])
    np.testing.assert_array_equal(oracle.swa_fp8_quantize(bits), codes)


def test_swa_fp8_rounds_to_nearest_and_saturates():
    """Brute force over bf16 values spanning the E4M3 range: the chosen code is
    a nearest finite value (ties to the even code), signs kept, |x| >= 448 ->
    448; the row shape is kept."""
    g = np.random.default_rng(31)
    x = np.concatenate([g.standard_normal(3000) * 4.0, g.uniform(-600, 600, 500),
                        2.0 ** g.uniform(-12, -6, 500) * g.choice([-1, 1], 500)]).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)[:4000].reshape(8, 500)
    got = oracle.swa_fp8_quantize(bits)
    assert got.shape == (8, 500)
    vals = oracle.e4m3_values()
    finite = np.array([c for c in range(128) if c != 0x7F])
    for b, c in zip(bits.ravel(), got.ravel()):
        v = float(synth.bf16_bits_to_f32(np.array([b], np.uint16))[0])
        a = abs(v)
        if a >= 448:
            assert vals[c] == math.copysign(448.0, v)
            continue
        d = np.abs(vals[finite] - a)
        best = finite[d == d.min()]
        want = best[0] if len(best) == 1 else [k for k in best if k % 2 == 0][0]
        assert (c & 0x7F) == want and (vals[c] == 0 or math.copysign(1, vals[c]) == math.copysign(1, v))


def test_attention_fp8_window_is_attention_over_its_values():
    """FP8 rows enter the softmax as their E4M3 values: the same attention as
    bf16 rows holding those values (E4M3 is a subset of bf16), and not the
    attention over the unrounded rows."""
    g, main, q, swa = _attn_inputs(18, 30, 300)
    sel = np.arange(1, 30, 4).astype(np.int32)
    t, base = 250, 50
    fp8 = oracle.swa_fp8_quantize(swa)
    as_bf16 = synth.f32_to_bf16_bits(oracle.e4m3_values()[fp8].astype(np.float32))
    a = oracle.attention(q, sel, main, fp8, base, t, 1 / math.sqrt(512))
    b = oracle.attention(q, sel, main, as_bf16, base, t, 1 / math.sqrt(512))
    c = oracle.attention(q, sel, main, swa, base, t, 1 / math.sqrt(512))
    np.testing.assert_array_equal(a, b)
    assert np.abs(a - c).max() > 1e-6


# ---------------------------------------------------------------- modes
def test_modes_reuse_equals_full_attention_and_reindex_all_blocks():
    g = synth.rng(18)
    n = 120
    x = synth.latents(g, n)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    main, codes, scales = oracle.compress_quantize(x, 1, w0, w1, W)
    q = synth.main_queries(g)
    q_idx = synth.index_queries(g)
    wh = synth.head_weights(g)
    swa = synth.swa_rows(g, 200)
    common = dict(t=n - 1, m=1, n_entries=n, main_kv=main, idx_codes=codes, idx_scales=scales,
                  q=q, swa=swa, swa_base=0, scale=1 / math.sqrt(512), K=9)
    pool, sel, out_full = oracle.decode_query(oracle.FULL, M=15, q_idx=q_idx, w_head=wh, **common)
    _, _, out_reuse = oracle.decode_query(oracle.REUSE, M=15, sel=sel, **common)
    np.testing.assert_array_equal(out_full, out_reuse)
    _, sel_x, _ = oracle.decode_query(oracle.REINDEX, M=15, q_idx=q_idx, w_head=wh,
                                      pool_blocks=np.arange(15, dtype=np.int32), **common)
    np.testing.assert_array_equal(sel_x, sel)                   # pool = all blocks -> same as Full
    assert len(oracle.pool_entries(pool, n)) <= 15 * 8


def _reindex_brute_force(scores_all, pool_blocks, nv, K):
    """Reindex selection written out from the page's statement (a Reindex layer
    scores only the candidate pool and takes its own top-K there; zartbot
    §2.3.4): walk the pool's blocks, keep their entries that the query sees,
    rank them by (score desc, id asc), keep K, list them ascending, pad -1."""
    cand = []
    for blk in pool_blocks:
        if blk < 0:
            continue
        for r in range(8):
            j = 8 * int(blk) + r
            if j < nv:
                cand.append(j)
    ranked = sorted(cand, key=lambda j: (-scores_all[j], j))[:K]
    return sorted(ranked) + [-1] * (K - len(ranked))


@pytest.mark.parametrize("K,pool", [(16, [4, 1, -1]), (5, [4, 1, -1]), (6, [2, -1, 0, -1])])
def test_reindex_partial_pool_brute_force(K, pool):
    """Reindex with a pool that covers only some blocks: the newest chosen block
    (entries 32..39) is seen only up to entry 36, and with K = 16 the pool holds
    fewer visible entries (13) than K.  Entries outside the pool or past the
    visible width must never be chosen, and the output is the attention over
    exactly that selection."""
    g = synth.rng(19)
    n, t = 40, 36                                # 40 entries cached, 37 visible at t = 36 (m = 1)
    x = synth.latents(g, n)
    w0, w1 = synth.compressor_weights(g)
    W = synth.index_projection(g)
    main, codes, scales = oracle.compress_quantize(x, 1, w0, w1, W)
    q = synth.main_queries(g)
    q_idx = synth.index_queries(g)
    wh = synth.head_weights(g)
    swa = synth.swa_rows(g, 64)
    nv = oracle.visible_entries(t, 1, n)
    assert nv == 37
    pool_blocks = np.array(pool, np.int32)
    scores_all = oracle.index_scores(q_idx, wh, codes, scales)        # every entry, no domain argument
    want_sel = _reindex_brute_force(scores_all, pool, nv, K)
    common = dict(t=t, m=1, n_entries=n, main_kv=main, idx_codes=codes, idx_scales=scales, q=q, swa=swa,
                  swa_base=0, scale=1 / math.sqrt(512), K=K, M=len(pool))
    got_pool, sel, out = oracle.decode_query(oracle.REINDEX, q_idx=q_idx, w_head=wh, pool_blocks=pool_blocks,
                                             **common)
    assert list(sel) == want_sel
    np.testing.assert_array_equal(got_pool, pool_blocks)             # the pool is an input, passed through
    if K == 16:
        assert want_sel[13:] == [-1, -1, -1] and max(want_sel) <= 36
    # the best entries overall lie outside the pool: ignoring the pool would change the selection
    top_all = sorted(range(nv), key=lambda j: (-scores_all[j], j))[:K]
    assert set(top_all) != set(j for j in want_sel if j >= 0)
    np.testing.assert_array_equal(out, oracle.attention(q, np.array(want_sel, np.int32), main, swa, 0, t,
                                                        1 / math.sqrt(512)))


def test_visibility_rule():
    assert oracle.visible_entries(4095, 2, 2048) == 2048
    assert oracle.visible_entries(4092, 2, 2048) == 2046
    assert oracle.visible_entries(4093, 2, 2048) == 2047
    assert oracle.visible_entries(0, 2, 2048) == 0
    assert oracle.visible_entries(10, 1, 5) == 5

"""Pins of the FP8 attention reference (oracle/fp8.py) against things other than
itself: the e4m3 bit layout enumerated exhaustively, torch's own e4m3 cast, the
orthogonality of the rotation, the exactness of attention under the rotation
without rounding, the e4m3 relative-error bound, hand-derived values of the
block and per-tensor quantisers and of the P quantisation, and an error study
(block quantisation with incoherent processing against per-tensor FP8, the
comparison the pages make) on inputs with outlier feature columns, where the
pages' 2.6x gain is reproduced."""
import numpy as np
import pytest
import torch

from oracle import fp8
from oracle import reference as ref


def test_e4m3_round_matches_exhaustive_nearest_with_ties_to_even():
    vals = fp8.e4m3_values()
    assert len(vals) == 127 and vals[-1] == 448.0 and vals[1] == 2.0 ** -9
    # every representable value is fixed
    np.testing.assert_array_equal(fp8.e4m3_round(vals), vals)
    np.testing.assert_array_equal(fp8.e4m3_round(-vals), -vals)
    # midpoints go to the neighbour whose mantissa is even (its index in the table is even
    # within a binade: the bit pattern's last mantissa bit is 0)
    mids = (vals[:-1] + vals[1:]) / 2
    got = fp8.e4m3_round(mids)
    for i, m in enumerate(mids):
        lo, hi = vals[i], vals[i + 1]
        lo_bits = i % 8 if lo >= fp8.E4M3_MIN_NORMAL else i
        # the mantissa of lo is even when its position in the binade is even
        expect = lo if (lo_bits % 2 == 0) else hi
        assert got[i] == expect, (m, got[i], lo, hi)
    # random values: brute-force nearest
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-9, 6, 20000))
    x = x[np.abs(x) <= 448]
    d = np.abs(np.abs(x)[:, None] - vals[None, :])
    nearest = vals[np.argmin(d, axis=1)]
    ties = np.sum(d == d.min(axis=1, keepdims=True), axis=1) > 1
    np.testing.assert_array_equal(np.abs(fp8.e4m3_round(x))[~ties], nearest[~ties])


def test_e4m3_round_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50000) * np.exp(rng.uniform(-10, 6, 50000))
    x = x[np.abs(x) < 448]
    t = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x.astype(np.float32).astype(np.float64)), t)


def test_e4m3_relative_error_bound_in_the_normal_range():
    rng = np.random.default_rng(2)
    x = rng.uniform(2.0 ** -6, 448, 100000)
    rel = np.abs(fp8.e4m3_round(x) - x) / x
    assert rel.max() <= 2.0 ** -4 + 1e-15  # half an ulp of a 3-bit mantissa


@pytest.mark.parametrize("n", [1, 2, 64, 128, 256])
def test_rotation_is_orthogonal(n):
    m = fp8.hadamard_rotation(n, seed=n)
    np.testing.assert_allclose(m @ m.T, np.eye(n), rtol=0, atol=1e-14)
    assert np.allclose(np.abs(m), 1 / np.sqrt(n))


@pytest.mark.parametrize("causal", [False, True])
def test_rotation_without_rounding_is_exact_attention(causal):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 40, 64))
    k = rng.standard_normal((1, 2, 40, 64))
    v = rng.standard_normal((1, 2, 40, 64))
    o, lse = fp8.fp8_attention(q, k, v, causal, 0.125, mode="block_incoherent", quantize=False)
    o_ref, lse_ref = ref.attn_fwd(q, k, v, causal, 0.125)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def _outlier_inputs(seed, B=1, H=2, N=512, d=128):
    # N(0,1) entries plus a few large ones (about 0.1%, scale 10) in Q, K and V
    rng = np.random.default_rng(seed)

    def t(shape):
        x = rng.standard_normal(shape)
        mask = rng.random(shape) < 1e-3
        return x + mask * rng.standard_normal(shape) * 10.0
    return t((B, H, N, d)), t((B, H, N, d)), t((B, H, N, d))


def test_fp8_error_study_on_outlier_inputs():
    """Scattered element outliers (0.1% of entries, scale 10) are not the case incoherent
    processing targets: e4m3 keeps about 2^-4 relative error over 17 binades, so outliers of
    this size never push typical values out of its normal range, and the P and V roundings,
    equal in every mode, set the error floor; the gain is small here.  The test pins what
    holds: every mode stays within the e4m3 error scale and the block modes are not worse
    than per-tensor.  (Outlier feature columns, below, reproduce the pages' gain.)"""
    for seed in range(3):
        q, k, v = _outlier_inputs(seed)
        scale = 128 ** -0.5
        o_ref, lse_ref = ref.attn_fwd(q, k, v, True, scale)
        rmse = {}
        for mode in ("tensor", "block", "block_incoherent"):
            o, lse = fp8.fp8_attention(q, k, v, True, scale, mode=mode, seed=seed)
            rmse[mode] = float(np.sqrt(np.mean((o - o_ref) ** 2)))
            assert np.mean(np.abs(lse - lse_ref)) < 0.05  # scores carry e4m3 rounding
        assert max(rmse.values()) < 0.05, rmse
        assert rmse["block"] <= rmse["tensor"] * 1.1, rmse
        assert rmse["block_incoherent"] <= rmse["tensor"] * 1.1, rmse


# ---------------------------------------------------------------- hand-derived quantiser values
# e4m3 keeps 3 mantissa bits in every binade of its normal range [2^-6, 448], so a common
# power-of-ten rescaling changes nothing there; block and per-tensor scales differ only where
# one of them pushes a block into the subnormal range (quantum 2^-9).  Each expected value is
# derived in the comment beside it.

def test_quantize_blocks_two_blocks_with_different_scales():
    x = np.array([[4.0], [1.0], [1e-4], [2e-4]])[None, None]        # [1, 1, N=4, d=1], block = 2
    got = fp8.quantize_blocks(x, block=2)[0, 0, :, 0]
    # block 0: amax 4, s = 4/448 = 1/112: 4 -> 448 and 1 -> 112 = 1.75 * 2^6 are exact
    # block 1: amax 2e-4, s = 2e-4/448: 2e-4 -> 448 and 1e-4 -> 224 = 1.75 * 2^7 are exact
    np.testing.assert_allclose(got, [4.0, 1.0, 1e-4, 2e-4], rtol=1e-15, atol=0)


def test_quantize_tensor_uses_one_scale_for_the_whole_tensor():
    x = np.array([[4.0], [1.0], [1e-4], [2e-4]])[None, None]
    got = fp8.quantize_tensor(x)[0, 0, :, 0]
    # one scale s = 4/448 = 1/112 for all four values:
    #   1e-4 * 112 = 0.0112 < 2^-6 is subnormal: 0.0112 * 2^9 = 5.73 -> 6, value 6 * 2^-9 / 112
    #   2e-4 * 112 = 0.0224 in [2^-6, 2^-5), spacing 2^-9: 0.0224 * 2^9 = 11.47 -> 11
    expect = [4.0, 1.0, 6 * 2.0 ** -9 / 112, 11 * 2.0 ** -9 / 112]
    np.testing.assert_allclose(got, expect, rtol=1e-15, atol=0)


def test_quantize_blocks_never_spans_two_heads():
    # two heads of two rows each, block = 128: each head is one block of its own, so the small
    # head keeps its own scale (exact values) instead of the large head's (subnormal values)
    x = np.array([[[4.0], [1.0]], [[1e-4], [2e-4]]])[None]           # [1, H=2, N=2, d=1]
    got = fp8.quantize_blocks(x, block=128)[0, :, :, 0]
    np.testing.assert_allclose(got, [[4.0, 1.0], [1e-4, 2e-4]], rtol=1e-15, atol=0)


def test_quantize_blocks_rounds_inside_a_binade_with_ties_to_even():
    x = np.array([[1.0], [3.0], [4.0], [0.01]])[None, None]          # one block, s = 1/112
    got = fp8.quantize_blocks(x, block=128)[0, 0, :, 0]
    # 3 -> 336 in [256, 512), spacing 32: 336 / 32 = 10.5 -> 10 (even) -> 320 / 112
    # 0.01 -> 1.12 in [1, 2), spacing 1/8: 8.96 -> 9 -> 1.125 / 112
    np.testing.assert_allclose(got, [1.0, 320 / 112, 4.0, 1.125 / 112], rtol=1e-15, atol=0)


def test_p_quantisation_and_normalisation_closed_form():
    # one query, three keys (scale 1, no rotation): scores q.k = (0, 0, 1), all inputs exact
    # in e4m3 under their block scales (Q, K: amax 1; V: amax 4, v/s = 112, 224, 448)
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[0.0, 1.0], [0.0, 1.0], [1.0, 0.0]]]])
    v = np.array([[[[1.0, 0.0], [2.0, 0.0], [4.0, 0.0]]]])
    o, lse = fp8.fp8_attention(q, k, v, False, 1.0, mode="block")
    # P = (1, 1, e) / (2 + e); 448 P = (94.95, 94.95, 258.1):
    #   94.95 in [64, 128), spacing 8: 11.87 -> 12 -> 96;  258.1 in [256, 512), spacing 32: 8.07 -> 8 -> 256
    # O = (96 * 1 + 96 * 2 + 256 * 4) / (96 + 96 + 256): normalised by the quantised weights
    assert o[0, 0, 0, 0] == pytest.approx(1312 / 448, rel=1e-15)
    assert o[0, 0, 0, 1] == 0.0
    # (here the quantised weights happen to sum to 448, so the next test checks the normaliser)
    assert lse[0, 0, 0] == pytest.approx(np.log(2 + np.e), rel=1e-15)   # LSE of the unquantised softmax


def test_p_quantisation_normalises_by_the_quantised_sum():
    # scores (0, 0, ln 3) are not exact, so build them from scale: q.k = (0, 0, 1), scale = ln 3
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[0.0, 1.0], [0.0, 1.0], [1.0, 0.0]]]])
    v = np.array([[[[1.0, 0.0], [2.0, 0.0], [4.0, 0.0]]]])
    o, lse = fp8.fp8_attention(q, k, v, False, float(np.log(3.0)), mode="block")
    # P = (1, 1, 3) / 5 = (0.2, 0.2, 0.6); 448 P = (89.6, 89.6, 268.8):
    #   89.6 in [64, 128), spacing 8: 11.2 -> 11 -> 88;  268.8 in [256, 512), spacing 32: 8.4 -> 8 -> 256
    # sum of the quantised weights 88 + 88 + 256 = 432 (not 448):
    #   O = (88 + 176 + 1024) / 432;  dividing by the unquantised sum would give 1288 / 448
    assert o[0, 0, 0, 0] == pytest.approx(1288 / 432, rel=1e-15)
    assert lse[0, 0, 0] == pytest.approx(np.log(5.0), rel=1e-14)


def _channel_outlier_inputs(seed, mag, N=512, d=128, H=2, ncols=4):
    # N(0,1) entries; a few head-dim columns of Q and K scaled by `mag` (the outlier features
    # that incoherent processing spreads over all dimensions)
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((1, H, N, d)) for _ in range(3))
    cols = rng.choice(d, ncols, replace=False)
    q[..., cols] *= mag
    k[..., cols] *= mag
    return q, k, v


@pytest.mark.parametrize("mag", [10.0, 50.0, 100.0])
def test_fp8_incoherent_processing_gain_on_outlier_channels(mag):
    """The wiki's FA3 item 3 reports 2.6x lower error for block quantisation with incoherent
    processing than for baseline (per-tensor) FP8.  With outlier feature columns (4 of 128
    head-dim columns of Q and K scaled by 10-100) the rotation spreads each outlier over all
    columns before rounding; the O error drops by 2.1-4.5x here (two seeds per magnitude), so
    the claim holds in this regime: the pin is a gain of at least 2x on both seeds, and at
    least 1.5x on the LSE error."""
    for seed in range(2):
        q, k, v = _channel_outlier_inputs(seed, mag)
        scale = 128 ** -0.5
        o_ref, lse_ref = ref.attn_fwd(q, k, v, True, scale)
        err = {}
        for mode in ("tensor", "block_incoherent"):
            o, lse = fp8.fp8_attention(q, k, v, True, scale, mode=mode, seed=seed)
            err[mode] = (float(np.sqrt(np.mean((o - o_ref) ** 2))), float(np.mean(np.abs(lse - lse_ref))))
        assert err["tensor"][0] >= 2.0 * err["block_incoherent"][0], err
        assert err["tensor"][1] >= 1.5 * err["block_incoherent"][1], err


# ---------------------------------------------------------------- the FP8 kernel's steps

def test_fwht_fp32_equals_the_sylvester_matrix_exactly_on_integers():
    # integer inputs keep every fp32 sum exact, so the butterfly must equal x @ H bit for bit
    rng = np.random.default_rng(4)
    x = rng.integers(-8, 9, size=(5, 128)).astype(np.float64)
    h = np.array([[1.0]])
    while h.shape[0] < 128:
        h = np.block([[h, h], [h, -h]])
    np.testing.assert_array_equal(fp8.fwht_fp32(x).astype(np.float64), x @ h)


def test_rotate_fp32_is_the_hadamard_rotation_to_fp32_precision():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 128))
    m = fp8.hadamard_rotation(128, seed=9)
    signs = np.sign(m[0])  # the first row of H is all ones, so row 0 of M is r / sqrt(d)
    got = fp8.rotate_fp32(x.astype(np.float32), signs).astype(np.float64)
    np.testing.assert_allclose(got, x.astype(np.float32).astype(np.float64) @ m, rtol=0, atol=2e-6)


def test_e4m3_bytes_match_torch_bit_patterns():
    vals = fp8.e4m3_values()
    allv = np.concatenate([vals, -vals[1:]])
    t = torch.from_numpy(allv.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.e4m3_bytes(allv), t)


def test_quantize_fp32_hand_values():
    # one block, amax 4: inv = 448 / 4 = 112 and scale = 4 / 448 exactly in fp32;
    # 3 * 112 = 336 -> tie between 320 and 352 (spacing 32 in [256, 512)) -> 320 (even)
    x = np.array([[4.0], [3.0], [1.0], [0.01]], dtype=np.float32)[None, None]
    codes, sc = fp8.quantize_fp32(x)
    np.testing.assert_array_equal(codes[0, 0, :, 0], [448.0, 320.0, 112.0, fp8.e4m3_round(np.float32(0.01) * np.float32(112))])
    assert sc[0, 0, 0] == np.float32(4.0) / np.float32(448.0)


def test_quantize_fp32_agrees_with_the_fp64_quantiser():
    # same method, the code decided in fp32 instead of fp64: equal except where the scaled value
    # lies within fp32 rounding of an e4m3 rounding boundary
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((2, 3, 300, 64)) * np.exp(rng.uniform(-3, 3, (2, 3, 300, 1)))).astype(np.float32)
    codes, sc = fp8.quantize_fp32(x)
    x64 = x.astype(np.float64)
    codes64 = np.empty_like(x64)
    for ib in range(3):
        blk = x64[..., 128 * ib:128 * (ib + 1), :]
        s64 = np.max(np.abs(blk), axis=(-2, -1), keepdims=True) / 448.0
        codes64[..., 128 * ib:128 * (ib + 1), :] = fp8.e4m3_round(blk / s64)
        np.testing.assert_allclose(sc[..., ib], s64[..., 0, 0], rtol=2 ** -23, atol=0)
    differ = np.mean(codes != codes64)
    assert differ < 1e-3, differ
    np.testing.assert_allclose(codes, codes64, rtol=2 ** -3, atol=0)


def _quantised_inputs(seed, B=1, H=2, Hkv=1, N=300, d=64):
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((B, H, N, d)), rng.standard_normal((B, Hkv, N, d)), rng.standard_normal((B, Hkv, N, d))
    v[..., 200:, :] *= 5.0  # a different V scale in the last blocks
    (q8, sq), (k8, sk), (v8, sv) = (fp8.quantize_fp32(t) for t in (q, k, v))
    return q8, sq, k8, sk, v8, sv


@pytest.mark.parametrize("causal", [False, True])
def test_tiled_fp8_attention_without_p_rounding_is_exact_attention(causal):
    q8, sq, k8, sk, v8, sv = _quantised_inputs(7)
    o, lse = fp8.fp8_attention_tiled(q8, k8, v8, sq, sk, sv, causal, 0.125, quantize_p=False)
    deq = lambda c, s: c * np.repeat(s.astype(np.float64), 128, axis=-1)[..., :c.shape[-2], None]
    o_ref, lse_ref = ref.attn_fwd(deq(q8, sq), deq(k8, sk), deq(v8, sv), causal, 0.125)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_tiled_fp8_attention_constant_v_is_returned_exactly():
    q8, sq, k8, sk, _, _ = _quantised_inputs(8)
    v8 = np.full(k8.shape, 112.0)
    sv = np.full(sk.shape, 1.0 / 112, dtype=np.float32)
    o, _ = fp8.fp8_attention_tiled(q8, k8, v8, sq, sk, sv, True, 0.125)
    np.testing.assert_allclose(o, 112.0 * np.float64(np.float32(1.0 / 112)), rtol=1e-14, atol=0)


def test_tiled_fp8_attention_hand_case():
    # one query, three keys in one tile, scores (0, 0, ln 3) from unit codes and scale ln 3;
    # weights exp(s - max) = (1/3, 1/3, 1); 448 * (1/3) = 149.3 in [128, 256), spacing 16:
    # 9.33 -> 9 -> 144; 448 stays.  O = (144 * 1 + 144 * 2 + 448 * 4) / (144 + 144 + 448)
    q8 = np.array([[[[1.0, 0.0]]]])
    k8 = np.array([[[[0.0, 1.0], [0.0, 1.0], [1.0, 0.0]]]])
    v8 = np.array([[[[1.0, 0.0], [2.0, 0.0], [4.0, 0.0]]]])
    one = np.ones((1, 1, 1), dtype=np.float32)
    o, lse = fp8.fp8_attention_tiled(q8, k8, v8, one, one, one, False, float(np.log(3.0)))
    assert o[0, 0, 0, 0] == pytest.approx(2224.0 / 736.0, rel=1e-14)
    assert lse[0, 0, 0] == pytest.approx(np.log(5.0), rel=1e-14)

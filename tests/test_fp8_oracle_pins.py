"""Pins of the FP8 attention reference (oracle/fp8.py) against things other than
itself: the e4m3 bit layout enumerated exhaustively, torch's own e4m3 cast, the
orthogonality of the rotation, the exactness of attention under the rotation
without rounding, the e4m3 relative-error bound, and an error study on inputs
with outlier features (block quantisation with incoherent processing against
per-tensor FP8, the comparison the pages make; the pages' 2.6x gain is not
reproduced under these readings, see the study's docstring)."""
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
    """The pages report 2.6x lower error for block quantisation with incoherent processing
    than for baseline FP8.  Under the readings of oracle/fp8.py (e4m3 with amax scaling per
    128-row block or per tensor, a random-sign Hadamard rotation, P in e4m3) the measured
    gain on this recipe is small: e4m3 keeps about 2^-4 relative error over 17 binades, so
    outliers of this size never push typical values out of its normal range, and the P and
    V roundings, equal in every mode, set the error floor.  The test pins what holds: every
    mode stays within the e4m3 error scale, the block modes are not worse than per-tensor,
    and the rotation does not change which mode is best by more than a few percent."""
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

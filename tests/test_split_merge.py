"""CPU pin of the split-KV merge rule used by the decoding path.

The decoding forward splits the keys of a row into ranges, computes each
range's softmax result (O_s normalised over its keys, LSE_s) and merges them:

    LSE = log sum_s exp(LSE_s),    O = sum_s exp(LSE_s - LSE) O_s

This is the online-softmax update (the explainer's online-softmax paragraph)
applied to whole ranges.  Here the fp64 oracle is run on each key range alone
and the merged result is compared with the oracle on all keys: exact up to
fp64 rounding, including ranges that a causal row does not see at all
(LSE_s = -inf, weight 0)."""
import numpy as np
import pytest

from oracle import reference as ref


def merge(parts):
    lses = np.stack([p[1] for p in parts])            # [S, ...rows]
    m = np.max(lses, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe), 0.0)
    wsum = w.sum(axis=0)
    o = sum(wi[..., None] * p[0] for wi, p in zip(w, parts))
    o = np.where(wsum[..., None] > 0, o / np.where(wsum > 0, wsum, 1.0)[..., None], 0.0)
    lse = np.where(wsum > 0, m_safe + np.log(np.where(wsum > 0, wsum, 1.0)), -np.inf)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bounds", [(0, 7, 19, 40), (0, 1, 40), (0, 13, 26, 39, 40)])
def test_split_ranges_merge_to_the_full_result(causal, bounds):
    rng = np.random.default_rng(3)
    B, H, Hkv, Nq, Nk, d = 1, 4, 2, 5, 40, 8
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    scale = 0.4
    qpos = np.arange(Nq) + (Nk - Nq)      # bottom-right causal alignment
    o_full, lse_full = ref.attn_fwd(q, k, v, causal, scale, qpos=qpos)
    parts = []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        # a range of keys [lo, hi): the oracle on those keys, with query positions shifted so
        # that the mask compares the same absolute key and query positions
        parts.append(ref.attn_fwd(q, k[:, :, lo:hi], v[:, :, lo:hi], causal, scale, qpos=qpos - lo))
    o, lse = merge(parts)
    np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_full, rtol=0, atol=1e-13)


def test_merge_with_rows_that_see_no_key_in_some_ranges():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 2, 6, 4))
    k = rng.standard_normal((1, 2, 6, 4))
    v = rng.standard_normal((1, 2, 6, 4))
    qpos = np.arange(6)
    o_full, lse_full = ref.attn_fwd(q, k, v, True, 0.5, qpos=qpos)
    parts = [ref.attn_fwd(q, k[:, :, lo:hi], v[:, :, lo:hi], True, 0.5, qpos=qpos - lo) for lo, hi in ((0, 2), (2, 6))]
    assert np.isneginf(parts[1][1][0, 0, 0])  # row 0 sees no key of the second range
    o, lse = merge(parts)
    np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_full, rtol=0, atol=1e-13)

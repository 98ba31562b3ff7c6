"""Pins of the fp64 CPU oracle against things other than itself.

The oracle is the definition of exact attention ("FlashAttention" wiki note,
section 定義; online-softmax paragraph of the singularity-lens.com explainer:
the tiled result equals standard attention).  The pages print no worked
example, so the oracle is pinned by:

* a pure-Python brute force (with the full softmax Jacobian) on tiny shapes;
* a separate CPU online-softmax implementation at tile sizes 1, 3 and 16;
* central finite differences of L = sum(O * dO) for the backward;
* hand-derived closed forms (tests/golden/closed_form.json);
* invariants: probability rows sum to 1, a single key returns its V row,
  constant V gives constant O, the first causal row attends only to itself,
  key permutation invariance, softmax gradient rows that sum to zero;
* a library routine: torch's CPU float64 scaled_dot_product_attention and
  its autograd.

Each test is chosen so that a plausible mistake (a dropped term, a wrong sign
or index, a transposed operand, a wrong mask direction, a wrong GQA mapping)
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import brute, online
from oracle import reference as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _case(seed, B, H, Hkv, N, d, Nk=None):
    rng = np.random.default_rng(seed)
    Nk = N if Nk is None else Nk
    q = _rand(rng, B, H, N, d)
    k = _rand(rng, B, Hkv, Nk, d)
    v = _rand(rng, B, Hkv, Nk, d)
    do = _rand(rng, B, H, N, d)
    return q, k, v, do


SHAPES = [
    # B, H, Hkv, N, d
    (1, 1, 1, 1, 1),
    (1, 2, 1, 5, 3),
    (2, 2, 2, 7, 4),
    (1, 4, 2, 8, 2),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_forward(shape, causal):
    q, k, v, _ = _case(1, *shape)
    scale = 0.7
    o, lse = ref.attn_fwd(q, k, v, causal, scale)
    ob, lseb = brute.fwd(q.tolist(), k.tolist(), v.tolist(), causal, scale)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(lseb), rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_backward(shape, causal):
    q, k, v, do = _case(2, *shape)
    scale = 0.6
    dq, dk, dv = ref.attn_bwd(q, k, v, do, causal, scale)
    dqb, dkb, dvb = brute.bwd(q.tolist(), k.tolist(), v.tolist(), do.tolist(), causal, scale)
    np.testing.assert_allclose(dq, np.array(dqb), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, np.array(dkb), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, np.array(dvb), rtol=0, atol=1e-11)


@pytest.mark.parametrize("tile", [1, 3, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_matches_materialised(tile, causal):
    q, k, v, _ = _case(3, 2, 4, 2, 37, 8)
    # spread the scores so the running max moves often and by a lot
    q = q * 3.0
    scale = 1.0 / math.sqrt(8)
    o, lse = ref.attn_fwd(q, k, v, causal, scale)
    oo, lseo = online.fwd(q, k, v, causal, scale, tile)
    np.testing.assert_allclose(oo, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lseo, lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 1, 6, 3), (1, 1, 1, 16, 4)])
def test_finite_differences(causal, shape):
    q, k, v, do = _case(4, *shape)
    scale = 0.8
    dq, dk, dv = ref.attn_bwd(q, k, v, do, causal, scale)

    def loss(qq, kk, vv):
        o, _ = ref.attn_fwd(qq, kk, vv, causal, scale)
        return float(np.sum(o * do))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy()
            xp[idx] += h
            xm = x.copy()
            xm[idx] -= h
            plus = {"q": q, "k": k, "v": v}
            minus = dict(plus)
            plus[name] = xp
            minus[name] = xm
            fd[idx] = (loss(plus["q"], plus["k"], plus["v"])
                       - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)


def test_closed_forms():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    env = {"exp": math.exp, "log": math.log}
    for c in cases:
        q = np.array(c["q"])[None, None]
        k = np.array(c["k"])[None, None]
        v = np.array(c["v"])[None, None]
        o, lse = ref.attn_fwd(q, k, v, c["causal"], c["scale"])
        exp_o = np.array([eval(e, env) for e in c["o"]])
        exp_lse = np.array([eval(e, env) for e in c["lse"]])
        np.testing.assert_allclose(o[0, 0, :, 0], exp_o, rtol=1e-14, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], exp_lse, rtol=1e-14, atol=1e-14, err_msg=c["name"])
        if "do" in c:
            do = np.array(c["do"])[None, None]
            dq, dk, dv = ref.attn_bwd(q, k, v, do, c["causal"], c["scale"])
            for key, got in (("dq", dq), ("dk", dk), ("dv", dv)):
                want = np.array([[eval(e, env) for e in row] for row in c[key]])
                np.testing.assert_allclose(got[0, 0], want, rtol=1e-13, atol=1e-14,
                                           err_msg=c["name"] + " " + key)


def test_probability_rows_sum_to_one():
    # V = identity (Nk = d) makes O_i equal to the probability row P_i.
    rng = np.random.default_rng(5)
    N = 9
    q = rng.standard_normal((1, 1, N, N))
    k = rng.standard_normal((1, 1, N, N))
    v = np.eye(N)[None, None]
    for causal in (False, True):
        p, _ = ref.attn_fwd(q, k, v, causal, 0.9)
        p = p[0, 0]
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
        assert (p >= 0).all()
        if causal:
            assert np.all(np.triu(p, 1) == 0.0)
            assert p[0, 0] == 1.0


def test_single_key_returns_its_value():
    q, k, v, _ = _case(6, 2, 3, 1, 4, 5, Nk=1)
    o, lse = ref.attn_fwd(q, k, v, False, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :1], o.shape), atol=1e-15)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("bhnc,bgc->bhn", q, k[:, :, 0]), atol=1e-14)


def test_constant_v_gives_constant_o():
    q, k, v, _ = _case(7, 1, 2, 2, 11, 6)
    v[:] = np.array([1.5, -2.0, 0.25, 3.0, -1.0, 7.0])
    for causal in (False, True):
        o, _ = ref.attn_fwd(q, k, v, causal, 1.1)
        np.testing.assert_allclose(o, np.broadcast_to(v[0, 0, 0], o.shape), atol=1e-13)


def test_first_causal_row_attends_only_to_itself():
    q, k, v, _ = _case(8, 2, 2, 1, 13, 7)
    scale = 0.4
    o, lse = ref.attn_fwd(q, k, v, True, scale)
    for b in range(2):
        for h in range(2):
            np.testing.assert_allclose(o[b, h, 0], v[b, 0, 0], atol=1e-15)
            np.testing.assert_allclose(lse[b, h, 0], scale * q[b, h, 0] @ k[b, 0, 0], atol=1e-14)


def test_key_permutation_invariance_and_query_equivariance():
    q, k, v, do = _case(9, 1, 2, 1, 10, 4)
    rng = np.random.default_rng(10)
    pk = rng.permutation(10)
    pq = rng.permutation(10)
    o, lse = ref.attn_fwd(q, k, v, False, 0.5)
    o2, lse2 = ref.attn_fwd(q[:, :, pq], k[:, :, pk], v[:, :, pk], False, 0.5)
    np.testing.assert_allclose(o2, o[:, :, pq], atol=1e-13)
    np.testing.assert_allclose(lse2, lse[:, :, pq], atol=1e-13)
    dq, dk, dv = ref.attn_bwd(q, k, v, do, False, 0.5)
    dq2, dk2, dv2 = ref.attn_bwd(q[:, :, pq], k[:, :, pk], v[:, :, pk], do[:, :, pq], False, 0.5)
    np.testing.assert_allclose(dq2, dq[:, :, pq], atol=1e-12)
    np.testing.assert_allclose(dk2, dk[:, :, pk], atol=1e-12)
    np.testing.assert_allclose(dv2, dv[:, :, pk], atol=1e-12)


def test_gradient_invariants():
    q, k, v, do = _case(11, 1, 2, 1, 12, 3)
    # constant K rows: every score in a row is equal, so dS rows (which sum to
    # zero) give dQ = sum_j dS_ij k = 0.
    kc = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dq, _, _ = ref.attn_bwd(q, kc, v, do, False, 0.7)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    # constant V and constant dO: dP is constant per row, so dS = 0 and
    # dQ = dK = 0, while dV_j = sum_i P_ij dO.
    vc = np.broadcast_to(v[:, :, :1], v.shape).copy()
    doc = np.broadcast_to(do[:, :, :1], do.shape).copy()
    for causal in (False, True):
        dq, dk, dv = ref.attn_bwd(q, k, vc, doc, causal, 0.7)
        np.testing.assert_allclose(dq, 0.0, atol=1e-13)
        np.testing.assert_allclose(dk, 0.0, atol=1e-13)
        # sum_j dV_j = sum_h sum_i (sum_j P_ij) dO_h = (number of rows) * sum_h dO_h
        np.testing.assert_allclose(dv.sum(axis=2), 12 * doc[:, :, 0].sum(axis=1)[:, None, :], atol=1e-11)


def test_masked_row_guard():
    # rows with no visible key (only possible with a query position before
    # every key): O = 0 and LSE = -inf, never NaN
    q, k, v, _ = _case(12, 1, 1, 1, 3, 2, Nk=4)
    o, lse = ref.attn_fwd(q, k, v, True, 1.0, qpos=np.array([-1, 0, 5]))
    assert np.all(o[0, 0, 0] == 0.0) and lse[0, 0, 0] == -np.inf
    np.testing.assert_allclose(o[0, 0, 1], v[0, 0, 0], atol=1e-15)
    full, lfull = ref.attn_fwd(q, k, v, False, 1.0)
    np.testing.assert_allclose(o[0, 0, 2], full[0, 0, 2], atol=1e-15)


def test_row_subset_matches_full():
    q, k, v, _ = _case(13, 1, 2, 1, 40, 4)
    rows = np.array([0, 7, 8, 39])
    o, lse = ref.attn_fwd(q, k, v, True, 0.5)
    os_, ls_ = ref.attn_fwd(q[:, :, rows], k, v, True, 0.5, qpos=rows)
    np.testing.assert_allclose(os_, o[:, :, rows], atol=0)
    np.testing.assert_allclose(ls_, lse[:, :, rows], atol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_torch_sdpa_float64(causal):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    q, k, v, do = _case(14, 2, 4, 2, 19, 8)
    scale = 0.35
    o, lse = ref.attn_fwd(q, k, v, causal, scale)
    dq, dk, dv = ref.attn_bwd(q, k, v, do, causal, scale)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    # grouped heads: query head h uses K/V head h // (H/Hkv)
    kr = tk.repeat_interleave(2, dim=1)
    vr = tv.repeat_interleave(2, dim=1)
    to = F.scaled_dot_product_attention(tq, kr, vr, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(o, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)
    s = scale * torch.einsum("bhnc,bhmc->bhnm", torch.tensor(q), kr.detach())
    if causal:
        s = s.masked_fill(torch.ones(19, 19, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


# ---- Nq != Nk: the causal mask places query row i at position i + qoff, qoff = Nk - Nq
# (bottom-right alignment: the query block follows Nk - Nq earlier keys).

QK_SHAPES = [
    # B, H, Hkv, Nq, d, Nk
    (1, 2, 1, 3, 3, 7),    # fewer queries than keys (a KV cache in front)
    (1, 2, 2, 6, 2, 4),    # more queries than keys: the first two rows see no key
    (2, 4, 2, 1, 4, 9),    # one query (decode)
]


@pytest.mark.parametrize("shape", QK_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_qk(shape, causal):
    B, H, Hkv, Nq, d, Nk = shape
    q, k, v, do = _case(11, B, H, Hkv, Nq, d, Nk)
    qoff = Nk - Nq
    scale = 0.7
    o, lse = ref.attn_fwd(q, k, v, causal, scale, qpos=np.arange(Nq) + qoff)
    ob, lseb = brute.fwd(q.tolist(), k.tolist(), v.tolist(), causal, scale, qoff)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(np.array(lseb)))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], np.array(lseb)[fin], rtol=0, atol=1e-12)
    dq, dk, dv = ref.attn_bwd(q, k, v, do, causal, scale, qoff)
    dqb, dkb, dvb = brute.bwd(q.tolist(), k.tolist(), v.tolist(), do.tolist(), causal, scale, qoff)
    np.testing.assert_allclose(dq, np.array(dqb), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, np.array(dkb), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, np.array(dvb), rtol=0, atol=1e-11)


def test_bottom_right_special_cases():
    # one query at the end of the sequence sees every key: causal equals non-causal
    q, k, v, do = _case(12, 1, 2, 1, 1, 4, 11)
    qoff = 10
    oc, lc = ref.attn_fwd(q, k, v, True, 0.5, qpos=np.arange(1) + qoff)
    on, ln = ref.attn_fwd(q, k, v, False, 0.5)
    np.testing.assert_allclose(oc, on, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lc, ln, rtol=0, atol=1e-14)
    gc = ref.attn_bwd(q, k, v, do, True, 0.5, qoff)
    gn = ref.attn_bwd(q, k, v, do, False, 0.5)
    for a, b in zip(gc, gn):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    # with qoff = 0 the offset backward is the square causal backward
    q, k, v, do = _case(13, 1, 2, 2, 9, 3)
    for a, b in zip(ref.attn_bwd(q, k, v, do, True, 0.4, 0), ref.attn_bwd(q, k, v, do, True, 0.4)):
        np.testing.assert_array_equal(a, b)
    # more queries than keys: rows with i + qoff < 0 see nothing (O = 0, LSE = -inf, dQ = 0)
    # and contribute nothing to dK, dV; the remaining rows equal a square problem on the
    # last Nk queries
    q, k, v, do = _case(14, 1, 2, 1, 7, 3, 4)
    qoff = 4 - 7
    o, lse = ref.attn_fwd(q, k, v, True, 0.6, qpos=np.arange(7) + qoff)
    dq, dk, dv = ref.attn_bwd(q, k, v, do, True, 0.6, qoff)
    assert np.all(o[:, :, :3] == 0) and np.all(np.isneginf(lse[:, :, :3])) and np.all(dq[:, :, :3] == 0)
    o2, lse2 = ref.attn_fwd(q[:, :, 3:], k, v, True, 0.6)
    dq2, dk2, dv2 = ref.attn_bwd(q[:, :, 3:], k, v, do[:, :, 3:], True, 0.6)
    np.testing.assert_allclose(o[:, :, 3:], o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 3:], lse2, rtol=0, atol=1e-14)
    for a, b in ((dq[:, :, 3:], dq2), (dk, dk2), (dv, dv2)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_finite_differences_qk():
    q, k, v, do = _case(15, 1, 2, 1, 4, 3, 9)
    qoff = 5
    scale = 0.8
    dq, dk, dv = ref.attn_bwd(q, k, v, do, True, scale, qoff)
    pos = np.arange(4) + qoff

    def loss(qq, kk, vv):
        o, _ = ref.attn_fwd(qq, kk, vv, True, scale, qpos=pos)
        return float(np.sum(o * do))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy()
            xp[idx] += h
            xm = x.copy()
            xm[idx] -= h
            plus = {"q": q, "k": k, "v": v}
            minus = dict(plus)
            plus[name] = xp
            minus[name] = xm
            fd[idx] = (loss(plus["q"], plus["k"], plus["v"]) - loss(minus["q"], minus["k"], minus["v"])) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)

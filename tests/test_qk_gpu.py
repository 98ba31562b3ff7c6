"""GPU parity with different query and key lengths (fa_fwd_qk, fa_bwd_qk).

With Nq != Nk a causal mask is aligned bottom-right: query row i sits at
position i + (Nk - Nq).  Cases: fewer queries than keys (a query block after a
KV cache), a single query (decode), more queries than keys (the first
Nq - Nk rows see no key: O = 0, LSE = -inf, dQ = 0), ragged lengths, GQA in
both backward modes, and the degenerate Nk = 0 / Nq = 0 problems.  Every
element is compared with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from exact_attention_49_gb300 import binding as fa
from exact_attention_49_gb300.inputs import make_inputs
from oracle import reference as ref
from parity import GRAD_RTOL, LSE_TOL, O_TOL, max_abs, o_error, record, rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_attention_49_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()


@pytest.fixture(autouse=True, params=[0, 1], ids=["1cta", "2cta"])
def pair_mode(request):
    """Every test runs on both forward kernels (one CTA per 256-row block, and CTA pairs over
    512 rows with P in shared memory, used at head dimension 128) and both backward main-stage
    kernels (one CTA per key tile, CTA pairs over 256 keys)."""
    old = (fa.fa_get_option("fwd_2cta"), fa.fa_get_option("bwd_2cta"))
    assert fa.fa_set_option("fwd_2cta", request.param) == fa.FA_OK
    assert fa.fa_set_option("bwd_2cta", request.param) == fa.FA_OK
    yield request.param
    fa.fa_set_option("fwd_2cta", old[0])
    fa.fa_set_option("bwd_2cta", old[1])


def _lse_err(lse, lse_ref):
    lse = to64(lse)
    masked = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), masked), "rows that see no key must have LSE = -inf"
    return max_abs(lse[~masked], lse_ref[~masked]) if (~masked).any() else 0.0


CASES = [
    # B, H, Hkv, Nq, Nk, d
    (1, 2, 2, 128, 512, 64),
    (2, 4, 2, 100, 333, 128),
    (1, 4, 1, 1, 1000, 128),
    (1, 2, 2, 512, 128, 64),
    (2, 4, 2, 300, 200, 128),
    (1, 2, 1, 640, 1280, 128),
    (1, 2, 2, 500, 200, 128),  # causal: whole query tiles that see no key (dQ = 0 there)
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES)
def test_qk_forward_backward(case, causal):
    B, H, Hkv, Nq, Nk, d = case
    q, k, v, do = make_inputs(B, H, Hkv, Nq, d, seed=400 + Nq + Nk + d, Nk=Nk)
    scale = d ** -0.5
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    qoff = Nk - Nq
    o_ref, lse_ref = ref.attn_fwd(to64(q), to64(k), to64(v), causal, scale, qpos=np.arange(Nq) + qoff)
    eo, el = o_error(to64(o), o_ref), _lse_err(lse, lse_ref)
    rq, rk, rv = ref.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale, qoff)
    errs = (rel_fro(to64(dq), rq), rel_fro(to64(dk), rk), rel_fro(to64(dv), rv))
    record("fwd", shape=[B, H, Hkv, Nq, Nk, d], causal=bool(causal), qk_mult=1.0, o_err=eo, lse_err=el,
           o_maxabs=max_abs(to64(o), o_ref), poly=0.0, tau=8.0)
    record("bwd", shape=[B, H, Hkv, Nq, Nk, d], causal=bool(causal), qk_mult=1.0, deterministic=False,
           dq_rel=errs[0], dk_rel=errs[1], dv_rel=errs[2])
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)
    assert max(errs) <= GRAD_RTOL, errs
    if causal and Nq > Nk:  # rows that see no key
        assert torch.all(o[:, :, :Nq - Nk] == 0) and torch.all(dq[:, :, :Nq - Nk] == 0)


@pytest.mark.parametrize("det", [False, True])
def test_qk_gqa_deterministic(det):
    B, H, Hkv, Nq, Nk, d = 2, 8, 2, 384, 1000, 128
    q, k, v, do = make_inputs(B, H, Hkv, Nq, d, seed=41, Nk=Nk)
    scale = d ** -0.5
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=True, scale=scale)
    outs = [fa.attention_backward(qd, kd, vd, o, dod, lse, causal=True, scale=scale, deterministic=det)
            for _ in range(2 if det else 1)]
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    rq, rk, rv = ref.attn_bwd(to64(q), to64(k), to64(v), to64(do), True, scale, Nk - Nq)
    dq, dk, dv = outs[0]
    errs = (rel_fro(to64(dq), rq), rel_fro(to64(dk), rk), rel_fro(to64(dv), rv))
    record("bwd", shape=[B, H, Hkv, Nq, Nk, d], causal=True, qk_mult=1.0, deterministic=det,
           dq_rel=errs[0], dk_rel=errs[1], dv_rel=errs[2])
    assert max(errs) <= GRAD_RTOL, errs
    if det:
        for a, b in zip(outs[0], outs[1]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_qk_no_keys_and_no_queries():
    B, H, Hkv, d = 1, 2, 1, 64
    q = torch.randn(B, H, 5, d, device="cuda").to(torch.bfloat16)
    k = torch.empty(B, Hkv, 0, d, device="cuda", dtype=torch.bfloat16)
    o, lse = fa.attention_forward(q, k, k.clone(), causal=True)
    dq, dk, dv = fa.attention_backward(q, k, k.clone(), o, torch.ones_like(q), lse, causal=True)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse)) and torch.all(dq == 0)
    q0 = torch.empty(B, H, 0, d, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(B, Hkv, 7, d, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, 7, d, device="cuda").to(torch.bfloat16)
    o0, lse0 = fa.attention_forward(q0, k, v)
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(v, 3.0)
    fa.attention_backward(q0, k, v, o0, q0.clone(), lse0, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
    assert fa.fa_last_device_status() == fa.FA_OK

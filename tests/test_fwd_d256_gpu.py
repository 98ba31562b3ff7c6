"""GPU parity of the d = 256 forward (one 128-row query tile per CTA: S and O take
384 of the 512 TMEM columns, and a second S buffer the rest) against the fp64
oracle, element by element: square and non-square shapes, causal and not, ragged
N, GQA, CTAs that run several units, and split-KV decoding."""
import numpy as np
import pytest
import torch

from exact_attention_49_gb300 import binding as fa
from exact_attention_49_gb300.inputs import make_inputs
from oracle import reference as ref
from parity import LSE_TOL, O_TOL, max_abs, o_error, record, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_attention_49_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()


@pytest.mark.parametrize("case", [
    # B, H, Hkv, Nq, Nk, causal
    (1, 2, 2, 256, 256, False),
    (1, 2, 2, 256, 256, True),
    (1, 3, 1, 333, 333, True),
    (2, 4, 2, 512, 512, True),
    (1, 2, 2, 100, 700, True),
    (1, 2, 1, 640, 200, True),
    # more units than SMs: each CTA runs several units, so the alternation of the two S
    # buffers carries across units (key-tile counts odd and even)
    (1, 32, 8, 1536, 1536, True),
    (1, 24, 24, 1000, 1000, False),
])
def test_fwd_d256(case):
    B, H, Hkv, Nq, Nk, causal = case
    d = 256
    q, k, v, _ = make_inputs(B, H, Hkv, Nq, d, seed=600 + Nq + Nk, Nk=Nk)
    scale = d ** -0.5
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    o_ref, lse_ref = ref.attn_fwd(to64(q), to64(k), to64(v), causal, scale, qpos=np.arange(Nq) + (Nk - Nq))
    masked = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(to64(lse)), masked)
    eo = o_error(to64(o), o_ref)
    el = max_abs(to64(lse)[~masked], lse_ref[~masked])
    record("fwd", shape=[B, H, Hkv, Nq, Nk, d], causal=bool(causal), qk_mult=1.0, o_err=eo, lse_err=el,
           o_maxabs=max_abs(to64(o), o_ref), poly=0.0, tau=8.0)
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)


def test_decode_d256():
    B, H, Hkv, Nq, Nk, d = 2, 8, 2, 1, 3000, 256
    q, k, v, _ = make_inputs(B, H, Hkv, Nq, d, seed=77, Nk=Nk)
    scale = d ** -0.5
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale, splits=0)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    o_ref, lse_ref = ref.attn_fwd(to64(q), to64(k), to64(v), True, scale, qpos=np.arange(Nq) + (Nk - Nq))
    eo, el = o_error(to64(o), o_ref), max_abs(to64(lse), lse_ref)
    record("fwd", shape=[B, H, Hkv, Nq, Nk, d], causal=True, qk_mult=1.0, o_err=eo, lse_err=el,
           o_maxabs=max_abs(to64(o), o_ref), poly=0.0, tau=8.0, splits=0)
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)


"""GPU parity of the split-KV (decoding) forward, fa_fwd_splitkv.

Few queries against many keys: the query heads of a K/V group are processed as
one block of rows and the keys are split over several CTAs whose partial
results are merged by their LSE.  The result is the same attention as
fa_fwd_qk (bottom-right causal mask when Nq != Nk), so every case is compared
with the fp64 oracle on every element: one decoding query, a few queries with
a causal mask (per-row positions inside the packed block), MQA/GQA/MHA, d = 64
and 128, ragged key counts, more splits than key tiles and the library's own
split choice; blocks of up to 128 rows with more than one split run in the
decoding configuration (two CTAs per SM), larger ones in the default form.
"""
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


CASES = [
    # B, H, Hkv, Nq, Nk, d, causal, splits
    (2, 8, 2, 1, 1000, 128, True, 0),
    (2, 8, 2, 1, 4096, 128, False, 0),
    (1, 4, 4, 1, 333, 64, True, 3),
    (2, 16, 2, 4, 2048, 128, True, 0),
    (1, 8, 1, 3, 700, 64, True, 5),
    (1, 4, 2, 16, 16384, 128, True, 0),
    (2, 4, 4, 1, 128, 128, True, 16),
    (1, 32, 8, 1, 8192, 128, True, 64),
    (1, 4, 2, 200, 600, 64, True, 2),
    (1, 32, 1, 4, 3000, 128, True, 0),   # 128 rows: the last size of the two-CTAs-per-SM form
    (1, 43, 1, 3, 1500, 64, True, 4),    # 129 rows: the 256-row form with splits
]


@pytest.mark.parametrize("case", CASES)
def test_decode_matches_oracle(case):
    B, H, Hkv, Nq, Nk, d, causal, splits = case
    q, k, v, _ = make_inputs(B, H, Hkv, Nq, d, seed=500 + Nq + Nk, Nk=Nk)
    scale = d ** -0.5
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    o_ref, lse_ref = ref.attn_fwd(to64(q), to64(k), to64(v), causal, scale, qpos=np.arange(Nq) + (Nk - Nq))
    eo, el = o_error(to64(o), o_ref), max_abs(to64(lse), lse_ref)
    record("fwd", shape=[B, H, Hkv, Nq, Nk, d], causal=bool(causal), qk_mult=1.0, o_err=eo, lse_err=el,
           o_maxabs=max_abs(to64(o), o_ref), poly=0.0, tau=8.0, splits=splits)
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)


def test_decode_workspace_and_split_choice():
    B, H, Hkv, Nq, Nk, d = 2, 8, 2, 1, 4096, 128
    assert fa.fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, 1) == 0
    auto = fa.fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, 0)
    four = fa.fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, 4)
    assert auto > 0 and four > 0
    q, k, v, _ = make_inputs(B, H, Hkv, Nq, d, seed=9, Nk=Nk)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = torch.empty_like(qd), torch.empty((B, H, Nq), device="cuda")
    ws = torch.empty(four, dtype=torch.uint8, device="cuda")
    args = (qd, kd, vd, o, lse, B, H, Hkv, Nq, Nk, d, 1, d ** -0.5, 4)
    assert fa.fa_fwd_splitkv(*args, ws, four - 256) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, None, four) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_splitkv(*args, ws, four) == fa.FA_OK
    o1, lse1 = fa.attention_forward(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    # the same attention: the split-KV result agrees with the one-pass forward to bf16 rounding
    assert (o.float() - o1.float()).abs().max().item() <= 2e-2
    assert (lse - lse1).abs().max().item() <= 1e-4

"""The device-side failure path, exercised without faulting the GPU.

Every wait inside the kernels is bounded.  The "debug_drop_kv_load" test hook
makes the forward's copy warp skip one K/V tile load, so the MMA warp's wait
for it runs out (about 2 s): the CTA raises its abort flag, the other roles stop
waiting, in-flight copies and MMAs drain, tensor memory is freed and the kernel
returns normally; fa_last_device_status() then reports FA_ERR_DEVICE_TIMEOUT.
The next call on the same context must work and be correct.

The backward has two hooks ("debug_bwd_hook"): 1 makes the first CTA never
release the deterministic mode's ordering counters, so the next key tile's
bounded spin on the counter runs out (at d = 256: the first pair of CTAs, both
head-dimension halves of one key tile); 2 makes the copy warp skip one Q/dO tile
load (at d = 256: stop loading after the first query tile), so the MMA warp's wait
on that stage's mbarrier runs out.
"""
import pytest
import torch

from exact_attention_49_gb300 import binding as fa
from exact_attention_49_gb300.inputs import make_inputs
from oracle import reference as ref
from parity import GRAD_RTOL, LSE_TOL, O_TOL, max_abs, o_error, rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_attention_49_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()


@pytest.mark.parametrize("d,pair", [(64, 0), (128, 1)], ids=["1cta", "2cta"])
def test_bounded_wait_reports_timeout_and_context_survives(d, pair):
    B, H, Hkv, N = 1, 1, 1, 512
    old_pair = fa.fa_get_option("fwd_2cta")
    assert fa.fa_set_option("fwd_2cta", pair) == fa.FA_OK
    q, k, v, _ = make_inputs(B, H, Hkv, N, d, seed=5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert fa.fa_set_option("debug_drop_kv_load", 1) == fa.FA_OK
    try:
        fa.attention_forward(qd, kd, vd, causal=False)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    finally:
        assert fa.fa_set_option("debug_drop_kv_load", 0) == fa.FA_OK
    # the status was cleared by the read; the context is healthy and results are right
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse = fa.attention_forward(qd, kd, vd, causal=False)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    fa.fa_set_option("fwd_2cta", old_pair)
    o_ref, lse_ref = ref.attn_fwd(to64(q), to64(k), to64(v), False, d ** -0.5)
    assert o_error(to64(o), o_ref) <= O_TOL
    assert max_abs(to64(lse), lse_ref) <= LSE_TOL


@pytest.mark.parametrize("d,pair", [(128, 0), (128, 1), (256, 0)], ids=["1cta", "2cta", "d256"])
@pytest.mark.parametrize("hook,causal,det", [(1, True, True), (2, False, False)])
def test_backward_bounded_waits_report_timeout(hook, causal, det, d, pair):
    B, H, Hkv, N = 1, 1, 1, 512
    q, k, v, do = make_inputs(B, H, Hkv, N, d, seed=6)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    old_pair = fa.fa_get_option("bwd_2cta")
    assert fa.fa_set_option("bwd_2cta", pair) == fa.FA_OK
    assert fa.fa_set_option("debug_bwd_hook", hook) == fa.FA_OK
    try:
        fa.attention_backward(qd, kd, vd, o, dod, lse, causal=causal, deterministic=det)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    finally:
        assert fa.fa_set_option("debug_bwd_hook", 0) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, causal=causal, deterministic=det)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    fa.fa_set_option("bwd_2cta", old_pair)
    rq, rk, rv = ref.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, d ** -0.5)
    for got, want in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel_fro(to64(got), want) <= GRAD_RTOL

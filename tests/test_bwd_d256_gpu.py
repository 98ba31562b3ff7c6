"""GPU parity of the d = 256 backward against the fp64 oracle's analytic backward.

At d = 256 the main stage runs two CTAs per 128-key tile, one per head-dimension half, on
64-row query tiles.  The cases cover both halves meeting in every output (dQ through the fp32
reductions of both CTAs, dK and dV written half by half), causal and not, ragged N (a query
tile and a key tile past N), GQA (dK, dV summed over the group inside the CTA), Nq != Nk
(bottom-right causal alignment, rows that see no key), the deterministic mode (one ordering
counter per query tile and half; bit-identical across runs), and a key tile that no query row
sees (zero dK, dV).
"""
import numpy as np
import pytest
import torch

from exact_attention_49_gb300 import binding as fa
from exact_attention_49_gb300.inputs import make_inputs
from oracle import reference as ref
from parity import GRAD_RTOL, ROW_TOL, record, rel_fro, row_err, to64

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_attention_49_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()


def _run(B, H, Hkv, Nq, Nk, causal, seed, det=False, repeats=1):
    q, k, v, do = make_inputs(B, H, Hkv, Nq, D, seed=seed, Nk=Nk)
    scale = D ** -0.5
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    outs = [fa.attention_backward(qd, kd, vd, o, dod, lse, causal=causal, scale=scale, deterministic=det)
            for _ in range(repeats)]
    torch.cuda.synchronize()
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.status_string(st)
    rq, rk, rv = ref.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale, Nk - Nq)
    return outs, (rq, rk, rv)


def _check(outs, refs, shape, causal, det, per_head=False):
    errs, rows = [], []
    for got, want in zip(outs[0], refs):
        g64 = to64(got)
        if per_head:  # every head on its own, so a tile spilling into a neighbour shows up
            errs.append(max(rel_fro(g64[b, h], want[b, h]) for b in range(g64.shape[0])
                            for h in range(g64.shape[1])))
        else:
            errs.append(rel_fro(g64, want))
        rows.append(row_err(g64, want))
    record("bwd", shape=shape, causal=bool(causal), qk_mult=1.0, deterministic=bool(det), pair=0,
           dq_rel=errs[0], dk_rel=errs[1], dv_rel=errs[2], dq_row=rows[0], dk_row=rows[1], dv_row=rows[2])
    assert max(errs) <= GRAD_RTOL, errs
    assert max(rows) <= ROW_TOL, rows


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 256, 640])
def test_bwd_d256_small(N, causal):
    outs, refs = _run(1, 2, 2, N, N, causal, seed=700 + N)
    _check(outs, refs, [1, 2, 2, N, D], causal, False)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 200, 333, 1000])
def test_bwd_d256_ragged(N, causal):
    outs, refs = _run(2, 4, 2, N, N, causal, seed=710 + N)
    _check(outs, refs, [2, 4, 2, N, D], causal, False, per_head=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("det", [False, True])
def test_bwd_d256_gqa(causal, det):
    outs, refs = _run(2, 8, 2, 512, 512, causal, seed=720, det=det)
    _check(outs, refs, [2, 8, 2, 512, D], causal, det)


@pytest.mark.parametrize("Nq,Nk", [(100, 700), (640, 200), (300, 300)])
def test_bwd_d256_nq_ne_nk(Nq, Nk):
    outs, refs = _run(1, 4, 2, Nq, Nk, True, seed=730 + Nq + Nk)
    _check(outs, refs, [1, 4, 2, Nq, Nk, D], True, False)
    dq = outs[0][0]
    if Nq > Nk:  # query rows placed before the first key see nothing
        assert torch.all(dq[:, :, :Nq - Nk] == 0)


@pytest.mark.parametrize("Hkv", [2, 8], ids=["grouped", "one_head_per_group"])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_d256_deterministic_bit_identical(causal, Hkv):
    outs, refs = _run(2, 8, Hkv, 1024, 1024, causal, seed=740, det=True, repeats=3)
    _check(outs, refs, [2, 8, Hkv, 1024, D], causal, True)
    for again in outs[1:]:
        for a, b in zip(outs[0], again):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bwd_d256_workspace_counters():
    """The deterministic mode's counters at d = 256: one per 64-row query tile and half."""
    B, H, Hkv, N = 2, 4, 2, 300
    plain = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, D, 0)
    det = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, D, 1)
    rows = B * H * 384
    assert plain >= rows * D * 4 + 2 * rows * 4
    assert det - plain >= rows // 32 * 4

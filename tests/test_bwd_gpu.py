"""GPU parity of fa_bwd against the fp64 CPU oracle's analytic backward.

The GPU backward consumes the GPU forward's O and LSE (as a training step
would); the oracle computes the gradients of sum(O * dO) from Q, K, V, dO
alone.  Small cases are compared on every element; the full-size workloads run
on the GPU at full size and are compared on sampled query heads (dQ) and on the
K/V heads they belong to (dK, dV summed over the whole group).  The
deterministic mode is also checked for bit-identical results across runs.
"""
import numpy as np
import pytest
import torch

from exact_attention_49_gb300 import binding as fa
from exact_attention_49_gb300.inputs import WORKLOADS, make_inputs
from oracle import reference as ref
from parity import GRAD_RTOL, ROW_TOL, record, rel_fro, row_err, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_attention_49_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()


@pytest.fixture(autouse=True, params=[0, 1], ids=["1cta", "2cta"])
def bwd_mode(request):
    """Every backward test runs on both main-stage kernels: one CTA per 128-key tile, and CTA
    pairs over 256 keys with tcgen05 cta_group::2 MMAs (head dimension 128; at d = 64 both
    settings run the one-CTA kernel)."""
    old = fa.fa_get_option("bwd_2cta")
    assert fa.fa_set_option("bwd_2cta", request.param) == fa.FA_OK
    yield request.param
    fa.fa_set_option("bwd_2cta", old)


def gpu_fwd_bwd(q, k, v, do, causal, scale, deterministic=False):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, dod, lse, causal=causal, scale=scale,
                                       deterministic=deterministic)
    torch.cuda.synchronize()
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.status_string(st)
    return dq, dk, dv


def check_full(B, H, Hkv, N, d, causal, seed, qk_mult=1.0, deterministic=False):
    q, k, v, do = make_inputs(B, H, Hkv, N, d, seed, qk_mult)
    scale = d ** -0.5
    dq, dk, dv = gpu_fwd_bwd(q, k, v, do, causal, scale, deterministic)
    rq, rk, rv = ref.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale)
    errs = (rel_fro(to64(dq), rq), rel_fro(to64(dk), rk), rel_fro(to64(dv), rv))
    rows = (row_err(to64(dq), rq), row_err(to64(dk), rk), row_err(to64(dv), rv))
    record("bwd", shape=[B, H, Hkv, N, d], causal=bool(causal), qk_mult=qk_mult, deterministic=bool(deterministic),
           pair=fa.fa_get_option("bwd_2cta"), dq_rel=errs[0], dk_rel=errs[1], dv_rel=errs[2], dq_row=rows[0],
           dk_row=rows[1], dv_row=rows[2])
    assert max(errs) <= GRAD_RTOL, errs
    assert max(rows) <= ROW_TOL, rows
    return errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 256, 640])
def test_bwd_small(N, causal, d):
    check_full(1, 2, 2, N, d, causal, seed=200 + N + d)


def test_bwd_c1():
    w = WORKLOADS["C1"]
    check_full(w.B, w.H, w.Hkv, w.N, w.d, w.causal, w.seed)


def test_bwd_c2():
    w = WORKLOADS["C2"]
    check_full(w.B, w.H, w.Hkv, w.N, w.d, w.causal, w.seed)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("det", [False, True])
def test_bwd_gqa_small(causal, d, det):
    check_full(2, 8, 2, 512, d, causal, seed=17, deterministic=det)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 200, 333, 1000])
def test_bwd_ragged(N, causal, d):
    """N not a multiple of 128: the last query and key tiles run past N (TMA zero fill, padded
    workspace rows, masked key rows).  Every head is compared on its own, so a tile that
    spilled into a neighbouring head's rows would show up."""
    B, H, Hkv = 2, 4, 2
    q, k, v, do = make_inputs(B, H, Hkv, N, d, seed=300 + N + d)
    scale = d ** -0.5
    dq, dk, dv = gpu_fwd_bwd(q, k, v, do, causal, scale)
    rq, rk, rv = ref.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale)
    errs, rows = [], []
    for got, want in ((dq, rq), (dk, rk), (dv, rv)):
        g64 = to64(got)
        errs.append(max(rel_fro(g64[b, h], want[b, h]) for b in range(B) for h in range(got.shape[1])))
        rows.append(row_err(g64, want))
    record("bwd", shape=[B, H, Hkv, N, d], causal=bool(causal), qk_mult=1.0, deterministic=False,
           pair=fa.fa_get_option("bwd_2cta"), dq_rel=errs[0], dk_rel=errs[1], dv_rel=errs[2], dq_row=rows[0],
           dk_row=rows[1], dv_row=rows[2])
    assert max(errs) <= GRAD_RTOL, errs
    assert max(rows) <= ROW_TOL, rows


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_deterministic_one_head_per_group(causal, d):
    """Deterministic mode without grouped heads: under a causal mask the contributions run in
    descending key-tile order (the schedule for H == Hkv); ragged N, bit-identical reruns."""
    B, H, Hkv, N = 2, 4, 4, 700
    check_full(B, H, Hkv, N, d, causal, seed=29 + d, deterministic=True)
    q, k, v, do = make_inputs(B, H, Hkv, N, d, seed=29 + d)
    first = gpu_fwd_bwd(q, k, v, do, causal, d ** -0.5, deterministic=True)
    again = gpu_fwd_bwd(q, k, v, do, causal, d ** -0.5, deterministic=True)
    for a, b in zip(first, again):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("det", [False, True])
def test_bwd_ragged_gqa(det):
    check_full(2, 8, 2, 700, 128, True, seed=23, deterministic=det)


def test_bwd_stress_rescale_inputs():
    check_full(1, 4, 4, 1024, 128, True, seed=19, qk_mult=4.0)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_deterministic_bit_identical(causal):
    B, H, Hkv, N, d = 2, 8, 2, 1024, 128
    q, k, v, do = make_inputs(B, H, Hkv, N, d, seed=23)
    scale = d ** -0.5
    first = gpu_fwd_bwd(q, k, v, do, causal, scale, deterministic=True)
    for _ in range(2):
        again = gpu_fwd_bwd(q, k, v, do, causal, scale, deterministic=True)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bwd_workspace_checks():
    B, H, Hkv, N, d = 1, 2, 2, 256, 64
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, Hkv, N, d, seed=1))
    o, lse = fa.attention_forward(q, k, v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (q, k, v, o, do, lse, dq, dk, dv, B, H, Hkv, N, d, 0, d ** -0.5, 0)
    assert fa.fa_bwd(*args, ws, need - 256) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd(*args, None, need) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd(*args, ws, need) == fa.FA_OK
    bad = (q, k, v, o, do, lse, dq, dk, dv, B, H, Hkv, N, 96, 0, d ** -0.5, 0)
    assert fa.fa_bwd(*bad, ws, need) == fa.FA_ERR_UNSUPPORTED
    torch.cuda.synchronize()


def _sample_heads(B, H, seed, n=4):
    rng = np.random.default_rng(seed)
    pick = {(0, 0), (B - 1, H - 1)}
    while len(pick) < min(n, B * H):
        pick.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(pick)


@pytest.mark.parametrize("name,det", [("C3", False), ("C3b", False), ("C4", False), ("C4", True)])
def test_bwd_full_size_sampled(name, det):
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w.B, w.H, w.Hkv, w.N, w.d, w.seed, w.qk_mult)
    dq, dk, dv = gpu_fwd_bwd(q, k, v, do, w.causal, w.scale, deterministic=det)
    grp = w.H // w.Hkv
    # whole K/V groups around sampled query heads: (0,0), (B-1,H-1) and, for
    # single-head groups, two seeded-random heads (GQA groups are 4x the oracle work)
    groups = sorted({(b, h // grp) for b, h in _sample_heads(w.B, w.H, w.seed, n=4 if grp == 1 else 2)})
    for b, g in groups:
        hs = slice(g * grp, (g + 1) * grp)
        rq, rk, rv = ref.attn_bwd(to64(q[b:b + 1, hs]), to64(k[b:b + 1, g:g + 1]), to64(v[b:b + 1, g:g + 1]),
                                  to64(do[b:b + 1, hs]), w.causal, w.scale)
        got = (to64(dq[b:b + 1, hs]), to64(dk[b:b + 1, g:g + 1]), to64(dv[b:b + 1, g:g + 1]))
        errs = tuple(rel_fro(x, r) for x, r in zip(got, (rq, rk, rv)))
        rows = tuple(row_err(x, r) for x, r in zip(got, (rq, rk, rv)))
        record("bwd_full_size", workload=w.name, deterministic=bool(det), pair=fa.fa_get_option("bwd_2cta"),
               group=[b, g], dq_rel=errs[0],
               dk_rel=errs[1], dv_rel=errs[2], dq_row=rows[0], dk_row=rows[1], dv_row=rows[2])
        assert max(errs) <= GRAD_RTOL, ((b, g), errs)
        assert max(rows) <= ROW_TOL, ((b, g), rows)


@pytest.mark.parametrize("name", ["C3", "C4"])
def test_bwd_deterministic_bit_identical_full_size(name):
    """Deterministic mode at the full benchmark sizes (B4 H16 N8192 and the GQA B2 Hq32 Hkv8
    N16384 workload), where many CTAs contend for each query tile's ordering counter: two runs
    give the same dQ, dK, dV bits."""
    w = WORKLOADS[name]
    q, k, v, do = (t.cuda() for t in make_inputs(w.B, w.H, w.Hkv, w.N, w.d, w.seed, w.qk_mult))
    o, lse = fa.attention_forward(q, k, v, causal=w.causal, scale=w.scale)
    first = fa.attention_backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, deterministic=True)
    again = fa.attention_backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, deterministic=True)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for a, b in zip(first, again):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bwd_pair_matches_single_cta():
    """The two main-stage kernels compute the same sums in a different order (the pair adds
    each query tile's dQ over 256 keys on chip before the fp32 reductions): their results
    agree to the rounding of those orders."""
    B, H, Hkv, N, d = 2, 8, 2, 1000, 128
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, Hkv, N, d, seed=29))
    o, lse = fa.attention_forward(q, k, v, causal=True)
    res = []
    for mode in (0, 1):
        assert fa.fa_set_option("bwd_2cta", mode) == fa.FA_OK
        res.append(fa.attention_backward(q, k, v, o, do, lse, causal=True, deterministic=True))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for a, b in zip(*res):
        assert rel_fro(to64(a), to64(b)) < 5e-3
    # the option switched the kernel: dQ's fp32 sums run in another order, so some of its bf16
    # values differ (about 1e-4 of them round the other way)
    assert not torch.equal(res[0][0], res[1][0])

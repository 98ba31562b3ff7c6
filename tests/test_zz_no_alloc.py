"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers have no device allocator at the point of the call (a plugin run
by a framework that owns all device memory, or a latency-critical path where
cudaMalloc is not allowed).  fa_bwd_noalloc serves them by using a fixed scratch
array inside the library instead of a caller-allocated workspace.  This test
calls it through the C ABI twice in a row and checks both results against the
ordinary fa_bwd (with a caller-allocated workspace), within the gradient
tolerance the other backward tests use.  It lives in its own file, named to be
collected last, and works both alone in a fresh process and after the others.
"""
import ctypes

import pytest
import torch

from exact_attention_49_gb300 import binding as fa
from exact_attention_49_gb300.inputs import make_inputs
from parity import GRAD_RTOL, rel_fro, to64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


@pytest.fixture(scope="module")
def noalloc():
    from exact_attention_49_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fn = fa.lib().fa_bwd_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P] * 9 + [I] * 6 + [ctypes.c_float, I, P]
    fn.restype = I
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("d,causal,det", [(64, True, 0), (128, True, 0), (128, False, 1), (128, True, 1),
                                           (256, True, 1)])
def test_noalloc_matches_fa_bwd_twice(noalloc, d, causal, det):
    B, H, Hkv, N = 2, 4, 2, 512
    scale = d ** -0.5
    q, k, v, do = (t.cuda() for t in make_inputs(B, H, Hkv, N, d, seed=31 + d))
    o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale)
    ref = fa.attention_backward(q, k, v, o, do, lse, causal=causal, scale=scale, deterministic=bool(det))
    torch.cuda.synchronize()
    assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d, det) <= SCRATCH_BYTES
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                     B, H, Hkv, N, d, int(causal), scale, det, stream)
        assert st == fa.FA_OK, fa.status_string(st)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        for got, want in zip((dq, dk, dv), ref):
            assert rel_fro(to64(got), to64(want)) <= GRAD_RTOL
            if det:
                assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_noalloc_large_then_small_problem(noalloc):
    """The scratch keeps whatever the previous call left in it; a smaller problem after a
    larger one (deterministic, so the ordering counters are reused too) must still match
    fa_bwd bit for bit."""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for B, H, Hkv, N in ((2, 8, 2, 1024), (1, 2, 1, 384)):
        d, causal = 128, True
        scale = d ** -0.5
        assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d, 1) <= SCRATCH_BYTES
        q, k, v, do = (t.cuda() for t in make_inputs(B, H, Hkv, N, d, seed=40 + N))
        o, lse = fa.attention_forward(q, k, v, causal=causal, scale=scale)
        want = fa.attention_backward(q, k, v, o, do, lse, causal=causal, scale=scale, deterministic=True)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                     B, H, Hkv, N, d, int(causal), scale, 1, stream)
        assert st == fa.FA_OK, fa.status_string(st)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        for got, ref_t in zip((dq, dk, dv), want):
            assert torch.equal(got.view(torch.int16), ref_t.view(torch.int16))


def test_noalloc_rejects_problems_beyond_the_scratch(noalloc):
    B, H, Hkv, N, d = 8, 16, 16, 1024, 128
    assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d, 0) > SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = noalloc(*([fake] * 9), B, H, Hkv, N, d, 1, d ** -0.5, 0, None)
    assert st == fa.FA_ERR_WORKSPACE

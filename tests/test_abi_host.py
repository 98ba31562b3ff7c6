"""Host-only checks of the C ABI: the library builds and loads, exports every
function that include/fa.h declares, and rejects bad arguments with the
documented status code before touching any GPU (these calls run on machines
with no GPU at all)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    from exact_attention_49_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_set_option",
                     "fa_status_string", "fa_last_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    from exact_attention_49_gb300 import binding as fa
    assert fa.fa_version() >= 100
    for code in range(-6, 1):
        assert fa.status_string(code) not in ("", "unknown status")
    assert fa.status_string(42) == "unknown status"


def test_options_roundtrip(L):
    from exact_attention_49_gb300 import binding as fa
    old = fa.fa_get_option("rescale_threshold")
    assert fa.fa_set_option("rescale_threshold", 0.0) == fa.FA_OK
    assert fa.fa_get_option("rescale_threshold") == 0.0
    assert fa.fa_set_option("rescale_threshold", old) == fa.FA_OK
    assert fa.fa_set_option("rescale_threshold", -1.0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_option("poly_exp", 33) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_option("poly_exp", 2.5) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_option("poly_exp", 6) == fa.FA_ERR_INVALID_ARG
    for ok in (-1, 0, 4, 8, 12, 16):
        assert fa.fa_set_option("poly_exp", ok) == fa.FA_OK
    assert fa.fa_set_option("poly_exp", -1) == fa.FA_OK
    assert fa.fa_set_option("no_such_option", 1.0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_option("debug_drop_kv_load", 2) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_get_option("debug_drop_kv_load") == 0.0
    # the exponential split as a fraction of the exponentials (columns of 32 / 32)
    for frac, cols in ((0.0, 0), (0.125, 4), (0.25, 8), (0.375, 12), (0.5, 16)):
        assert fa.fa_set_option("poly_fraction", frac) == fa.FA_OK
        assert fa.fa_get_option("poly_exp") == cols
        assert fa.fa_get_option("poly_fraction") == frac
    assert fa.fa_set_option("poly_fraction", 0.3) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_option("poly_fraction", -1) == fa.FA_OK
    assert fa.fa_get_option("poly_exp") == -1
    for key, good, bad in (("debug_bwd_hook", (0, 1, 2), (3, -1, 0.5)), ("count_rescales", (0, 1), (2, 0.5)),
                           ("bwd_2cta", (0, 1), (2, -1)), ("fwd_2cta", (0, 1), (2, -1))):
        for val in good:
            assert fa.fa_set_option(key, val) == fa.FA_OK
            assert fa.fa_get_option(key) == val
        for val in bad:
            assert fa.fa_set_option(key, val) == fa.FA_ERR_INVALID_ARG
        assert fa.fa_set_option(key, 0) == fa.FA_OK
    # the event counter can only be cleared (to 0), and only with a device
    assert fa.fa_set_option("rescale_events", 5) == fa.FA_ERR_INVALID_ARG


def test_row_diagnostic_catches_one_wrong_row():
    """The per-row gradient diagnostic of the parity tests: rounding-size noise scores far
    below its bound, one row replaced by another row's values scores about 1."""
    import numpy as np
    from parity import ROW_TOL, rel_fro, row_err
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((1, 2, 8192, 128))
    noisy = ref * (1 + 2.0 ** -8 * rng.standard_normal(ref.shape))
    assert row_err(noisy, ref) < 0.05 * ROW_TOL
    bad = noisy.copy()
    bad[0, 1, 4000] = ref[0, 1, 17]
    assert rel_fro(bad, ref) < 0.02          # hidden by the whole-tensor norm
    assert row_err(bad, ref) > 4 * ROW_TOL   # caught by the row diagnostic


P = ctypes.c_void_p
GOOD = P(1 << 20)          # never dereferenced: every case below fails validation first
BAD = P((1 << 20) + 8)     # 8-byte aligned only


def fwd(L, q=GOOD, k=GOOD, v=GOOD, o=GOOD, lse=GOOD, B=1, H=2, Hkv=1, N=128, d=64, causal=0, scale=0.125):
    return L.fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, None)


def test_fwd_validation(L):
    from exact_attention_49_gb300 import binding as fa
    assert fwd(L, q=None) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, lse=None) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, H=3, Hkv=2) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, d=96) == fa.FA_ERR_UNSUPPORTED
    assert fwd(L, d=192) == fa.FA_ERR_UNSUPPORTED  # d = 256 is a forward-only size
    assert fwd(L, q=BAD) == fa.FA_ERR_MISALIGNED
    assert fwd(L, o=BAD) == fa.FA_ERR_MISALIGNED
    assert fwd(L, lse=P((1 << 20) + 2)) == fa.FA_ERR_MISALIGNED
    assert fwd(L, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, causal=2) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, B=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd(L, N=-5) == fa.FA_ERR_INVALID_ARG
    # empty problems are valid and launch nothing, even with NULL pointers
    assert fwd(L, N=0, q=None, k=None, v=None, o=None, lse=None) == fa.FA_OK
    assert fwd(L, B=0, q=None, k=None, v=None, o=None, lse=None) == fa.FA_OK


def test_workspace_size(L):
    from exact_attention_49_gb300 import binding as fa
    B, H, N, d = 2, 4, 256, 64
    ws = fa.fa_bwd_workspace_bytes(B, H, 2, N, d, 0)
    assert ws >= B * H * N * d * 4 + B * H * N * 4
    assert fa.fa_bwd_workspace_bytes(B, H, 2, N, d, 1) > ws
    assert fa.fa_bwd_workspace_bytes(B, 3, 2, N, d, 0) == 0
    assert fa.fa_bwd_workspace_bytes(B, H, 2, N, 96, 0) == 0
    # d = 256: same accumulator layout; its counters are one per 64-row query tile and half
    assert fa.fa_bwd_workspace_bytes(B, H, 2, N, 256, 0) >= B * H * N * 256 * 4 + B * H * N * 8
    assert (fa.fa_bwd_workspace_bytes(B, H, 2, N, 256, 1) - fa.fa_bwd_workspace_bytes(B, H, 2, N, 256, 0)
            >= B * H * N // 32 * 4)
    # rows are padded per head to a multiple of 128
    assert fa.fa_bwd_workspace_bytes(B, H, 2, 200, d, 0) == fa.fa_bwd_workspace_bytes(B, H, 2, 256, d, 0)
    assert fa.fa_bwd_workspace_bytes(B, H, 2, 1, d, 1) == fa.fa_bwd_workspace_bytes(B, H, 2, 128, d, 1)


def test_bwd_validation(L):
    from exact_attention_49_gb300 import binding as fa
    def bwd(q=GOOD, B=1, H=2, Hkv=1, N=256, d=64, causal=0, scale=0.125, det=0, ws=GOOD, wsb=1 << 30):
        return L.fa_bwd(q, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, B, H, Hkv, N, d, causal, scale, det,
                        ws, wsb, None)
    assert bwd(q=None) == fa.FA_ERR_INVALID_ARG
    assert bwd(H=3, Hkv=2) == fa.FA_ERR_INVALID_ARG
    assert bwd(d=80) == fa.FA_ERR_UNSUPPORTED
    assert bwd(d=192) == fa.FA_ERR_UNSUPPORTED  # the backward supports d = 64, 128 and 256
    # any N is accepted; a ragged N needs the workspace of N rounded up to 128 rows per head
    assert bwd(N=200, wsb=fa.fa_bwd_workspace_bytes(1, 2, 1, 200, 64, 0) - 256) == fa.FA_ERR_WORKSPACE
    assert bwd(ws=None) == fa.FA_ERR_WORKSPACE
    assert bwd(wsb=1024) == fa.FA_ERR_WORKSPACE
    assert bwd(ws=P((1 << 20) + 16)) == fa.FA_ERR_MISALIGNED
    assert bwd(q=BAD) == fa.FA_ERR_MISALIGNED
    assert bwd(det=2) == fa.FA_ERR_INVALID_ARG
    assert bwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert bwd(N=0, q=None, ws=None) == fa.FA_OK


def test_qk_and_splitkv_validation(L):
    """fa_fwd_qk / fa_bwd_qk / fa_fwd_splitkv reject bad arguments before any launch."""
    from exact_attention_49_gb300 import binding as fa

    def fwd_qk(q=GOOD, k=GOOD, B=1, H=2, Hkv=1, Nq=64, Nk=300, d=64, causal=1, scale=0.125):
        return L.fa_fwd_qk(q, k, GOOD, GOOD, GOOD, B, H, Hkv, Nq, Nk, d, causal, scale, None)

    assert fwd_qk(q=None) == fa.FA_ERR_INVALID_ARG
    assert fwd_qk(Nk=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd_qk(d=96) == fa.FA_ERR_UNSUPPORTED
    assert fwd_qk(k=BAD) == fa.FA_ERR_MISALIGNED
    assert fwd_qk(causal=3) == fa.FA_ERR_INVALID_ARG
    assert fwd_qk(Nq=0, q=None, k=None) == fa.FA_OK  # no query: nothing to do

    def bwd_qk(q=GOOD, Nq=64, Nk=300, d=64, ws=GOOD, wsb=1 << 30, det=0):
        return L.fa_bwd_qk(q, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, 1, 2, 1, Nq, Nk, d, 1, 0.125, det,
                           ws, wsb, None)

    assert bwd_qk(q=None) == fa.FA_ERR_INVALID_ARG
    assert bwd_qk(Nk=-3) == fa.FA_ERR_INVALID_ARG
    assert bwd_qk(ws=None) == fa.FA_ERR_WORKSPACE
    assert bwd_qk(det=5) == fa.FA_ERR_INVALID_ARG
    # the workspace depends on Nq only (rows padded to 128), not on Nk
    w1 = fa.fa_bwd_qk_workspace_bytes(1, 2, 1, 64, 300, 64, 0)
    assert w1 == fa.fa_bwd_qk_workspace_bytes(1, 2, 1, 100, 5000, 64, 0) == fa.fa_bwd_workspace_bytes(1, 2, 1, 128, 64, 0)
    assert fa.fa_bwd_qk_workspace_bytes(1, 2, 1, 64, -1, 64, 0) == 0

    def dec(splits=4, ws=GOOD, wsb=1 << 30, Nq=1, Nk=4096, d=128):
        return L.fa_fwd_splitkv(GOOD, GOOD, GOOD, GOOD, GOOD, 2, 8, 2, Nq, Nk, d, 1, 0.125, splits, ws, wsb, None)

    assert dec(splits=-1) == fa.FA_ERR_INVALID_ARG
    assert dec(splits=5000) == fa.FA_ERR_INVALID_ARG
    assert dec(d=80) == fa.FA_ERR_UNSUPPORTED
    assert dec(ws=None) == fa.FA_ERR_WORKSPACE
    assert dec(wsb=16) == fa.FA_ERR_WORKSPACE
    assert dec(ws=P((1 << 20) + 16)) == fa.FA_ERR_MISALIGNED
    # one split needs no workspace; several need room for their fp32 partials and LSEs
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 2, 1, 4096, 128, 1) == 0
    rows = 2 * 8 * 1
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 2, 1, 4096, 128, 4) >= 4 * rows * 128 * 4 + 4 * rows * 4
    # more splits than key tiles are clamped to the key tiles
    assert (fa.fa_fwd_splitkv_workspace_bytes(2, 8, 2, 1, 256, 128, 64)
            == fa.fa_fwd_splitkv_workspace_bytes(2, 8, 2, 1, 256, 128, 2))
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 2, 1, 4096, 128, 0) > 0


def test_header_is_plain_c(tmp_path):
    """include/fa.h is usable from C99 (no C++ in the interface): a translation unit that
    calls every entry point compiles with gcc -std=c99 -Wall -Wextra -Werror."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_fa.c"
    src.write_text(r'''
#include <stddef.h>
#include "fa.h"
int use_fa(void* q, void* k, void* v, void* o, float* lse, void* ws, size_t wsb) {
  int st = fa_fwd(q, k, v, o, lse, 1, 2, 1, 128, 64, 1, 0.125f, NULL);
  st |= fa_fwd_qk(q, k, v, o, lse, 1, 2, 1, 1, 128, 64, 1, 0.125f, NULL);
  st |= fa_fwd_splitkv(q, k, v, o, lse, 1, 2, 1, 1, 128, 64, 1, 0.125f, 0, ws,
                       fa_fwd_splitkv_workspace_bytes(1, 2, 1, 1, 128, 64, 0), NULL);
  st |= fa_bwd(q, k, v, o, o, lse, q, k, v, 1, 2, 1, 128, 64, 1, 0.125f, 0, ws,
               fa_bwd_workspace_bytes(1, 2, 1, 128, 64, 0), NULL);
  st |= fa_bwd_qk(q, k, v, o, o, lse, q, k, v, 1, 2, 1, 64, 128, 64, 1, 0.125f, 1, ws,
                  fa_bwd_qk_workspace_bytes(1, 2, 1, 64, 128, 64, 1), NULL);
  st |= fa_bwd_preprocess(o, o, lse, 1, 2, 1, 128, 64, 0, ws, wsb, NULL);
  st |= fa_bwd_main(q, k, v, o, lse, k, v, 1, 2, 1, 128, 64, 1, 0.125f, 0, ws, wsb, NULL);
  st |= fa_bwd_postprocess(q, 1, 2, 1, 128, 64, 0, ws, wsb, NULL);
  st |= fa_bwd_noalloc(q, k, v, o, o, lse, q, k, v, 1, 2, 1, 128, 64, 1, 0.125f, 0, NULL);
  double val = 0.0;
  st |= fa_set_option("rescale_threshold", 8.0) | fa_get_option("rescale_threshold", &val);
  (void)fa_status_string(st);
  (void)fa_last_error_detail();
  st |= fa_last_device_status(NULL) | fa_version();
  return st + (val > 0.0 ? 0 : 1) + (int)(FA_NOALLOC_SCRATCH_BYTES > 0u);
}
''')
    out = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c", str(src),
                          "-I", os.path.join(ROOT, "include"), "-o", str(tmp_path / "use_fa.o")],
                         capture_output=True, text=True)
    assert out.returncode == 0, out.stderr


def test_noalloc_validates_like_fa_bwd(L):
    """fa_bwd_noalloc makes fa_bwd's checks in fa_bwd's order (the scratch standing in for the
    workspace), so both give the same status on every rejected call; none of these touches
    the GPU."""
    L.fa_bwd_noalloc.restype = ctypes.c_int
    L.fa_bwd_noalloc.argtypes = [P] * 9 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, P]
    big_ws = 1 << 40  # any size: the checks below fail before the workspace size matters
    cases = [
        dict(d=96, N=0),                 # unsupported d even with no rows
        dict(d=192, N=128),              # unsupported d with rows
        dict(H=3, Hkv=2),                # H % Hkv != 0
        dict(det=2),                     # bad deterministic flag
        dict(causal=2),                  # bad causal flag
        dict(scale=float("nan")),        # bad scale
        dict(q=None),                    # null pointer
        dict(k=BAD),                     # misaligned pointer
    ]
    for c in cases:
        a = dict(q=GOOD, k=GOOD, v=GOOD, o=GOOD, do=GOOD, lse=GOOD, dq=GOOD, dk=GOOD, dv=GOOD, B=1, H=2, Hkv=1,
                 N=128, d=64, causal=0, scale=0.125, det=0)
        a.update(c)
        ptrs = [a[n] for n in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv")]
        sizes = (a["B"], a["H"], a["Hkv"], a["N"], a["d"], a["causal"])
        want = L.fa_bwd(*ptrs, *sizes, a["scale"], a["det"], GOOD, big_ws, None)
        got = L.fa_bwd_noalloc(*ptrs, *sizes, a["scale"], a["det"], None)
        assert want != 0 and got == want, (c, got, want)
    # nothing to do: both return FA_OK without touching the GPU
    assert L.fa_bwd_noalloc(*([GOOD] * 9), 0, 2, 1, 128, 64, 0, 0.125, 0, None) == 0


def test_fp8_validation(L):
    """FP8 entry points: sizes, head dimension, arguments and workspace checks, all before any
    GPU call."""
    from exact_attention_49_gb300 import binding as fa
    need = fa.fa_fp8_workspace_bytes(2, 4, 2, 300, 128)
    off = fa.fa_fp8_workspace_layout(2, 4, 2, 300, 128)
    nb, Np = 3, 304
    assert off[1] >= 2 * 4 * 300 * 128 and off[2] - off[1] >= 2 * 2 * 300 * 128
    assert off[3] - off[2] >= 2 * 2 * 128 * Np and off[4] - off[3] >= 2 * 4 * nb * 4
    assert all(o % 256 == 0 for o in off) and off[7] == need
    assert fa.fa_fp8_workspace_bytes(2, 4, 2, 300, 64) == 0
    assert fa.fa_fp8_workspace_bytes(2, 4, 3, 300, 128) == 0
    P_ = ctypes.c_void_p
    L.fa_fwd_fp8.argtypes = [P_, ctypes.c_size_t, P_, P_] + [ctypes.c_int] * 6 + [ctypes.c_float, P_]
    L.fa_fwd_fp8.restype = ctypes.c_int
    L.fa_fp8_quantize.argtypes = [P_] * 4 + [ctypes.c_int] * 5 + [P_, ctypes.c_size_t, P_]
    L.fa_fp8_quantize.restype = ctypes.c_int
    ws = P((1 << 20) * 256)
    args = dict(B=2, H=4, Hkv=2, N=300, d=128, causal=0, scale=0.125)
    def fwd(**kw):
        a = dict(args, **kw)
        return L.fa_fwd_fp8(kw.get("ws", ws), kw.get("nbytes", need), GOOD, GOOD, a["B"], a["H"], a["Hkv"], a["N"],
                            a["d"], a["causal"], a["scale"], None)
    assert fwd(d=64) == fa.FA_ERR_UNSUPPORTED
    assert fwd(H=3) == fa.FA_ERR_INVALID_ARG
    assert fwd(causal=2) == fa.FA_ERR_INVALID_ARG
    assert fwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(nbytes=need - 1) == fa.FA_ERR_WORKSPACE
    assert fwd(ws=P((1 << 20) * 256 + 16)) == fa.FA_ERR_MISALIGNED
    assert fwd(B=0) == fa.FA_OK and fwd(N=0) == fa.FA_OK
    assert L.fa_fp8_quantize(GOOD, GOOD, GOOD, None, 2, 4, 2, 300, 128, ws, need - 1, None) == fa.FA_ERR_WORKSPACE
    assert L.fa_fp8_quantize(BAD, GOOD, GOOD, None, 2, 4, 2, 300, 128, ws, need, None) == fa.FA_ERR_MISALIGNED
    assert L.fa_fp8_quantize(None, GOOD, GOOD, None, 2, 4, 2, 300, 128, ws, need, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fp8_quantize(GOOD, GOOD, GOOD, None, 2, 4, 2, 300, 64, ws, need, None) == fa.FA_ERR_UNSUPPORTED

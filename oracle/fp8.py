"""FP8 attention reference (fp64 arithmetic on FP8-quantised operands).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Nothing on the product
path may import this module.

The "FlashAttention" wiki note (section FA3, item 3, and the insight on FP8
numerical stability) names two steps that make FP8 attention accurate: block
quantisation (one scale per block instead of one per tensor) and incoherent
processing (multiplying Q and K by a random orthogonal matrix, which leaves
Q K^T unchanged and spreads outlier features over all head dimensions), with
FP8 inputs and higher-precision accumulation; it reports 2.6x lower error than
baseline FP8.  The pages give no formats, block sizes or matrices; the
readings taken here (listed with the design notes):

* format: e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
  infinities, largest finite 448, subnormals k * 2^-9), round to nearest with
  ties to even, saturating at +-448;
* block: 128 consecutive rows of one head of Q, K or V, one scale
  s = amax / 448 per block (s = 1 for an all-zero block);
* incoherent processing: M = H diag(r) / sqrt(d) with H the Sylvester
  Hadamard matrix and r a seeded random sign vector; Q and K are multiplied by
  M along d before quantisation;
* P: quantised as e4m3(448 P) / 448 (P <= 1), O normalised by the sum of the
  quantised P (the weights the PV product used), LSE from the unquantised
  softmax of the quantised scores;
* baseline FP8: one scale per tensor (Q, K, V each), no incoherent processing.

Arithmetic after quantisation is exact fp64 (the role of the fp32 tensor-core
accumulation in the kernel).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9


def e4m3_values() -> np.ndarray:
    """All finite non-negative e4m3 values, ascending (from the bit layout)."""
    vals = set()
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:        # the NaN encoding
                continue
            if e == 0:
                vals.add(m * 2.0 ** -9)   # subnormals: m/8 * 2^(1-7)
            else:
                vals.add((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(sorted(vals))


def _rne(x: np.ndarray) -> np.ndarray:
    return np.round(x)  # numpy rounds halves to even


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even mantissa), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.empty_like(a)
    small = a < E4M3_MIN_NORMAL
    out[small] = _rne(a[small] / E4M3_SUBNORMAL_QUANTUM) * E4M3_SUBNORMAL_QUANTUM
    big = ~small
    e = np.floor(np.log2(a[big]))
    q = 2.0 ** (e - 3)                    # spacing of the binade [2^e, 2^(e+1))
    out[big] = _rne(a[big] / q) * q
    out = np.minimum(out, E4M3_MAX)
    return np.copysign(out, x)


def hadamard_rotation(n: int, seed: int) -> np.ndarray:
    """M = H diag(r) / sqrt(n): Sylvester Hadamard H (n a power of two) and seeded signs r."""
    assert n > 0 and n & (n - 1) == 0
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    r = np.where(np.random.default_rng(seed).random(n) < 0.5, -1.0, 1.0)
    return h * r[None, :] / np.sqrt(n)


def quantize_blocks(x: np.ndarray, block: int = 128) -> np.ndarray:
    """x [..., N, d]: e4m3 with one scale per block of `block` rows (of each leading index)."""
    out = np.empty_like(x, dtype=np.float64)
    N = x.shape[-2]
    for r0 in range(0, N, block):
        blk = x[..., r0:r0 + block, :]
        amax = np.max(np.abs(blk), axis=(-2, -1), keepdims=True)
        s = np.where(amax > 0, amax / E4M3_MAX, 1.0)
        out[..., r0:r0 + block, :] = e4m3_round(blk / s) * s
    return out


def quantize_tensor(x: np.ndarray) -> np.ndarray:
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    s = amax / E4M3_MAX if amax > 0 else 1.0
    return e4m3_round(x / s) * s


def fp8_attention(q, k, v, causal: bool, scale: float, mode: str = "block_incoherent", seed: int = 0,
                  quantize: bool = True):
    """Attention with FP8-quantised Q, K, V and P; q [B,H,N,d], k/v [B,Hkv,N,d] (N equal).

    mode: "block_incoherent" (the pages' method), "block" (no rotation) or "tensor"
    (baseline FP8).  quantize=False skips every rounding (to check that the rotation alone
    leaves the result exact).  Returns (o [B,H,N,d], lse [B,H,N]) in fp64."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    if mode == "block_incoherent":
        m = hadamard_rotation(d, seed)
        q, k = q @ m, k @ m
    if quantize:
        quant = quantize_tensor if mode == "tensor" else quantize_blocks
        q, k, v = quant(q), quant(k), quant(v)
    o = np.zeros((B, H, N, d))
    lse = np.full((B, H, N), -np.inf)
    for b in range(B):
        for h in range(H):
            s = scale * q[b, h] @ k[b, h // g].T
            if causal:
                s = np.where(np.arange(N)[None, :] > np.arange(N)[:, None], -np.inf, s)
            mx = np.max(s, axis=1, keepdims=True)
            e = np.exp(s - mx)
            z = e.sum(axis=1, keepdims=True)
            p = e / z
            lse[b, h] = (mx + np.log(z))[:, 0]
            pq = e4m3_round(E4M3_MAX * p) / E4M3_MAX if quantize else p
            o[b, h] = (pq @ v[b, h // g]) / pq.sum(axis=1, keepdims=True)
    return o, lse


# ---------------------------------------------------------------- the FP8 forward kernel's steps
# A one-pass kernel cannot quantise the normalised P (the normaliser is known only at the end
# of the row).  The readings below are the ones the GB300 FP8 forward implements; they are
# written out here from the method (block quantisation with incoherent processing, wiki FA3
# item 3) and the online softmax (the explainer's online-softmax paragraph), not from the
# kernel, so that the kernel can be checked against them.
#
# Quantisation (per tensor, in fp32, the precision in which the kernel decides each code):
#   * incoherent processing of Q and K: a fast Walsh-Hadamard transform of every row along d in
#     fp32, stages h = 1, 2, 4, ..., d/2, each pair (a, b) = (x_i, x_{i+h}) (bit h of i clear)
#     becoming (a + b, a - b); then each column j multiplied by r_j * fp32(1/sqrt(d)), r_j = +-1
#     the caller's sign vector.  Without rounding this is x @ hadamard_rotation (pinned below).
#   * blocks of 128 rows of one head: amax in fp32, inv = fp32(448 / amax), scale =
#     fp32(amax / 448) (both correctly rounded divisions), code = e4m3(fp32(x * inv)) with
#     round-to-nearest-even and saturation at +-448; an all-zero block has scale 1.
#
# Attention on the codes (key tiles of 128 in order; tile j's V block scale sv_j, the head's
# largest V scale sv_max, f_j = sv_j / sv_max):
#   * S = (q8 . k8^T) * sq_block * sk_j * softmax_scale;
#   * running max m (exact: every growth rescales, so every weight below is at most 1);
#     p = exp(S - m);
#   * P8 = e4m3(448 * f_j * p): the V block scale is folded into the weight so that every tile's
#     product P8 . v8 carries the same factor sv_max / 448;
#   * O_acc += P8 . v8_j,  l_q += sum(P8) / (448 f_j)  (the weights the product used),
#     l += sum(p);
#   * O = O_acc * (sv_max / 448) / l_q,  LSE = m + log(l).

def fwht_fp32(x) -> np.ndarray:
    """Fast Walsh-Hadamard transform along the last axis in float32, in the stage order stated
    above (Sylvester ordering: equals x @ H without rounding)."""
    x = np.array(x, dtype=np.float32)
    n = x.shape[-1]
    assert n > 0 and n & (n - 1) == 0
    lead = x.shape[:-1]
    h = 1
    while h < n:
        y = x.reshape(*lead, n // (2 * h), 2, h)
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        x = y.reshape(*lead, n)
        h *= 2
    return x


def rotate_fp32(x, signs) -> np.ndarray:
    """Incoherent processing in fp32: FWHT of every row, then column j times r_j * fp32(1/sqrt(d))."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    c = np.float32(1.0 / np.sqrt(d))
    col = np.where(np.asarray(signs) > 0, c, -c).astype(np.float32)
    return (fwht_fp32(x) * col).astype(np.float32)


def quantize_fp32(x, block: int = 128):
    """Block quantisation in fp32: returns (codes as e4m3 values in float64, scales float32
    [..., ceil(N/block)]).  x [..., N, d]."""
    x = np.asarray(x, dtype=np.float32)
    N = x.shape[-2]
    nb = (N + block - 1) // block
    codes = np.empty(x.shape, dtype=np.float64)
    scales = np.empty(x.shape[:-2] + (nb,), dtype=np.float32)
    for ib in range(nb):
        blk = x[..., ib * block:(ib + 1) * block, :]
        amax = np.max(np.abs(blk), axis=(-2, -1))
        pos = amax > 0
        safe = np.where(pos, amax, np.float32(1))
        inv = np.where(pos, np.float32(448) / safe, np.float32(1)).astype(np.float32)
        sc = np.where(pos, safe / np.float32(448), np.float32(1)).astype(np.float32)
        y = (blk * inv[..., None, None]).astype(np.float32)
        codes[..., ib * block:(ib + 1) * block, :] = e4m3_round(y.astype(np.float64))
        scales[..., ib] = sc
    return codes, scales


def e4m3_bytes(vals) -> np.ndarray:
    """The e4m3 bit patterns (uint8) of e4m3 values: sign, 4 exponent bits (bias 7), 3 mantissa
    bits; subnormals have exponent field 0."""
    v = np.asarray(vals, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    out = np.zeros(v.shape, dtype=np.uint8)
    sub = a < E4M3_MIN_NORMAL
    m_sub = np.rint(a[sub] / E4M3_SUBNORMAL_QUANTUM).astype(np.int64)
    out[sub] = m_sub.astype(np.uint8)
    nrm = ~sub
    e = np.floor(np.log2(a[nrm])).astype(np.int64)
    m = np.rint((a[nrm] / np.exp2(e) - 1.0) * 8).astype(np.int64)
    out[nrm] = (((e + 7) << 3) | m).astype(np.uint8)
    return out | sign


def fp8_attention_tiled(q8, k8, v8, sq, sk, sv, causal: bool, scale: float, tile: int = 128,
                        quantize_p: bool = True):
    """FP8 attention as the one-pass kernel computes it (see the readings above), in fp64.
    q8 [B,H,N,d], k8/v8 [B,Hkv,N,d] e4m3 code values; sq [B,H,nb], sk/sv [B,Hkv,nb] block
    scales.  Returns (o [B,H,N,d], lse [B,H,N])."""
    q8, k8, v8 = (np.asarray(t, dtype=np.float64) for t in (q8, k8, v8))
    sq, sk, sv = (np.asarray(t, dtype=np.float64) for t in (sq, sk, sv))
    B, H, N, d = q8.shape
    Nk = k8.shape[2]  # a causal mask assumes Nk == N (query i sees keys 0..i)
    g = H // k8.shape[1]
    o = np.zeros((B, H, N, d))
    lse = np.full((B, H, N), -np.inf)
    nt = (Nk + tile - 1) // tile
    for b in range(B):
        for h in range(H):
            kv = h // g
            svmax = np.max(sv[b, kv])
            rows = np.arange(N)
            qs = q8[b, h] * np.repeat(sq[b, h], tile)[:N, None]      # dequantised query rows
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            lq = np.zeros(N)
            acc = np.zeros((N, d))
            for j in range(nt):
                keys = np.arange(j * tile, min(Nk, (j + 1) * tile))
                s = (qs @ k8[b, kv, keys].T) * sk[b, kv, j] * scale
                if causal:
                    s = np.where(keys[None, :] > rows[:, None], -np.inf, s)
                m_new = np.maximum(m, np.max(s, axis=1))
                alpha = np.where(np.isneginf(m_new), 1.0, np.exp(m - m_new))
                acc *= alpha[:, None]
                l *= alpha
                lq *= alpha
                m = m_new
                p = np.where(np.isneginf(s), 0.0, np.exp(s - np.where(np.isneginf(m), 0.0, m)[:, None]))
                f = sv[b, kv, j] / svmax
                pw = e4m3_round(448.0 * f * p) if quantize_p else 448.0 * f * p
                acc += pw @ v8[b, kv, keys]
                lq += pw.sum(axis=1) / (448.0 * f)
                l += p.sum(axis=1)
            ok = lq > 0
            o[b, h] = np.where(ok[:, None], acc * (svmax / 448.0) / np.where(ok, lq, 1.0)[:, None], 0.0)
            lse[b, h] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse

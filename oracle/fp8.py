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

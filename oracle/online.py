"""A separate CPU online-softmax forward, tile by tile, in fp64 (numpy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows "FlashAttention：GPUハードウェア階層を考慮した高速・省メモリな厳密
アテンション" (singularity-lens.com): the tiling paragraph (split the inputs
into blocks, compute local scores for one block at a time) and the
online-softmax paragraph (keep the running maximum and the running sum of
exponentials; when a later block brings a larger maximum, correct the earlier
partial sums by the difference; the result equals standard attention).  The
"FlashAttention" wiki note, section 定義 item (1), states the same.

Written independently of the C oracle; the pins check that both agree to
about 1e-12, which is the exactness claim of the tiled method.
"""
from __future__ import annotations

import numpy as np


def fwd(q, k, v, causal: bool, scale: float, tile: int):
    """q: [B,H,N,d], k/v: [B,Hkv,Nk,d] -> (o, lse), key blocks of ``tile`` rows."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, H, N, d = q.shape
    _, Hkv, Nk, _ = k.shape
    grp = H // Hkv
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            g = h // grp
            m = np.full(N, -np.inf)      # running max per query row
            l = np.zeros(N)              # running sum of exp(s - m)
            acc = np.zeros((N, d))       # running unnormalised output
            for j0 in range(0, Nk, tile):
                kb = k[b, g, j0:j0 + tile]
                vb = v[b, g, j0:j0 + tile]
                s = scale * (q[b, h] @ kb.T)                       # local scores
                if causal:
                    cols = np.arange(j0, j0 + kb.shape[0])
                    s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
                m_new = np.maximum(m, s.max(axis=1))
                # rows that have seen no visible key yet keep m = -inf
                seen = m_new > -np.inf
                corr = np.where(seen, np.exp(np.where(seen, m - m_new, 0.0)), 0.0)
                p = np.where(seen[:, None], np.exp(s - np.where(seen, m_new, 0.0)[:, None]), 0.0)
                l = l * corr + p.sum(axis=1)
                acc = acc * corr[:, None] + p @ vb
                m = m_new
            with np.errstate(divide="ignore", invalid="ignore"):
                o[b, h] = np.where(l[:, None] > 0, acc / l[:, None], 0.0)
                lse[b, h] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse

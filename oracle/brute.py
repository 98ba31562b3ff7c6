"""Pure-Python brute-force attention for tiny shapes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

A second, independent transcription of standard (materialising) attention
("FlashAttention" wiki note, section 定義) with explicit loops over Python
floats, used to pin the C oracle on shapes with N <= 8 and d <= 4.  The
backward is the textbook gradient of sum(O * dO), written with the full
Jacobian of the softmax rather than the dS = P(dP - D) shortcut, so that a
mistake in that shortcut would show up as a disagreement:

    dS_ij = sum_j' dP_ij' * P_ij' * (delta_jj' - P_ij)

Inputs are nested lists ``x[b][h][n][c]``.  For the causal mask query row i
sits at position i + qoff (bottom-right alignment for Nq != Nk: qoff = Nk - Nq).
"""
from __future__ import annotations

import math


def _shape(x):
    return len(x), len(x[0]), len(x[0][0]), len(x[0][0][0])


def fwd(q, k, v, causal, scale, qoff=0):
    B, H, N, d = _shape(q)
    _, Hkv, Nk, _ = _shape(k)
    grp = H // Hkv
    o = [[[[0.0] * d for _ in range(N)] for _ in range(H)] for _ in range(B)]
    lse = [[[0.0] * N for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            g = h // grp
            for i in range(N):
                s = []
                for j in range(Nk):
                    if causal and j > i + qoff:
                        s.append(-math.inf)
                    else:
                        s.append(scale * sum(q[b][h][i][c] * k[b][g][j][c] for c in range(d)))
                m = max(s) if s else -math.inf
                if m == -math.inf:  # the row sees no key: O = 0, LSE = -inf
                    lse[b][h][i] = -math.inf
                    continue
                e = [math.exp(x - m) if x != -math.inf else 0.0 for x in s]
                z = sum(e)
                for c in range(d):
                    o[b][h][i][c] = sum(e[j] / z * v[b][g][j][c] for j in range(Nk))
                lse[b][h][i] = m + math.log(z)
    return o, lse


def bwd(q, k, v, do, causal, scale, qoff=0):
    B, H, N, d = _shape(q)
    _, Hkv, Nk, _ = _shape(k)
    grp = H // Hkv
    dq = [[[[0.0] * d for _ in range(N)] for _ in range(H)] for _ in range(B)]
    dk = [[[[0.0] * d for _ in range(Nk)] for _ in range(Hkv)] for _ in range(B)]
    dv = [[[[0.0] * d for _ in range(Nk)] for _ in range(Hkv)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            g = h // grp
            for i in range(N):
                s = []
                for j in range(Nk):
                    if causal and j > i + qoff:
                        s.append(-math.inf)
                    else:
                        s.append(scale * sum(q[b][h][i][c] * k[b][g][j][c] for c in range(d)))
                m = max(s) if s else -math.inf
                if m == -math.inf:  # the row sees no key: no gradient
                    continue
                e = [math.exp(x - m) if x != -math.inf else 0.0 for x in s]
                z = sum(e)
                p = [x / z for x in e]
                # O_i = sum_j p_j v_j  ->  dL/dp_j = <dO_i, v_j>,  dL/dv_j += p_j dO_i
                dp = [sum(do[b][h][i][c] * v[b][g][j][c] for c in range(d)) for j in range(Nk)]
                for j in range(Nk):
                    for c in range(d):
                        dv[b][g][j][c] += p[j] * do[b][h][i][c]
                # softmax Jacobian: dS_j = sum_j' dp_j' * dP_j'/dS_j = sum_j' dp_j' p_j' (delta - p_j)
                ds = []
                for j in range(Nk):
                    acc = 0.0
                    for jj in range(Nk):
                        acc += dp[jj] * p[jj] * ((1.0 if jj == j else 0.0) - p[j])
                    ds.append(acc)
                # S_ij = scale * <q_i, k_j>
                for j in range(Nk):
                    for c in range(d):
                        dq[b][h][i][c] += scale * ds[j] * k[b][g][j][c]
                        dk[b][g][j][c] += scale * ds[j] * q[b][h][i][c]
    return dq, dk, dv

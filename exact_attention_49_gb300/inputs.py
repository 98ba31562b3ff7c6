"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so that both the CUDA path and the CPU oracle can take
the very same bf16 tensors from it without sharing any computation.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws Q, K, V and dO, in that order, as fp32 N(0, 1) and rounds them
to bf16 (round-to-nearest-even).  An optional power-of-two multiplier on Q and
K (applied after rounding, so it is exact) spreads the scores to stress the
running-max rescale.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    causal: bool
    qk_mult: float = 1.0
    seed: int = 0
    backward: bool = True

    @property
    def scale(self) -> float:
        return self.d ** -0.5


# The five workloads of the hot path (shapes only).
WORKLOADS = {
    "C1": Workload("C1 B1 H2 N128 d64 non-causal", 1, 2, 2, 128, 64, False, seed=0),
    "C2": Workload("C2 B8 H16 N512 d64 non-causal", 8, 16, 16, 512, 64, False, seed=1),
    "C3": Workload("C3 B4 H16 N8192 d128 causal", 4, 16, 16, 8192, 128, True, seed=2),
    "C3b": Workload("C3b B4 H16 N8192 d128 causal, Q and K x4", 4, 16, 16, 8192, 128, True,
                    qk_mult=4.0, seed=3),
    "C4": Workload("C4 GQA B2 Hq32 Hkv8 N16384 d128 causal", 2, 32, 8, 16384, 128, True, seed=4),
    # head dimension 256, forward and backward (the wider-head shape of the general-shape row)
    "HD256": Workload("HD256 B1 H16 N8192 d256 causal", 1, 16, 16, 8192, 256, True, seed=6),
}


def long_context(N: int, d: int) -> Workload:
    """One point of the long-context forward sweep (B=1, H=16, causal)."""
    return Workload("C5 B1 H16 N%d d%d causal fwd" % (N, d), 1, 16, 16, N, d, True,
                    seed=5, backward=False)


def make_inputs(B: int, H: int, Hkv: int, N: int, d: int, seed: int, qk_mult: float = 1.0, Nk: int | None = None):
    """Return bf16 CPU tensors (q, k, v, do): q/do [B,H,N,d], k/v [B,Hkv,Nk,d] (Nk = N by default)."""
    Nk = N if Nk is None else Nk
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Nk, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    if qk_mult != 1.0:
        q = q * qk_mult
        k = k * qk_mult
    return q, k, v, do


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.Hkv, w.N, w.d, w.seed, w.qk_mult)

"""Seeded synthetic KDA prefill inputs.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no normalisation, no decay, no recurrence).  Both the
CUDA path's tests and benchmark and the CPU oracle's tests take their inputs
from here, so the two sides see identical bits.

Distributions follow the workloads of the pages: T = 8,192 tokens at 96 and 6
heads ("FlashKDA column split", section 4), head dimension 128 and BF16 q, k,
v, beta and state (flashinfer kda_prefill, "Optimized Blackwell prefill
subset"), log-decay g in (-5, 0) ("K3's KDA precision problem", introduction),
small batch x head with long sequences ("CAKE KDA prefill", B200 smoke
results) and packed variable-length batches with int64 offsets (flashinfer
kda_prefill, "Packed scheduling").

Draw order (CPU ``torch.Generator`` seeded once per call): sequence lengths
(packed workloads only), q, k, v, g, beta, initial state.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, distributions and seed."""

    name: str
    B: int
    H: int
    T: int                                # tokens per sequence (fixed) or 0 (packed)
    seed: int
    g_low: float = -5.0
    g_high: float = 0.0
    beta_std: float = 1.0                 # beta = sigmoid(N(0, beta_std^2))
    init_std: Optional[float] = None      # None: no initial state (zeros)
    packed_n: int = 0                     # > 0: packed layout with this many sequences
    len_low: int = 512
    len_high: int = 8192
    len_multiple: int = 16

    @property
    def packed(self) -> bool:
        return self.packed_n > 0


WORKLOADS = {
    # 16 chunks of 16 tokens, one head.
    "t256_h1": Workload("B=1,H=1,T=256,d=128", B=1, H=1, T=256, seed=0),
    # Small-head tensor-parallel shard at 8,192 tokens.
    "t8192_h6": Workload("B=1,H=6,T=8192,d=128", B=1, H=6, T=8192, seed=1, init_std=0.02),
    # Full head count at 8,192 tokens.
    "t8192_h96": Workload("B=1,H=96,T=8192,d=128", B=1, H=96, T=8192, seed=2),
    # Full head count, a batch of two sequences: more (sequence, head) chains
    # than the GPU has SMs (a measurement case beside the five above).
    "t8192_h96_b2": Workload("B=2,H=96,T=8192,d=128", B=2, H=96, T=8192, seed=5),
    # Packed: 8 sequences, lengths uniform in [512, 8192] rounded to multiples of 16.
    "varlen8_h12": Workload("packed B=1,H=12,d=128,N=8", B=1, H=12, T=0, seed=3,
                            init_std=0.02, packed_n=8),
    # One long sequence: 4,096 dependent chunks.
    "t65536_h1": Workload("B=1,H=1,T=65536,d=128", B=1, H=1, T=65536, seed=4,
                          g_low=-5.0, g_high=-0.01, beta_std=2.0, init_std=0.02),
}


def draw_lengths(gen: torch.Generator, n: int, low: int, high: int, multiple: int):
    raw = torch.randint(low, high + 1, (n,), generator=gen, dtype=torch.int64)
    if multiple > 1:
        raw = ((raw + multiple // 2) // multiple) * multiple
    return [int(x) for x in raw]


def cu_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int64)


def make_inputs(B: int, T: int, H: int, seed: int, *, dk: int = HEAD_DIM,
                dv: int = HEAD_DIM, g_low: float = -5.0, g_high: float = 0.0,
                beta_std: float = 1.0, init_std: Optional[float] = None,
                lengths: Optional[Sequence[int]] = None,
                gen: Optional[torch.Generator] = None) -> dict:
    """Draw one input set on the CPU.

    Fixed layout: ``B`` sequences of ``T`` tokens.  Packed layout: pass
    ``lengths`` (then ``B`` and ``T`` are ignored; tensors are ``[1, sum, H, d]``).
    Returns a dict with q, k, v (bf16), g (fp32), beta (bf16), init_state (bf16
    ``[N, H, dv, dk]`` or None), cu_seqlens (int64 or None) and N.
    """
    if gen is None:
        gen = torch.Generator(device="cpu")
        gen.manual_seed(seed)
    if lengths is not None:
        cu = cu_from_lengths(lengths)
        N, Bt, Tt = len(lengths), 1, int(cu[-1])
    else:
        cu = None
        N, Bt, Tt = B, B, T
    q = torch.randn((Bt, Tt, H, dk), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((Bt, Tt, H, dk), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((Bt, Tt, H, dv), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    g = torch.rand((Bt, Tt, H, dk), generator=gen, dtype=torch.float32)
    g = g * (g_high - g_low) + g_low
    beta = torch.sigmoid(beta_std * torch.randn((Bt, Tt, H), generator=gen,
                                                dtype=torch.float32)).to(torch.bfloat16)
    init = None
    if init_std is not None:
        init = (init_std * torch.randn((N, H, dv, dk), generator=gen,
                                       dtype=torch.float32)).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "init_state": init,
            "cu_seqlens": cu, "N": N}


def make_workload(key_or_workload) -> dict:
    """Inputs of one named workload (see ``WORKLOADS``)."""
    w = WORKLOADS[key_or_workload] if isinstance(key_or_workload, str) else key_or_workload
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    lengths = None
    if w.packed:
        lengths = draw_lengths(gen, w.packed_n, w.len_low, w.len_high, w.len_multiple)
    out = make_inputs(w.B, w.T, w.H, w.seed, g_low=w.g_low, g_high=w.g_high,
                      beta_std=w.beta_std, init_std=w.init_std, lengths=lengths, gen=gen)
    out["workload"] = w
    return out


# --- Stress families of "K3's KDA precision problem" (section "Numerical
# experiments on H200"), with the scalar per-token decay broadcast over the
# key channels. -------------------------------------------------------------

def stress_inputs(family: str, T: int, H: int, seed: int, dk: int = HEAD_DIM,
                  dv: int = HEAD_DIM) -> dict:
    """``floor_e-5``: g = -5 everywhere; ``weak_decay_correlated``: every key
    the same direction, g = -0.01, beta = 0.5; ``model_like``: per-token
    g = -5 sigmoid(N(0,1)) and beta = sigmoid(N(0,1))."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = torch.randn((1, T, H, dk), generator=gen, dtype=torch.float32)
    v = torch.randn((1, T, H, dv), generator=gen, dtype=torch.float32)
    if family == "weak_decay_correlated":
        key = torch.randn((1, 1, H, dk), generator=gen, dtype=torch.float32)
        k = key.expand(1, T, H, dk).contiguous()
        g = torch.full((1, T, H, dk), -0.01, dtype=torch.float32)
        beta = torch.full((1, T, H), 0.5, dtype=torch.float32)
    else:
        k = torch.randn((1, T, H, dk), generator=gen, dtype=torch.float32)
        if family == "floor_e-5":
            g = torch.full((1, T, H, dk), -5.0, dtype=torch.float32)
            beta = torch.sigmoid(torch.randn((1, T, H), generator=gen, dtype=torch.float32))
        elif family == "model_like":
            gate = torch.randn((1, T, H, 1), generator=gen, dtype=torch.float32)
            g = (-5.0 * torch.sigmoid(gate)).expand(1, T, H, dk).contiguous()
            beta = torch.sigmoid(torch.randn((1, T, H), generator=gen, dtype=torch.float32))
        else:
            raise ValueError("unknown stress family %r" % family)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16),
            "v": v.to(torch.bfloat16), "g": g, "beta": beta.to(torch.bfloat16),
            "init_state": None, "cu_seqlens": None, "N": 1}

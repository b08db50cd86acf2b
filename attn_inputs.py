"""Seeded synthetic inputs and named workloads for the attention forward.

This module is shared by the oracle tests, the GPU parity tests, the smoke
check and the benchmark.  It holds no attention arithmetic: only the random
input recipe and the shapes of the workloads.

Input recipe: Q, K and V are ``[B, H, L, D]``, each element drawn i.i.d. from a
normal distribution as fp32 by one CPU ``torch.Generator`` seeded with ``seed``
(drawn in the order q, k, v), multiplied by ``std`` and rounded to the
workload dtype (round to nearest even).  Seed 42 and N(0, 1) follow the
self-check of the "TLX Block Attention" page; seed 20, N(0, 0.5) and
``sm_scale = 0.5`` follow the test matrix of the "Fused Attention" page.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DENSE, CAUSAL, BLOCK_DIAG = 0, 1, 2
MASK_NAMES = {DENSE: "dense", CAUSAL: "causal", BLOCK_DIAG: "block_diag"}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    D: int
    mask: int
    dtype: torch.dtype
    sm_scale: float
    block_size: int = 0
    seed: int = 42
    std: float = 1.0
    note: str = field(default="", compare=False)

    def describe(self) -> dict:
        return {"workload": self.name, "batch": self.B, "heads": self.H,
                "seq_len": self.L, "head_dim": self.D, "mask": MASK_NAMES[self.mask],
                "block_size": self.block_size or None,
                "dtype": "fp16" if self.dtype == torch.float16 else "bf16",
                "sm_scale": self.sm_scale, "seed": self.seed, "std": self.std}


# The five workloads the attention forward is measured and checked on.
WORKLOADS = {
    w.name: w for w in [
        Workload("blockdiag_b1h2n256d128_bs64_f16", 1, 2, 256, 128, BLOCK_DIAG,
                 torch.float16, 1.0 / math.sqrt(128), 64,
                 note="self-check shape of the TLX Block Attention page"),
        Workload("dense_b4h16l1024d64_f16", 4, 16, 1024, 64, DENSE,
                 torch.float16, 1.0 / 8.0),
        Workload("causal_b2h32l4096d128_bf16", 2, 32, 4096, 128, CAUSAL,
                 torch.bfloat16, 1.0 / math.sqrt(128)),
        Workload("blockdiag_b8h16n8192d128_bs64_f16", 8, 16, 8192, 128, BLOCK_DIAG,
                 torch.float16, 1.0 / math.sqrt(128), 64),
        Workload("blockdiag_b8h16n8192d128_bs128_f16", 8, 16, 8192, 128, BLOCK_DIAG,
                 torch.float16, 1.0 / math.sqrt(128), 128),
        Workload("causal_b1h32l32768d128_bf16", 1, 32, 32768, 128, CAUSAL,
                 torch.bfloat16, 1.0 / math.sqrt(128)),
        Workload("dense_b1h16l16384d256_bf16", 1, 16, 16384, 256, DENSE,
                 torch.bfloat16, 1.0 / 16.0),
    ]
}

# The headline workload of the benchmark.
HEADLINE = "dense_b4h16l1024d64_f16"

# Shapes of the test matrix on the "Fused Attention" page (Z, H, N_CTX, HEAD_DIM,
# dtype); there they are all non-causal with sm_scale 0.5 and N(0, 0.5) inputs.
PAGE_TEST_MATRIX = [
    (1, 1, 128, 128, torch.float16),
    (1, 1, 128, 128, torch.bfloat16),
    (1, 2, 256, 256, torch.bfloat16),
    (2, 2, 128, 256, torch.float16),
    (4, 32, 64, 64, torch.float16),
    (4, 32, 1024, 64, torch.bfloat16),
    (4, 32, 4096, 64, torch.float16),
]


def make_qkv(B: int, H: int, L: int, D: int, dtype: torch.dtype, seed: int = 42,
             std: float = 1.0):
    """Seeded CPU Q, K, V of shape [B, H, L, D] in ``dtype`` (see module doc)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = []
    for _ in range(3):
        t = torch.randn((B, H, L, D), generator=g, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        out.append(t.to(dtype))
    return tuple(out)


def make_qkv_far_below_zero(B: int, H: int, L: int, D: int, dtype: torch.dtype, sign: int = 1,
                            seed: int = 5):
    """Seeded Q, K, V and sm_scale with every scaled score near -200: head-dim 0
    carries q0 = -sign*a and k0 = a with a^2 / sqrt(D) = 200, sm_scale is
    sign / sqrt(D), and the other dims stay N(0, 1), which spreads the scores a
    few units around -200.  With sign = -1 the scale is negative and the raw
    scores large and positive."""
    q, k, v = make_qkv(B, H, L, D, dtype, seed=seed)
    a = math.sqrt(200.0 * math.sqrt(D))
    q[..., 0] = -sign * a
    k[..., 0] = a
    return q, k, v, sign / math.sqrt(D)


def make_workload_inputs(w: Workload):
    return make_qkv(w.B, w.H, w.L, w.D, w.dtype, w.seed, w.std)



def make_vt_e5m2(v: torch.Tensor) -> torch.Tensor:
    """The FP8 P.V variant's V input: ``v`` ([B,H,L,D], fp16/bf16) rounded to
    float8 e5m2 (torch's conversion, round to nearest even) and transposed to
    ``[B,H,D,L]`` (keys innermost), contiguous."""
    return v.float().to(torch.float8_e5m2).transpose(-1, -2).contiguous()

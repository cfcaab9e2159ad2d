"""Seeded synthetic inputs for kernelized (linear) attention.

This module holds the workload shapes and the seeded input generators shared
by the tests, the smoke check and the benchmark.  It holds none of the
method's arithmetic: it only draws random numbers, scales them, casts them
and lays them out.

Recipe: q, k, v ~ iid N(0, 1) drawn with ``torch.randn`` from a CPU
``torch.Generator`` seeded with the workload's seed, in fp32, in the order
q, k, v; scaled by 1/sqrt(D) for the bf16 workloads (unscaled for the fp32
one); then cast to the workload dtype.  The PRF projection W [m, D] is iid
N(0, 1) fp32 from its own seed.  Decode inputs for step t come from seed
``DECODE_SEED + t``.  The output cotangent of a backward pass, dout
[B,H,N,Dv], is iid N(0, 1) from seed ``seed + DOUT_SEED_OFFSET``, cast to the
workload dtype.  The query token of prefix attention, q [B,H,D], is iid
N(0, 1) / sqrt(D) (unscaled for fp32 workloads) from seed
``seed + PREFIX_Q_SEED_OFFSET``.  The relative-position log-weights of
kernelized attention with RPE, b [H, 2N-1] fp32, are iid N(0, 0.5^2) from
seed ``seed + RPE_SEED_OFFSET``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    Dv: int
    causal: bool = True
    feature: str = "elu1"     # "elu1" | "prf"
    m: int = 0                # PRF feature count
    dtype: str = "bf16"       # "f32" | "bf16"
    scaled: bool = True       # divide by sqrt(D)
    seed: int = 1000

    @property
    def phi_dim(self) -> int:
        return self.m if self.feature == "prf" else self.D

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the method's benchmark table (sizes as named there).
TINY_F32 = Workload("causal_B1_H1_N64_D16_f32", 1, 1, 64, 16, 16, dtype="f32",
                    scaled=False, seed=1001)
IMAGE_3072 = Workload("causal_B4_H8_N3072_D64_bf16", 4, 8, 3072, 64, 64, seed=1002)
NONCAUSAL_4096 = Workload("noncausal_B8_H8_N4096_D64_bf16", 8, 8, 4096, 64, 64,
                          causal=False, seed=1003)
LONG_65536 = Workload("causal_B1_H16_N65536_D128_bf16", 1, 16, 65536, 128, 128, seed=1004)
PRF_16384 = Workload("causal_prf256_B2_H8_N16384_D64_bf16", 2, 8, 16384, 64, 64,
                     feature="prf", m=256, seed=1005)

WORKLOADS = {w.name: w for w in (TINY_F32, IMAGE_3072, NONCAUSAL_4096, LONG_65536, PRF_16384)}

# Decode from the long workload's final state, replicated into 64 batch rows.
DECODE_B = 64
DECODE_H = 16
DECODE_D = 128
DECODE_STEPS = 4096
DECODE_SEED = 4000
W_SEED = 5000
DOUT_SEED_OFFSET = 7000
PREFIX_Q_SEED_OFFSET = 8000
RPE_SEED_OFFSET = 9000

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _randn(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32)


def make_qkv(w: Workload, device="cpu"):
    """q, k [B,H,N,D] and v [B,H,N,Dv] in the workload dtype on ``device``."""
    gen = torch.Generator().manual_seed(w.seed)
    scale = 1.0 / math.sqrt(w.D) if w.scaled else 1.0
    dt = TORCH_DTYPE[w.dtype]
    out = []
    for shape in ((w.B, w.H, w.N, w.D), (w.B, w.H, w.N, w.D), (w.B, w.H, w.N, w.Dv)):
        x = _randn(shape, gen)
        if scale != 1.0:
            x.mul_(scale)
        out.append(x.to(dt).to(device).contiguous())
    return tuple(out)


def make_dout(w: Workload, device="cpu"):
    """Output cotangent dout [B,H,N,Dv] for a backward pass, iid N(0, 1)."""
    gen = torch.Generator().manual_seed(w.seed + DOUT_SEED_OFFSET)
    x = _randn((w.B, w.H, w.N, w.Dv), gen)
    return x.to(TORCH_DTYPE[w.dtype]).to(device).contiguous()


def make_prefix_q(w: Workload, device="cpu"):
    """Query token q [B,H,D] of prefix attention (one per head)."""
    gen = torch.Generator().manual_seed(w.seed + PREFIX_Q_SEED_OFFSET)
    x = _randn((w.B, w.H, w.D), gen)
    if w.scaled:
        x.mul_(1.0 / math.sqrt(w.D))
    return x.to(TORCH_DTYPE[w.dtype]).to(device).contiguous()


def make_rpe_bias(w: Workload, device="cpu"):
    """Relative-position log-weights b [H, 2N-1] fp32 (index t + N - 1)."""
    gen = torch.Generator().manual_seed(w.seed + RPE_SEED_OFFSET)
    return _randn((w.H, 2 * w.N - 1), gen).mul_(0.5).to(device).contiguous()


def make_W(m: int, D: int, seed: int = W_SEED, device="cpu"):
    """PRF projection W [m, D], iid N(0, 1), fp32."""
    gen = torch.Generator().manual_seed(seed)
    return _randn((m, D), gen).to(device).contiguous()


def make_decode_qkv(t: int, B=DECODE_B, H=DECODE_H, D=DECODE_D, Dv=DECODE_D,
                    dtype="bf16", device="cpu"):
    """Step-t decode inputs q, k [B,H,D], v [B,H,Dv], scaled by 1/sqrt(D)."""
    gen = torch.Generator().manual_seed(DECODE_SEED + t)
    dt = TORCH_DTYPE[dtype]
    scale = 1.0 / math.sqrt(D)
    q = _randn((B, H, D), gen).mul_(scale)
    k = _randn((B, H, D), gen).mul_(scale)
    v = _randn((B, H, Dv), gen).mul_(scale)
    return tuple(x.to(dt).to(device).contiguous() for x in (q, k, v))


def small(name="small", B=1, H=2, N=200, D=64, Dv=64, causal=True, feature="elu1", m=0,
          dtype="bf16", scaled=True, seed=7):
    """An ad-hoc small workload for parity and edge-case tests."""
    return Workload(name, B, H, N, D, Dv, causal, feature, m, dtype, scaled, seed)

"""Seeded synthetic inputs for the EXL3 trellis linear / MoE / int8-gather path.

This module holds random-number recipes only (no step of the method): it is
shared by the tests, the benchmark and the smoke check, and both the CPU oracle
and the CUDA path consume what it returns.  Everything is numpy on the host;
callers copy to the device themselves.

Floating-point values are returned as raw bit patterns (uint16) in the format
the method stores them in: bf16 for activations, fp16 for scale vectors.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Store float32 samples as bf16 (round to nearest even) bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def signed_uniform_f16(g: np.random.Generator, n: int, lo=0.5, hi=1.5) -> np.ndarray:
    """fp16 bits of random sign * U(lo, hi) (the scale-vector recipe)."""
    v = g.uniform(lo, hi, n) * np.where(g.random(n) < 0.5, -1.0, 1.0)
    return v.astype(np.float16).view(np.uint16)


def uniform_code(g: np.random.Generator, shape) -> np.ndarray:
    """Uniform random int16 trellis code words."""
    return g.integers(-32768, 32768, size=shape, dtype=np.int16)


def normal_bf16(g: np.random.Generator, M: int, N: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    """bf16 bits of x ~ N(0,1) [M][N]; optionally a seeded subset of channels
    (round(outlier_frac * N) of them) scaled by outlier_scale."""
    x = g.standard_normal((M, N), dtype=np.float32)
    if outlier_frac > 0:
        n_out = int(round(outlier_frac * N))
        ch = g.choice(N, size=n_out, replace=False)
        x[:, ch] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


@dataclass
class Shard:
    """One EXL3 tensor: code [IC/16][OC/16][16K] plus its four scale vectors."""
    code: np.ndarray
    K: int
    s_in: np.ndarray
    rin: np.ndarray
    rout: np.ndarray
    s_out: np.ndarray

    @property
    def IC(self):
        return self.code.shape[0] * 16

    @property
    def OC(self):
        return self.code.shape[1] * 16


def make_shard(g: np.random.Generator, IC: int, OC: int, K: int) -> Shard:
    code = uniform_code(g, (IC // 16, OC // 16, 16 * K))
    return Shard(code=code, K=K,
                 s_in=signed_uniform_f16(g, IC), rin=signed_uniform_f16(g, IC),
                 rout=signed_uniform_f16(g, OC), s_out=signed_uniform_f16(g, OC))


# ------------------------------------------------------------------ workloads
def linear_case(seed: int, M: int, IC: int, OC: int, K: int, outlier_frac: float = 0.0):
    """x bf16 [M][IC] and one shard."""
    g = rng(seed)
    shard = make_shard(g, IC, OC, K)
    x = normal_bf16(g, M, IC, outlier_frac)
    return x, shard


def single_linear(seed: int = 0):
    """Single EXL3 linear: IC = OC = 512, K = 2, M = 4."""
    return linear_case(seed, 4, 512, 512, 2)


def gate_up(seed: int = 1, M: int = 8, IC: int = 5120, OC: int = 17408, Ks=(2, 3)):
    """Merged gate (K=2) / up (K=3) shards written into one out[M][2*OC]."""
    g = rng(seed)
    shards = [make_shard(g, IC, OC, K) for K in Ks]
    x = normal_bf16(g, M, IC)
    return x, shards


def prefill(seed: int = 2, M: int = 8192, IC: int = 5120, OC: int = 17408, K: int = 2):
    """Prefill-shaped linear: x with 1 % of channels scaled x20."""
    return linear_case(seed + 10 * K, M, IC, OC, K, outlier_frac=0.01)


LAYER_PROJ = (("qkv", 5120, 7168, 4), ("o", 5120, 5120, 3), ("gate", 5120, 17408, 2),
              ("up", 5120, 17408, 3), ("down", 17408, 5120, 3))


def decoder_layer(seed: int = 4, M: int = 8):
    """The five projections of one hidden-5120 decoder layer, each with its own x."""
    g = rng(seed)
    out = []
    for name, IC, OC, K in LAYER_PROJ:
        out.append((name, normal_bf16(g, M, IC), make_shard(g, IC, OC, K)))
    return out


def embedding(seed: int = 5, V: int = 248320, H: int = 5120, N: int = 8192):
    """int8 table [V][H] uniform in [-127, 127], fp16 scales U(1e-3, 1e-2), N ids."""
    g = rng(seed)
    q = g.integers(-127, 128, size=(V, H), dtype=np.int8)
    s = g.uniform(1e-3, 1e-2, V).astype(np.float16).view(np.uint16)
    ids = g.integers(0, V, size=N, dtype=np.int32)
    return q, s, ids


# ------------------------------------------------------------------ MoE bank
def moe_bank(seed: int = 3, E: int = 128, H: int = 2048, I: int = 768, Ks=(2, 3, 4),
             distinct_down_k: bool = False):
    """A flat EXL3 expert bank with per-expert K drawn from Ks and K-sorted slots.

    Slots are ordered by (k_gu, k_d) ascending, ties by logical expert id.
    Returns a dict: w13, w2 (flat int16), off_w1/off_w3/off_w2 (int64 word
    offsets per slot), perm (int32 logical -> slot), k_gu/k_d (int32 per slot),
    w13_suh [E,2,H], w13_svh [E,2,I], w2_suh [E,I], w2_svh [E,H] (fp16 bits,
    per slot).
    """
    g = rng(seed)
    k_gu_l = g.choice(np.asarray(Ks), size=E).astype(np.int32)
    k_d_l = g.choice(np.asarray(Ks), size=E).astype(np.int32) if distinct_down_k else k_gu_l.copy()
    order = sorted(range(E), key=lambda e: (int(k_gu_l[e]), int(k_d_l[e]), e))
    perm = np.empty(E, np.int32)
    for p, e in enumerate(order):
        perm[e] = p
    k_gu = np.array([k_gu_l[e] for e in order], np.int32)
    k_d = np.array([k_d_l[e] for e in order], np.int32)
    words1 = H * I * k_gu.astype(np.int64) // 16
    words2 = I * H * k_d.astype(np.int64) // 16
    off_w1 = np.zeros(E, np.int64)
    off_w3 = np.zeros(E, np.int64)
    off_w2 = np.zeros(E, np.int64)
    acc13 = acc2 = 0
    for p in range(E):
        off_w1[p] = acc13
        off_w3[p] = acc13 + words1[p]
        acc13 += 2 * words1[p]
        off_w2[p] = acc2
        acc2 += words2[p]
    return dict(
        w13=uniform_code(g, (acc13,)), w2=uniform_code(g, (acc2,)),
        off_w1=off_w1, off_w3=off_w3, off_w2=off_w2, perm=perm, k_gu=k_gu, k_d=k_d,
        w13_suh=signed_uniform_f16(g, E * 2 * H).reshape(E, 2, H),
        w13_svh=signed_uniform_f16(g, E * 2 * I).reshape(E, 2, I),
        w2_suh=signed_uniform_f16(g, E * I).reshape(E, I),
        w2_svh=signed_uniform_f16(g, E * H).reshape(E, H),
    )


def moe_tokens(seed: int, T: int, H: int = 2048, E: int = 128):
    """x bf16 [T][H] ~ N(0,1) and router logits fp32 [T][E] ~ N(0,1)."""
    g = rng(seed)
    x = normal_bf16(g, T, H)
    logits = g.standard_normal((T, E), dtype=np.float32)
    return x, logits

"""Seeded synthetic inputs for log-linear attention (shared by tests, bench and oracle runs).

This module draws random numbers and rounds them to the storage types; it
holds none of the operator's arithmetic. Both the CUDA path and the CPU
oracle consume exactly the arrays made here: the GPU gets the bf16 bit
patterns, the oracle gets the same values widened to fp64.

Distributions follow the workload shapes of the benchmark configurations:
q, k ~ N(0, 1/dk) (or unit-norm rows), v ~ N(0, 1), log_a = -softplus(N(mu, 1)),
lambda = softplus(N(0, 1)) for every Fenwick level. The Gated DeltaNet variant
adds the delta-rule strength beta = sigmoid(N(0, 1)) per token and always uses
unit-norm key rows (the delta rule's transition I - beta k k^T is then a
contraction for beta in [0, 1]).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def num_levels(T: int) -> int:
    """Fenwick level count for length T: bit length of T-1, plus one (T >= 1)."""
    return int(T - 1).bit_length() + 1 if T > 1 else 1


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32, exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    chunk: int
    dtype: str  # "f32" or "bf16": storage type of q, k, v and out
    qk_unit_rows: bool = False  # L2-normalise q and k rows instead of N(0, 1/dk)
    log_a_mu: float = 0.0  # log_a = -softplus(N(log_a_mu, 1))

    @property
    def L(self) -> int:
        return num_levels(self.T)

    @property
    def tokens(self) -> int:
        return self.B * self.T


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    H: int
    dk: int
    dv: int
    t_max: int  # positions drawn uniformly from [1, t_max)
    steps: int
    Lmax: int = 18
    dtype: str = "bf16"


PREFILL_CONFIGS = {
    "oracle-scale": PrefillConfig("oracle-scale", 1, 1, 64, 16, 16, 16, "f32"),
    "small": PrefillConfig("small", 2, 4, 2048, 64, 64, 64, "bf16"),
    "headline": PrefillConfig("headline", 4, 16, 8192, 128, 64, 64, "bf16", qk_unit_rows=True, log_a_mu=-2.0),
    "long": PrefillConfig("long", 1, 16, 65536, 128, 64, 128, "bf16", qk_unit_rows=True, log_a_mu=-2.0),
}

DECODE_CONFIG = DecodeConfig("decode", batch=64, H=16, dk=128, dv=64, t_max=65536, steps=1000)

# Log-linear Gated DeltaNet workloads: the Mamba-2 prefill shapes with unit-norm q and k rows.
GDN_CONFIGS = {
    "gdn-oracle-scale": PrefillConfig("gdn-oracle-scale", 1, 1, 64, 16, 16, 16, "f32", qk_unit_rows=True),
    "gdn-small": PrefillConfig("gdn-small", 2, 4, 2048, 64, 64, 64, "bf16", qk_unit_rows=True),
    "gdn-headline": PrefillConfig("gdn-headline", 4, 16, 8192, 128, 64, 64, "bf16", qk_unit_rows=True,
                                  log_a_mu=-2.0),
}


def make_beta(seed: int, shape) -> np.ndarray:
    """Delta-rule strengths beta = sigmoid(N(0, 1)), float32, for the given shape."""
    shape = tuple(int(x) for x in shape)
    rng = np.random.default_rng(np.random.SeedSequence([0xBE7A, seed, *shape]))
    return (1.0 / (1.0 + np.exp(-rng.standard_normal(shape)))).astype(np.float32)


@dataclass
class PrefillInputs:
    """Host arrays for one prefill call. q/k/v are float32 arrays holding values exactly
    representable in the storage dtype; ``*_bits`` hold the bf16 patterns when dtype is bf16."""
    cfg: PrefillConfig
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    log_a: np.ndarray
    lam: np.ndarray
    bits: dict = field(default_factory=dict)


def _store(x: np.ndarray, dtype: str):
    if dtype == "bf16":
        b = f32_to_bf16_bits(x)
        return bf16_bits_to_f32(b).reshape(x.shape), b.reshape(x.shape)
    return np.ascontiguousarray(x, dtype=np.float32), None


def make_prefill(cfg: PrefillConfig, seed: int = 0, *, B: int | None = None, H: int | None = None,
                 T: int | None = None) -> PrefillInputs:
    """Draw one prefill problem. B/H/T override the config's sizes (same distributions)."""
    B = cfg.B if B is None else B
    H = cfg.H if H is None else H
    T = cfg.T if T is None else T
    L = num_levels(T)
    ss = np.random.SeedSequence([0x11A0, seed, B, H, T, cfg.dk, cfg.dv])
    rq, rk, rv, ra, rl = (np.random.default_rng(s) for s in ss.spawn(5))
    if cfg.qk_unit_rows:
        q = rq.standard_normal((B, H, T, cfg.dk), dtype=np.float32)
        k = rk.standard_normal((B, H, T, cfg.dk), dtype=np.float32)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    else:
        sd = np.float32(1.0 / np.sqrt(cfg.dk))
        q = rq.standard_normal((B, H, T, cfg.dk), dtype=np.float32) * sd
        k = rk.standard_normal((B, H, T, cfg.dk), dtype=np.float32) * sd
    v = rv.standard_normal((B, H, T, cfg.dv), dtype=np.float32)
    log_a = (-_softplus(ra.standard_normal((B, H, T)) + cfg.log_a_mu)).astype(np.float32)
    lam = _softplus(rl.standard_normal((B, H, T, L))).astype(np.float32)
    q, qb = _store(q, cfg.dtype)
    k, kb = _store(k, cfg.dtype)
    v, vb = _store(v, cfg.dtype)
    bits = {"q": qb, "k": kb, "v": vb} if cfg.dtype == "bf16" else {}
    return PrefillInputs(cfg, q, k, v, log_a, lam, bits)


@dataclass
class DecodeInputs:
    """Host arrays for one decode step: q,k [B,H,dk], v [B,H,dv], log_a [B,H], lam [B,H,Lmax]."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    log_a: np.ndarray
    lam: np.ndarray
    bits: dict = field(default_factory=dict)


def make_decode_token(cfg: DecodeConfig, seed: int, *, batch: int | None = None, H: int | None = None) -> DecodeInputs:
    """Draw one decode step's per-token inputs (bf16 or f32 q/k/v; fp32 log_a and lambda)."""
    batch = cfg.batch if batch is None else batch
    H = cfg.H if H is None else H
    ss = np.random.SeedSequence([0xDEC0, seed, batch, H, cfg.dk, cfg.dv])
    rq, rk, rv, ra, rl = (np.random.default_rng(s) for s in ss.spawn(5))
    sd = np.float32(1.0 / np.sqrt(cfg.dk))
    q = rq.standard_normal((batch, H, cfg.dk), dtype=np.float32) * sd
    k = rk.standard_normal((batch, H, cfg.dk), dtype=np.float32) * sd
    v = rv.standard_normal((batch, H, cfg.dv), dtype=np.float32)
    log_a = (-_softplus(ra.standard_normal((batch, H)))).astype(np.float32)
    lam = _softplus(rl.standard_normal((batch, H, cfg.Lmax))).astype(np.float32)
    q, qb = _store(q, cfg.dtype)
    k, kb = _store(k, cfg.dtype)
    v, vb = _store(v, cfg.dtype)
    bits = {"q": qb, "k": kb, "v": vb} if cfg.dtype == "bf16" else {}
    return DecodeInputs(q, k, v, log_a, lam, bits)


def make_positions(cfg: DecodeConfig, seed: int, *, batch: int | None = None, t_max: int | None = None) -> np.ndarray:
    """Per-sequence positions t ~ U[1, t_max), int64."""
    batch = cfg.batch if batch is None else batch
    t_max = cfg.t_max if t_max is None else t_max
    rng = np.random.default_rng(np.random.SeedSequence([0x7105, seed, batch, t_max]))
    return rng.integers(1, t_max, size=batch, dtype=np.int64)


def make_random_states(cfg: DecodeConfig, seed: int, *, batch: int | None = None, H: int | None = None) -> np.ndarray:
    """Random fp32 state sets [B,H,Lmax,dk,dv] with N(0, 1/dk) entries (bandwidth runs and parity
    runs that start from an arbitrary state)."""
    batch = cfg.batch if batch is None else batch
    H = cfg.H if H is None else H
    rng = np.random.default_rng(np.random.SeedSequence([0x57A7, seed, batch, H]))
    sd = np.float32(1.0 / np.sqrt(cfg.dk))
    return rng.standard_normal((batch, H, cfg.Lmax, cfg.dk, cfg.dv), dtype=np.float32) * sd

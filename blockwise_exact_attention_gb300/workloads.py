"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws and prepares inputs (random numbers, the bf16 rounding
of the uploaded bits, rotary embedding and per-head logit spreading applied to
q/k before upload). It holds none of the attention arithmetic and imports
neither the oracle nor the CUDA binding, so both sides can consume its arrays.

Recipe: ``numpy.random.default_rng(seed)`` (PCG64), ``standard_normal`` in
float32, draw order q, k, v, dout, then extras (per-head scales); then rotary
embedding, then the per-head scale, then rounding to bf16 (round to nearest
even) for the bf16 workloads. Seed = 1000 + workload index.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n: int
    l: int
    h: int
    h_kv: int
    d: int
    is_causal: bool
    window: tuple[int, int]
    dtype: str              # "bf16" or "f32"
    seed: int
    rope: bool = False
    head_scale: bool = False
    ring_chunks: int = 0    # > 0: ring-decomposed along l into this many chunks
    description: str = ""

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the measurement plan (the last one split in two).
WORKLOADS: dict[str, Workload] = {
    "tiny_fp32": Workload("tiny_fp32", 1, 128, 2, 2, 64, False, (-1, -1), "f32", 1000,
                          description="non-causal fp32 [1,128,2,64]"),
    "causal_mha_4k": Workload("causal_mha_4k", 2, 4096, 16, 16, 128, True, (-1, -1), "bf16", 1001,
                              description="causal MHA bf16 [2,4096,16,128]"),
    "causal_gqa_8k_rope": Workload("causal_gqa_8k_rope", 1, 8192, 32, 8, 128, True, (-1, -1), "bf16",
                                   1002, rope=True,
                                   description="causal GQA bf16 q[1,8192,32,128] kv[1,8192,8,128] + RoPE"),
    "ring_causal_16k": Workload("ring_causal_16k", 1, 16384, 16, 16, 128, True, (-1, -1), "bf16", 1003,
                                ring_chunks=8,
                                description="causal bf16 [1,16384,16,128] as 8 ring chunks of 2048"),
    "swa_32k_d128": Workload("swa_32k_d128", 1, 32768, 32, 32, 128, True, (1024, 0), "bf16", 1004,
                             head_scale=True,
                             description="sliding window (1024,0) causal bf16 [1,32768,32,128]"),
    "full_32k_d64": Workload("full_32k_d64", 1, 32768, 32, 32, 64, False, (-1, -1), "bf16", 1006,
                             head_scale=True,
                             description="non-causal bf16 [1,32768,32,64]"),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even); returns
    float32 arrays whose values are exactly representable in bf16."""
    x = np.array(x, dtype=np.float32, copy=True, order="C")
    if not np.isfinite(x).all():
        raise ValueError("round_to_bf16 expects finite inputs")
    bits = x.view(np.uint32)
    lsb = bits >> np.uint32(16)
    lsb &= np.uint32(1)
    lsb += np.uint32(0x7FFF)
    bits += lsb            # |x| < 2^128 - 2^112, so this cannot carry into the sign bit
    bits &= np.uint32(0xFFFF0000)
    return x


def rotary(x: np.ndarray, base: float = 10000.0) -> np.ndarray:
    """Rotate-half rotary position embedding on ``x [n, l, h, d]`` in fp64:
    pairs (x_k, x_{k+d/2}), angle = position * base**(-2k/d), positions 0..l-1.
    Returns float32."""
    n, l, h, d = x.shape
    half = d // 2
    inv = base ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = np.arange(l, dtype=np.float64)[:, None] * inv[None, :]          # [l, half]
    cos = np.cos(ang)[None, :, None, :]
    sin = np.sin(ang)[None, :, None, :]
    x64 = x.astype(np.float64)
    a, b = x64[..., :half], x64[..., half:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1).astype(np.float32)


def make_inputs(w: Workload, with_dout: bool = True) -> dict[str, np.ndarray]:
    """Draw q, k, v (and dout) for workload ``w`` as float32 arrays holding the
    exact values that are uploaded (bf16-representable for bf16 workloads)."""
    rng = np.random.default_rng(w.seed)
    q = rng.standard_normal((w.n, w.l, w.h, w.d), dtype=np.float32)
    k = rng.standard_normal((w.n, w.l, w.h_kv, w.d), dtype=np.float32)
    v = rng.standard_normal((w.n, w.l, w.h_kv, w.d), dtype=np.float32)
    dout = rng.standard_normal((w.n, w.l, w.h, w.d), dtype=np.float32) if with_dout else None
    if w.head_scale:
        c = rng.uniform(0.5, 2.0, size=(w.h,)).astype(np.float32)
    if w.rope:
        q = rotary(q)
        k = rotary(k)
    if w.head_scale:
        q = (q * c[None, None, :, None]).astype(np.float32)
    arrs = {"q": q, "k": k, "v": v}
    if dout is not None:
        arrs["dout"] = dout
    if w.dtype == "bf16":
        arrs = {name: round_to_bf16(a) for name, a in arrs.items()}
    return arrs


def small_case(n=1, l=300, h=4, h_kv=2, d=128, is_causal=True, window=(-1, -1),
               dtype="bf16", seed=7, lk=None) -> dict[str, np.ndarray]:
    """Seeded inputs of an arbitrary small shape (ragged tails, odd sizes).
    ``lk`` (default ``l``) sets the key length."""
    lk = l if lk is None else lk
    rng = np.random.default_rng(seed)
    arrs = {
        "q": rng.standard_normal((n, l, h, d), dtype=np.float32),
        "k": rng.standard_normal((n, lk, h_kv, d), dtype=np.float32),
        "v": rng.standard_normal((n, lk, h_kv, d), dtype=np.float32),
        "dout": rng.standard_normal((n, l, h, d), dtype=np.float32),
    }
    if dtype == "bf16":
        arrs = {name: round_to_bf16(a) for name, a in arrs.items()}
    return arrs

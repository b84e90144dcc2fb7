"""Seeded synthetic workloads: shapes, seeds and input draws.

This module holds no attention arithmetic. It only draws the fp16 inputs and
the key lengths that both the CUDA path and the CPU oracle are fed, so the two
sides see identical bits.

Recipe (one numpy PCG64 stream per workload, seeded with the workload's seed):
  Q ~ N(0, sigma_qk^2), then K ~ N(0, sigma_qk^2), then V ~ N(0, sigma_v^2),
  each drawn as float32 standard normals times sigma and rounded to fp16
  (round-to-nearest-even), shape [B, H, N, d]; then, for padded workloads,
  key_lengths[b] ~ uniform integer in [lo, hi] (inclusive). Cross-attention and
  grouped-query workloads draw Q as [B, H, N, d] and K, V as [B, H_kv, N_k, d] in the
  same order. bf16 workloads round the same float32 draws to bfloat16 (nearest even)
  and hold them as uint16 bit patterns; fp32 workloads keep the float32 draws.

The shapes are the workloads the method is measured on: a tiny exact check, a
cross-encoder reranking batch (the "cuda-reranker" README's shape class: many
short padded sequences at head dimension 32), an LLM prefill, a long-context
prefill whose naive score matrix would not fit ("Naive Attention Kernel",
section "The Memory Problem"), and a numerics stress case with peaked rows.
No public dataset is used; these synthetic draws stand in for the reranker's
retrieval corpus.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    key_len_range: tuple[int, int] | None = None  # inclusive [lo, hi] when padded
    check_lse: bool = False
    ignore_padded_queries: bool = False
    Hkv: int | None = None  # key/value heads (None: H, multi-head attention)
    Nk: int | None = None   # keys per head (None: N, self-attention)
    dtype: str = "f16"      # "f16", "bf16" (uint16 bit patterns) or "f32"

    @property
    def H_kv(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    @property
    def N_k(self) -> int:
        return self.N if self.Nk is None else self.Nk

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def describe(self) -> str:
        mask = "causal" if self.causal else "no mask"
        if self.key_len_range:
            mask = f"key padding L~U[{self.key_len_range[0]},{self.key_len_range[1]}]"
        kv = ""
        if self.H_kv != self.H:
            kv += f" H_kv={self.H_kv}"
        if self.N_k != self.N:
            kv += f" N_k={self.N_k}"
        dt = "" if self.dtype == "f16" else f" {self.dtype}"
        return f"{self.name} B={self.B} H={self.H} N={self.N}{kv} d={self.d}{dt} {mask}"


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 64, False, seed=1),
    "rerank": Workload("rerank", 50, 12, 256, 32, False, seed=2, key_len_range=(64, 256),
                       ignore_padded_queries=True),
    "prefill": Workload("prefill", 4, 32, 4096, 128, True, seed=3),
    "long": Workload("long", 1, 32, 32768, 128, True, seed=4),
    "stress": Workload("stress", 2, 16, 8192, 64, False, seed=5, sigma_qk=3.0, check_lse=True),
    # one long causal sequence of a single head: fewer query tile pairs than SMs (the case the
    # split-KV path is for)
    "one_head": Workload("one_head", 1, 1, 32768, 128, True, seed=6),
    # grouped-query prefill: 32 query heads sharing 8 key/value heads
    "gqa_prefill": Workload("gqa_prefill", 4, 32, 4096, 128, True, seed=7, Hkv=8),
    # a block of 1024 new queries over a cached context of 16384 keys (cross-attention shape,
    # causal diagonal at the last rows), grouped-query heads
    "chunk_prefill": Workload("chunk_prefill", 2, 32, 1024, 128, True, seed=8, Hkv=8, Nk=16384),
    # decoding one token per sequence over a cache of 8192 keys, 32 query heads over 8 key/value
    # heads (the diagonal of the causal mask leaves every key to the one query)
    "decode_gqa": Workload("decode_gqa", 8, 32, 1, 128, True, seed=11, Hkv=8, Nk=8192),
    # a block of 8 draft queries per sequence (speculative decoding) over 8192 keys, causal
    "spec_decode": Workload("spec_decode", 8, 32, 8, 128, True, seed=12, Hkv=8, Nk=8192),
    # the prefill shape with bf16 inputs
    "prefill_bf16": Workload("prefill_bf16", 4, 32, 4096, 128, True, seed=9, dtype="bf16"),
    # the reranking shape with fp32 inputs (the precision of the reranker's own kernel)
    "rerank_f32": Workload("rerank_f32", 50, 12, 256, 32, False, seed=10, key_len_range=(64, 256),
                           ignore_padded_queries=True, dtype="f32"),
}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), rounded to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def draw(B: int, H: int, N: int, d: int, seed: int, *, sigma_qk: float = 1.0,
         sigma_v: float = 1.0, key_len_range: tuple[int, int] | None = None):
    """Returns (q, k, v, key_lengths): fp16 arrays [B,H,N,d] and int32 [B] or None."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)

    def normal(sigma):
        x = rng.standard_normal(shape, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        return x.astype(np.float16)

    q = normal(sigma_qk)
    k = normal(sigma_qk)
    v = normal(sigma_v)
    kl = None
    if key_len_range is not None:
        lo, hi = key_len_range
        kl = rng.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)
    return q, k, v, kl


def draw_ex(B: int, H: int, Hkv: int, N: int, Nk: int, d: int, seed: int, *,
            sigma_qk: float = 1.0, sigma_v: float = 1.0,
            key_len_range: tuple[int, int] | None = None, dtype: str = "f16"):
    """Returns (q, k, v, key_lengths): q [B,H,N,d], k and v [B,Hkv,Nk,d] (fp16, uint16
    bfloat16 bit patterns for dtype "bf16", or float32 for "f32"), key_lengths int32 [B] or
    None. With Hkv = H, Nk = N and fp16 the draws are those of draw()."""
    if dtype not in ("f16", "bf16", "f32"):
        raise ValueError("dtype must be 'f16', 'bf16' or 'f32'")
    rng = np.random.Generator(np.random.PCG64(seed))

    def normal(shape, sigma):
        x = rng.standard_normal(shape, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        if dtype == "f32":
            return x
        return x.astype(np.float16) if dtype == "f16" else to_bf16_bits(x)

    q = normal((B, H, N, d), sigma_qk)
    k = normal((B, Hkv, Nk, d), sigma_qk)
    v = normal((B, Hkv, Nk, d), sigma_v)
    kl = None
    if key_len_range is not None:
        lo, hi = key_len_range
        kl = rng.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)
    return q, k, v, kl


def draw_workload(w: Workload):
    if w.Hkv is not None or w.Nk is not None or w.dtype != "f16":
        return draw_ex(w.B, w.H, w.H_kv, w.N, w.N_k, w.d, w.seed, sigma_qk=w.sigma_qk,
                       sigma_v=w.sigma_v, key_len_range=w.key_len_range, dtype=w.dtype)
    return draw(w.B, w.H, w.N, w.d, w.seed, sigma_qk=w.sigma_qk, sigma_v=w.sigma_v,
                key_len_range=w.key_len_range)


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Contract FLOP count: 4*B*H*N^2*d (2d for QK^T and 2d for PV per pair), halved when causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def attention_flops_ex(B: int, H: int, N: int, Nk: int, d: int, causal: bool) -> float:
    """Contract FLOP count of N queries over Nk keys: 4*B*H*N*Nk*d; under the causal mask
    (query i sees keys j <= i + Nk - N) the same convention as attention_flops, i.e. the
    allowed pairs counted as the area of the region, N*Nk - N^2/2 for N <= Nk."""
    if not causal:
        return 4.0 * B * H * N * Nk * d
    if N <= Nk:
        area = N * Nk - N * N / 2.0
    else:
        area = Nk * Nk / 2.0  # the first N - Nk rows see no key
    return 4.0 * B * H * area * d


def min_bytes_ex(B: int, H: int, Hkv: int, N: int, Nk: int, d: int, lse: bool = False) -> int:
    """Minimum HBM traffic: Q read and O written ([B,H,N,d] fp16), K and V read once
    ([B,Hkv,Nk,d] fp16), plus fp32 lse."""
    b = 2 * B * H * N * d * 2 + 2 * B * Hkv * Nk * d * 2
    if lse:
        b += 4 * B * H * N
    return b


def min_bytes(B: int, H: int, N: int, d: int, lse: bool = False) -> int:
    """Minimum HBM traffic: Q, K, V read once and O written once (fp16), plus fp32 lse."""
    b = 4 * B * H * N * d * 2
    if lse:
        b += 4 * B * H * N
    return b

"""Seeded synthetic attention inputs and the benchmark shapes.

This module holds no attention arithmetic: it only draws numbers, rounds them
to bf16 and describes shapes. Both the CUDA path's tests and the CPU oracle's
tests take their inputs from here, so the two sides see the same bits.

Recipe: numpy ``PCG64(seed)`` draws i.i.d. N(0, 1) float32 values for q, k, v
and dO in that order; each is rounded to bf16 (round to nearest, ties to even)
and kept as raw uint16 bits. Derived draws (the boosted key rows of the long
sequence workload, the sequence lengths of the packed workload) come from a
second generator seeded with ``seed + 7``.

Shapes follow the FlashAttention-4 benchmark setup (papercache.org summary,
"experimental setup": 32k tokens, hidden 2048, head dims 64/128 and the (192, 128)
query-key / value head dimensions of DeepSeek V3 with 16 heads, causal and not)
and the FlashAttention-1 kernel analysis shape (wq-win.github.io, section 4:
sequence 1024, head dim 64, 16 heads, batch 64).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "bf16_bits",
    "bf16_bits_to_f64",
    "bf16_bits_to_f32",
    "generate",
    "custom",
    "fwd_flops",
]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    N: int            # fixed length; for packed inputs: the mean-free upper bound of lengths
    d: int
    scale: float
    causal: bool
    seed: int
    varlen: tuple = None       # (n_seqs, min_len, max_len) for packed inputs
    boost_frac: float = 0.0    # fraction of key rows scaled before rounding
    boost: float = 1.0
    note: str = ""
    d_v: int = None            # value / output head dimension (None: same as d)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 128, 64, 1.0 / math.sqrt(8.0), False, 1001,
                     note="B1 H1 N128 d64, scale 1/sqrt(8), non-causal"),
    "short": Workload("short", 64, 16, 16, 1024, 64, 1.0 / 8.0, False, 1002,
                      note="B64 H16 N1024 d64, non-causal"),
    "short_causal": Workload("short_causal", 64, 16, 16, 1024, 64, 1.0 / 8.0, True, 1002,
                             note="B64 H16 N1024 d64, causal"),
    "mid": Workload("mid", 4, 16, 16, 8192, 128, 1.0 / math.sqrt(128.0), False, 1003,
                    note="B4 H16 N8192 d128, non-causal (32k tokens, hidden 2048)"),
    "mid_causal": Workload("mid_causal", 4, 16, 16, 8192, 128, 1.0 / math.sqrt(128.0), True, 1003,
                           note="B4 H16 N8192 d128, causal"),
    "long": Workload("long", 1, 16, 16, 32768, 128, 1.0 / math.sqrt(128.0), True, 1004,
                     boost_frac=0.05, boost=3.0,
                     note="B1 H16 N32768 d128 causal, 5% of key rows x3"),
    # forward only: the (192, 128) head dimensions of the DeepSeek V3 architecture
    # that the FlashAttention-4 benchmark also runs (16 heads, 32k tokens)
    "mla": Workload("mla", 4, 16, 16, 8192, 192, 1.0 / math.sqrt(192.0), False, 1006,
                    note="B4 H16 N8192 d_qk 192 d_v 128, non-causal", d_v=128),
    "mla_causal": Workload("mla_causal", 4, 16, 16, 8192, 192, 1.0 / math.sqrt(192.0), True, 1006,
                           note="B4 H16 N8192 d_qk 192 d_v 128, causal", d_v=128),
    "varlen_gqa": Workload("varlen_gqa", 16, 32, 8, 4096, 128, 1.0 / math.sqrt(128.0), True, 1005,
                           varlen=(16, 512, 4096),
                           note="16 packed sequences, lengths U[512,4096], H_q 32 / H_kv 8, causal"),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


@dataclass
class Inputs:
    """Raw bf16 bits plus the shape description.

    Fixed length: q [B, N, H_q, d], k [B, N, H_kv, d], v [B, N, H_kv, d_v],
    do [B, N, H_q, d_v]. Packed: the same without B and with T rows,
    cu_seqlens int32 [n_seqs + 1]. ``d_v`` defaults to ``d``."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    B: int
    H_q: int
    H_kv: int
    N_q: int
    N_k: int
    d: int
    scale: float
    causal: bool
    cu_seqlens: np.ndarray = None
    meta: dict = field(default_factory=dict)
    d_v: int = None

    def __post_init__(self):
        if self.d_v is None:
            self.d_v = self.d

    @property
    def varlen(self) -> bool:
        return self.cu_seqlens is not None

    def seqlens(self):
        if self.cu_seqlens is None:
            return [self.N_q] * self.B
        return list(np.diff(self.cu_seqlens).astype(int))


def _normal_bits(rng, shape):
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def custom(B, H_q, H_kv, N_q, N_k, d, scale=None, causal=False, seed=7, seqlens=None,
           boost_frac=0.0, boost=1.0, parts=("q", "k", "v", "do"), d_v=None) -> Inputs:
    """General generator. ``seqlens`` (list of ints) selects packed layout; then
    B = len(seqlens) and N_q = N_k = sum(seqlens). ``d_v`` (default ``d``) is the
    head dimension of v and dO."""
    if d_v is None:
        d_v = d
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rng = np.random.Generator(np.random.PCG64(seed))
    rng2 = np.random.Generator(np.random.PCG64(seed + 7))
    cu = None
    if seqlens is not None:
        seqlens = [int(x) for x in seqlens]
        cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(seqlens)
        B = len(seqlens)
        N_q = N_k = int(cu[-1])
        lead_q, lead_k = (N_q,), (N_k,)
    else:
        lead_q, lead_k = (B, N_q), (B, N_k)
    shapes = dict(q=lead_q + (H_q, d), k=lead_k + (H_kv, d), v=lead_k + (H_kv, d_v),
                  do=lead_q + (H_q, d_v))
    out = {}
    for name in ("q", "k", "v", "do"):
        shape = shapes[name]
        if name not in parts:
            out[name] = None
            # keep the stream aligned: draw and drop
            rng.standard_normal(size=shape, dtype=np.float32)
            continue
        x = rng.standard_normal(size=shape, dtype=np.float32)
        if name == "k" and boost_frac > 0.0:
            n_boost = int(math.floor(boost_frac * N_k))
            if cu is None:
                for b in range(B):
                    for g in range(H_kv):
                        rows = rng2.choice(N_k, size=n_boost, replace=False)
                        x[b, rows, g, :] *= np.float32(boost)
            else:
                for g in range(H_kv):
                    rows = rng2.choice(N_k, size=n_boost, replace=False)
                    x[rows, g, :] *= np.float32(boost)
        out[name] = bf16_bits(x)
        del x
    return Inputs(out["q"], out["k"], out["v"], out["do"], B, H_q, H_kv, N_q, N_k, d,
                  float(scale), bool(causal), cu,
                  meta=dict(seed=seed, boost_frac=boost_frac, boost=boost), d_v=d_v)


def generate(name: str, parts=("q", "k", "v", "do")) -> Inputs:
    """Inputs of one of the named workloads in ``WORKLOADS``."""
    w = WORKLOADS[name]
    if w.varlen is not None:
        n_seqs, lo, hi = w.varlen
        rng2 = np.random.Generator(np.random.PCG64(w.seed + 7))
        seqlens = rng2.integers(lo, hi, size=n_seqs, endpoint=True)
        inp = custom(n_seqs, w.H_q, w.H_kv, 0, 0, w.d, w.scale, w.causal, seed=w.seed,
                     seqlens=seqlens, parts=parts, d_v=w.d_v)
    else:
        inp = custom(w.B, w.H_q, w.H_kv, w.N, w.N, w.d, w.scale, w.causal, seed=w.seed,
                     boost_frac=w.boost_frac, boost=w.boost, parts=parts, d_v=w.d_v)
    inp.meta["workload"] = name
    return inp


def fwd_flops(B, H_q, N_q, N_k, d, causal, seqlens=None, d_v=None) -> float:
    """Convention of the FlashAttention-4 benchmark: 4 * N_q * N_k * d per head,
    halved for causal; packed inputs use sum of L^2. Backward is 2.5x this. With
    separate head dimensions the two contractions count 2 * N_q * N_k * d (QK^T)
    and 2 * N_q * N_k * d_v (PV)."""
    width = 2.0 * d if d_v is None else float(d + d_v)
    if seqlens is not None:
        pairs = float(sum(int(L) * int(L) for L in seqlens))
        f = 2.0 * pairs * width * H_q
    else:
        f = 2.0 * B * H_q * float(N_q) * float(N_k) * width
    return f / 2.0 if causal else f

"""Seeded synthetic workloads for MoE dispatch + combine.

This module only *makes inputs*: token rows ``x``, router choices ``topk_idx``,
router weights ``topk_w`` and the expert outputs ``y`` that the combine stage
gathers.  It contains none of the dispatch/combine arithmetic (no counting,
no scan, no placement, no weighted sum), so the CUDA path and the CPU oracle
can both be fed from it without sharing any of the method's code.

The router that produces ``topk_idx``/``topk_w`` is simulated here: a small
linear router turning logits into a distribution and keeping the top-K
experts ("Efficient and portable mixture-of-experts communication",
introduction).  Its shapes follow the five workloads below; no trained weights
or datasets are involved.

bf16 values are carried as ``numpy.uint16`` arrays holding the raw bf16 bit
patterns; they are produced with torch's float32 -> bfloat16 conversion
(round-to-nearest-even).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """Sizes of one dispatch+combine layer.

    T: total tokens over all logical ranks; N: logical ranks (rank s owns
    tokens [s*T/N, (s+1)*T/N)); E: experts (E/N per rank, contiguous);
    K: experts per token (top-k); H: hidden size (bf16 elements per row).
    """

    name: str
    T: int
    H: int
    K: int
    E: int
    N: int
    router: str
    index: int = 0  # position in WORKLOADS; seeds are 1234 + index

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def tokens_per_rank(self) -> int:
        return self.T // self.N

    @property
    def rows(self) -> int:
        return self.T * self.K

    def describe(self) -> Dict[str, int | str]:
        return {"workload": self.name, "T": self.T, "H": self.H, "K": self.K,
                "E": self.E, "N": self.N, "tokens_per_rank": self.tokens_per_rank,
                "router": self.router}


# The five workloads: a tiny smoke case, then shapes of Mixtral 8x7B,
# DeepSeek-R1 decode, Kimi-K2, and a worst case for the receive bound where
# every token picks only experts of rank 0.
WORKLOADS: List[Workload] = [
    Workload("tiny", T=64, H=256, K=2, E=8, N=2, router="softmax_topk", index=0),
    Workload("mixtral", T=4096, H=4096, K=2, E=8, N=8, router="uniform_topk_softmax", index=1),
    Workload("deepseek", T=32 * 128, H=7168, K=8, E=256, N=32, router="sigmoid_topk", index=2),
    Workload("kimi", T=64 * 256, H=7168, K=8, E=384, N=64, router="zipf_gumbel_topk", index=3),
    Workload("worst", T=16 * 512, H=7168, K=8, E=128, N=16, router="rank0_only", index=4),
]
BY_NAME: Dict[str, Workload] = {w.name: w for w in WORKLOADS}


def custom(name: str, T: int, H: int, K: int, E: int, N: int,
           router: str = "uniform_random", seed_index: int = 100) -> Workload:
    """A workload of arbitrary sizes for edge-case tests (router defaults to a
    uniformly random choice of K distinct experts)."""
    return Workload(name, T=T, H=H, K=K, E=E, N=N, router=router, index=seed_index)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns (torch RNE conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, rows: int, cols: int,
                 chunk_rows: int = 4096) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = to_bf16_bits(rng.standard_normal((r1 - r0, cols), dtype=np.float32))
    return out


def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    # Descending score; equal scores keep the lower expert index first.
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :k]


def _softmax(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def make_routing(w: Workload, rng: np.random.Generator):
    """Simulated router output: (topk_idx int32 [T,K], topk_w float32 [T,K])."""
    T, E, K, N = w.T, w.E, w.K, w.N
    if w.router == "softmax_topk":
        p = _softmax(rng.standard_normal((T, E)))
        idx = _topk_desc(p, K)
        wt = np.take_along_axis(p, idx, axis=1)
        wt = wt / wt.sum(axis=1, keepdims=True)
    elif w.router == "uniform_topk_softmax":
        logits = rng.random((T, E))
        idx = _topk_desc(logits, K)
        wt = _softmax(np.take_along_axis(logits, idx, axis=1))
    elif w.router == "sigmoid_topk":
        score = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, E))))
        idx = _topk_desc(score, K)
        wt = np.take_along_axis(score, idx, axis=1)
        wt = wt / wt.sum(axis=1, keepdims=True)
    elif w.router == "zipf_gumbel_topk":
        # Expert popularity p_e ~ (rank_e + 1)^-1.2 with ranks scattered over
        # experts by a seeded permutation; K distinct experts per token drawn
        # without replacement by Gumbel-top-k on log p_e.
        rank_of = rng.permutation(E)
        logp = -1.2 * np.log(rank_of + 1.0)
        u = rng.random((T, E))
        u = np.clip(u, 1e-300, 1.0)
        key = logp[None, :] - np.log(-np.log(u))
        idx = _topk_desc(key, K)
        wt = _softmax(np.take_along_axis(key, idx, axis=1))
    elif w.router == "rank0_only":
        L = E // N
        if L < K:
            raise ValueError("rank0_only needs E/N >= K")
        idx = np.stack([rng.permutation(L)[:K] for _ in range(T)]) if T else np.zeros((0, K), np.int64)
        wt = rng.random((T, K))
        wt = wt / wt.sum(axis=1, keepdims=True)
    elif w.router == "uniform_random":
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K] if T else np.zeros((0, K), np.int64)
        wt = rng.random((T, K)) + 0.05
        wt = wt / wt.sum(axis=1, keepdims=True)
    else:
        raise ValueError(f"unknown router {w.router!r}")
    return (np.ascontiguousarray(idx, dtype=np.int32).reshape(T, K),
            np.ascontiguousarray(wt, dtype=np.float32).reshape(T, K))


@dataclass
class LayerInputs:
    workload: Workload
    x: np.ndarray          # uint16 bf16 bits [T, H]
    topk_idx: np.ndarray   # int32 [T, K]
    topk_w: np.ndarray     # float32 [T, K]
    y: Optional[np.ndarray] = field(default=None)  # uint16 bf16 bits [T*K, H], expert outputs in dispatch layout


def make_inputs(w: Workload, with_y: bool = True, seed: Optional[int] = None) -> LayerInputs:
    """All inputs of one layer, from numpy PCG64 seeded with 1234 + index.

    x ~ N(0,1) rounded to bf16; y (the synthetic expert outputs, one row per
    dispatched (token, slot) pair, in the grouped row layout) ~ N(0,1) bf16.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    topk_idx, topk_w = make_routing(w, rng)
    x = _normal_bf16(rng, w.T, w.H)
    y = _normal_bf16(rng, w.T * w.K, w.H) if with_y else None
    return LayerInputs(w, x, topk_idx, topk_w, y)

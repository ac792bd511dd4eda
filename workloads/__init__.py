"""Seeded synthetic inputs for the MoE dispatch / combine layout path.

This module simulates the caller's side of the exchange: a router that emits
``topk_idx[T, K]`` (int64, -1 = unused slot) and ``topk_weights[T, K]``
(float32), and the bf16 hidden states ``x[T, H]`` that are dispatched.  The
router itself is not part of the method ("Deep Dive - DeepEP", section "Why
expert parallelism needs a communication layer": DeepEP does not implement the
router); it is simulated here only so that inputs have the shapes and routing
statistics of the workloads the pages describe.

Nothing in this module computes any step of layout, dispatch or combine.  Both
the CPU oracle (through the tests) and the CUDA path are fed from here, and
neither is imported by it.

Recipe (identical for every workload, seed 0 unless stated):

1. ``x = standard_normal((T, H), float32)`` rounded to bf16 by PyTorch's own
   round-to-nearest-even cast, kept as raw uint16 bit patterns.
2. ``logits = standard_normal((T, E), float32)``.
3. Skewed workloads only: ``perm = permutation(E)``, ``p_e ~ (perm[e]+1)^-alpha``,
   ``bias_e = ln p_e - mean(ln p)`` added to the logits used for selection.
4. Top-K selection by descending score, ties to the lower expert id.
   Weights: softmax over the K selected *unbiased* logits (they sum to 1).
5. Masking: exactly ``round(mask_frac * T * K)`` distinct (t, k) slots chosen
   without replacement are set to -1.  Their weights are left in place.
6. Expert outputs for combine (when requested): bf16 N(0, 1), drawn after the
   mask from the same stream.

All draws come from ``numpy.random.Generator(PCG64(seed))`` in that order.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and routing statistics of one synthetic workload."""

    name: str
    num_tokens: int          # T: tokens on the GPU (all logical source ranks)
    hidden: int              # H: hidden size (bf16 channels per row)
    num_experts: int         # E
    num_topk: int            # K
    num_ranks: int           # R: logical EP ranks, E / R experts each
    use_fp8_dispatch: bool   # dispatch payload format
    expert_alignment: int = 128
    zipf_alpha: Optional[float] = None
    mask_frac: float = 0.0

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.num_ranks

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _w(name, T, H, E, K, R, fp8, **kw) -> Workload:
    return Workload(name, T, H, E, K, R, fp8, **kw)


# The five workload families of the pages' DeepSeek-V3-shaped benchmarks
# (8K tokens per batch, hidden 7168, top-8, FP8 dispatch, BF16 combine are the
# README shapes named in "Deep Dive - DeepEP", section "Logical bandwidth is
# not a NIC counter").  The sweep is listed per T and per payload format.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        _w("tiny", 16, 128, 8, 2, 2, False),
        _w("decode", 128, 7168, 256, 8, 32, True),
        _w("prefill", 4096, 7168, 256, 8, 8, False),
        _w("skew", 8192, 4096, 64, 6, 8, True, zipf_alpha=1.2, mask_frac=0.05),
        _w("sweep1k", 1024, 7168, 256, 8, 64, False),
        _w("sweep4k", 4096, 7168, 256, 8, 64, False),
        _w("sweep16k", 16384, 7168, 256, 8, 64, False),
        _w("sweep1k_fp8", 1024, 7168, 256, 8, 64, True),
        _w("sweep4k_fp8", 4096, 7168, 256, 8, 64, True),
        _w("sweep16k_fp8", 16384, 7168, 256, 8, 64, True),
    ]
}


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns, via PyTorch's RNE cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def route(logits: np.ndarray, K: int, bias: Optional[np.ndarray] = None):
    """Simulated router: top-K by descending (biased) score, softmax weights.

    Returns ``(topk_idx int64 [T,K], topk_weights float32 [T,K])``.
    """
    score = logits if bias is None else logits + bias[None, :].astype(np.float32)
    # stable sort on the negated score: descending value, lower id on ties
    idx = np.argsort(-score, axis=1, kind="stable")[:, :K].astype(np.int64)
    sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    sel = np.exp(sel - sel.max(axis=1, keepdims=True))
    w = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.ascontiguousarray(idx), np.ascontiguousarray(w)


def make_inputs(wl: Workload, seed: int = 0, expert_output_rows: int = 0):
    """Draw one workload's inputs.

    Returns a dict with ``x`` (uint16 bf16 bits [T,H]), ``topk_idx`` (int64
    [T,K]), ``topk_weights`` (float32 [T,K]) and, if ``expert_output_rows`` >
    0, ``expert_out`` (uint16 bf16 bits [rows,H]) for combine.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    T, H, E, K = wl.num_tokens, wl.hidden, wl.num_experts, wl.num_topk
    x = to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    logits = rng.standard_normal((T, E), dtype=np.float32)
    bias = None
    if wl.zipf_alpha is not None:
        perm = rng.permutation(E)
        logp = -wl.zipf_alpha * np.log(perm.astype(np.float64) + 1.0)
        logp -= np.log(np.exp(logp).sum())
        bias = logp - logp.mean()
    idx, w = route(logits, K, bias)
    if wl.mask_frac > 0:
        n_mask = int(round(wl.mask_frac * T * K))
        flat = rng.choice(T * K, n_mask, replace=False)
        idx.reshape(-1)[flat] = -1
    out = {"x": x, "topk_idx": idx, "topk_weights": w}
    if expert_output_rows > 0:
        out["expert_out"] = to_bf16_bits(
            rng.standard_normal((expert_output_rows, H), dtype=np.float32)
        )
    return out


def random_routes(rng: np.random.Generator, T: int, E: int, K: int,
                  mask_frac: float = 0.0) -> np.ndarray:
    """Uniform random distinct-expert routes (no router), optionally masked."""
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    if mask_frac > 0:
        m = rng.random((T, K)) < mask_frac
        idx[m] = -1
    return idx

"""Seeded synthetic inputs for the mHC sublayer boundary.

This module only draws random numbers and stores them in the boundary's
input formats; it holds none of the boundary's arithmetic, and both the CPU
oracle's tests and the GPU path take their inputs from it.

Every tensor draws from its own child stream of ``numpy.random.SeedSequence
(seed)``, in the fixed order of ``STREAMS``, so a tensor's values do not
depend on which other tensors a problem needs.  Distributions follow the
workloads named for this boundary:

* partials, routed rows, shared-expert rows ~ N(0, 0.05), rounded to BF16;
* residual streams ~ N(0, 1), BF16;
* hc_fn ~ N(0, std = 1/sqrt(4H)), FP32, so that every prenorm mix is ~N(0, 1);
* base ~ N(0, 0.1) FP32; norm weight ~ 1 + N(0, 0.1), BF16; scale = (1, 1, 1);
* incoming post-mix ~ post_mult * U(0.02, 0.98) FP32 (inside (0, post_mult));
* incoming residual mix: a random convex combination (Dirichlet(1) weights)
  of the 24 permutation matrices of size 4, hence doubly stochastic, like the
  residual mix a previous boundary emits;
* MoE routing weights = normalised exponentials of N(0, 1) over top_k, FP32;
  route indices: per rank a random permutation of 0 .. m*top_k-1 (every rank
  holds every route), with an optional fraction of routes marked -1 ("expert
  not held by this rank").
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field

import numpy as np

HC = 4
MIX = 24

STREAMS = ("partials", "residual", "post", "comb", "hc_fn", "base", "gamma",
           "routed", "idx", "weights", "shared", "holes")


@dataclass(frozen=True)
class Workload:
    """A named workload: sizes of one boundary call."""
    name: str
    hidden: int
    tp: int
    m: int
    top_k: int = 0
    moe: bool = False
    mxfp8: bool = False
    bf16_fn: bool = False    # prenorm weight as BF16 [24][4H] instead of FP32 [4H][24]
    consume: bool = False    # the delayed-mHC consumer: carried pre, no GEMV
    residual_only: bool = False
    owner: bool = False      # two-shot reduction: an owner reduce sums the partials first


# The workloads this boundary is measured and checked on.
WORKLOADS = {
    "tiny": [Workload("tiny", 5120, 4, 4)],
    "decode": [Workload("decode", 5120, 8, m) for m in (1, 8, 32, 64)],
    "glm": [Workload("glm", 6144, 4, 1 << i) for i in range(10)],
    "moe": [Workload("moe", 5120, 8, 256, top_k=8, moe=True)],
    "large_mxfp8": [Workload("large_mxfp8", 6144, 8, 4096, mxfp8=True)],
    # the GLM shapes with the weight in the GLM page's BF16 [24][4H] form
    "glm_bf16fn": [Workload("glm_bf16fn", 6144, 4, m, bf16_fn=True) for m in (1, 64, 256, 512)],
    "large_bf16fn": [Workload("large_bf16fn", 6144, 8, 4096, mxfp8=True, bf16_fn=True)],
    # the delayed-mHC consumer (carried pre) and its residual-only form
    "consume": [Workload("consume", 6144, 8, m, consume=True) for m in (1, 256, 4096)],
    "residual_only": [Workload("residual_only", 6144, 8, 4096, consume=True, residual_only=True)],
    # the two-shot (owner-reduce) reduction emulated on one GPU
    "owner_reduce": [Workload("owner_reduce", 6144, 4, 256, owner=True),
                     Workload("owner_reduce", 6144, 8, 4096, mxfp8=True, owner=True)],
}


def bf16_bits(x) -> np.ndarray:
    """Store finite FP32 values as BF16 bit patterns (nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def _normal_bf16(rng, shape, std, mean=0.0) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    flat = out.reshape(-1, shape[-1])
    step = max(1, (1 << 24) // shape[-1])       # draw in slabs of ~16M values
    for start in range(0, flat.shape[0], step):
        z = rng.standard_normal((min(step, flat.shape[0] - start), shape[-1]), dtype=np.float32)
        flat[start:start + z.shape[0]] = bf16_bits(z * np.float32(std) + np.float32(mean))
    return out


_PERMUTATIONS = np.array(
    [np.eye(HC, dtype=np.float64)[list(p)] for p in itertools.permutations(range(HC))])


def make_inputs(hidden: int, tp: int, m: int, *, top_k: int = 0, moe: bool = False,
                seed: int = 0, post_mult: float = 2.0, holes: float = 0.0) -> dict:
    """All inputs of one boundary call as NumPy arrays (BF16 as uint16 bits)."""
    rngs = dict(zip(STREAMS, (np.random.default_rng(s)
                              for s in np.random.SeedSequence(seed).spawn(len(STREAMS)))))
    out = {}
    if moe:
        if top_k <= 0:
            raise ValueError("MoE inputs need top_k >= 1")
        rows = m * top_k
        out["routed"] = _normal_bf16(rngs["routed"], (tp, rows, hidden), 0.05)
        idx = np.stack([rngs["idx"].permutation(rows).reshape(m, top_k) for _ in range(tp)])
        if holes > 0:
            idx[rngs["holes"].random(idx.shape) < holes] = -1
        out["idx"] = idx.astype(np.int32)
        z = rngs["weights"].standard_normal((m, top_k))
        w = np.exp(z - z.max(axis=1, keepdims=True))
        out["weights"] = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
        out["shared"] = _normal_bf16(rngs["shared"], (tp, m, hidden), 0.05)
    else:
        out["partials"] = _normal_bf16(rngs["partials"], (tp, m, hidden), 0.05)
    out["residual"] = _normal_bf16(rngs["residual"], (m, HC, hidden), 1.0)
    out["post"] = (post_mult * rngs["post"].uniform(0.02, 0.98, (m, HC))).astype(np.float32)
    lam = rngs["comb"].dirichlet(np.ones(len(_PERMUTATIONS)), size=m)
    out["comb"] = np.einsum("mp,pij->mij", lam, _PERMUTATIONS).astype(np.float32)
    out["hc_fn"] = (rngs["hc_fn"].standard_normal((HC * hidden, MIX), dtype=np.float32)
                    * np.float32(1.0 / np.sqrt(HC * hidden)))
    out["scale"] = np.ones(3, np.float32)
    out["base"] = (rngs["base"].standard_normal(MIX) * 0.1).astype(np.float32)
    out["gamma"] = bf16_bits(1.0 + 0.1 * rngs["gamma"].standard_normal(hidden))
    return out


def bf16_weight(hc_fn: np.ndarray) -> np.ndarray:
    """The prenorm weight in the GLM page's form, BF16 [24][4H], from the FP32
    [4H][24] draw (the same values, transposed and rounded to BF16)."""
    return bf16_bits(np.ascontiguousarray(hc_fn.T))


def inputs_for(w: Workload, seed: int = 0) -> dict:
    out = make_inputs(w.hidden, w.tp, w.m, top_k=w.top_k, moe=w.moe, seed=seed)
    if w.bf16_fn:
        out["hc_fn_bf16"] = bf16_weight(out.pop("hc_fn"))
    if w.consume and not w.residual_only:
        # a carried pre-mix: sigmoid outputs plus hc_eps lie in (0, 1]
        out["pre"] = np.random.default_rng(seed + 7919).uniform(0.05, 1.0, (w.m, HC)).astype(np.float32)
    return out

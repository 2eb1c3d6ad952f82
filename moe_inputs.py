"""Seeded synthetic inputs for the fused MoE-FFN workloads.

This module is shared by the oracle-side tests, the CUDA-side tests and the
benchmark.  It holds no arithmetic of the method itself: it only draws random
numbers (numpy PCG64, one sub-stream per tensor and per expert) and rounds them
to bf16 (round to nearest even on the fp32 bit pattern).  The routing
generators pick expert ids and softmax-normalised routing weights, which in a
real model come from the router and are inputs to the fused operator.

Workloads (dimension names follow the HyperMegaMoE API, §3.1):

========  =====  ====  ====  ===  =  ===============================
name        T      H     I    E   K  routing
========  =====  ====  ====  ===  =  ===============================
tiny         64   128    64    8  2  uniform, K distinct per token
prefill    4096  2048  1408   64  6  uniform
skewed    16384  7168  2048   32  8  Zipf(1.2) over a seeded expert
                                     permutation, 3 experts never drawn
decode      128  7168  2048  256  8  uniform
backward   4096  2048  1408   64  6  uniform, with dy
skewed_bwd 4096  2048  1408   64  6  Zipf(1.2) as above, with dy
========  =====  ====  ====  ===  =  ===============================

x ~ N(0,1), up_proj ~ N(0, 1/H), down_proj ~ N(0, 1/I), dy ~ N(0,1),
topk_weights = softmax over K of N(0,1) logits.  Everything is drawn in fp32
and rounded once to bf16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

# sub-stream tags
_TAG_X, _TAG_IDS, _TAG_W, _TAG_DY, _TAG_W1, _TAG_W2, _TAG_PERM = 1, 2, 3, 4, 5, 6, 7
_TAG_SW1, _TAG_SW2 = 8, 9  # the optional shared expert


@dataclass(frozen=True)
class Shape:
    T: int
    H: int
    I: int
    E: int
    K: int

    @property
    def TK(self) -> int:
        return self.T * self.K


CONFIGS = {
    "tiny": dict(shape=Shape(64, 128, 64, 8, 2), routing="uniform", seed=1000),
    "prefill": dict(shape=Shape(4096, 2048, 1408, 64, 6), routing="uniform", seed=1001),
    "skewed": dict(shape=Shape(16384, 7168, 2048, 32, 8), routing="zipf", seed=1002),
    "decode": dict(shape=Shape(128, 7168, 2048, 256, 8), routing="uniform", seed=1003),
    "backward": dict(shape=Shape(4096, 2048, 1408, 64, 6), routing="uniform", seed=1004),
    # hot-expert backward: the prefill shape with the skewed workload's routing law
    "skewed_bwd": dict(shape=Shape(4096, 2048, 1408, 64, 6), routing="zipf", seed=1005),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        v *= np.float32(scale)
    return f32_to_bf16_bits(v)


def uniform_distinct_ids(rng: np.random.Generator, T: int, E: int, K: int) -> np.ndarray:
    """Per token, the first K entries of a uniformly random permutation of E."""
    u = rng.random(size=(T, E), dtype=np.float64)
    return np.argsort(u, axis=1, kind="stable")[:, :K].astype(np.int32)


def zipf_ids(rng: np.random.Generator, perm_rng: np.random.Generator, T: int, E: int,
             K: int, s: float = 1.2, n_empty: int = 3) -> np.ndarray:
    """K distinct experts per token, drawn without replacement from a Zipf(s)
    law over a seeded expert permutation; the last n_empty experts of the
    permutation have probability zero (Gumbel-top-K sampling)."""
    pi = perm_rng.permutation(E)
    n = E - n_empty
    ranks = np.arange(1, n + 1, dtype=np.float64)
    p = np.zeros(E, np.float64)
    p[pi[:n]] = ranks ** (-s)
    p /= p.sum()
    with np.errstate(divide="ignore"):
        logp = np.log(p)
    g = -np.log(-np.log(rng.random(size=(T, E), dtype=np.float64)))
    keys = logp[None, :] + g
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)
    return ids


def softmax_weights_bf16(rng: np.random.Generator, T: int, K: int) -> np.ndarray:
    logits = rng.standard_normal(size=(T, K), dtype=np.float32)
    logits -= logits.max(axis=1, keepdims=True)
    ex = np.exp(logits)
    return f32_to_bf16_bits(ex / ex.sum(axis=1, keepdims=True))


class Problem:
    """One seeded workload.  Small tensors are materialised eagerly; expert
    weights are drawn per expert (so a caller may build only the experts it
    needs, or stream them to the device one at a time)."""

    def __init__(self, shape: Shape, seed: int, routing: str = "uniform"):
        self.shape = shape
        self.seed = seed
        self.routing = routing
        T, H, I, E, K = shape.T, shape.H, shape.I, shape.E, shape.K
        self.x = normal_bf16(_rng(seed, _TAG_X), (T, H))
        if routing == "uniform":
            self.topk_ids = uniform_distinct_ids(_rng(seed, _TAG_IDS), T, E, K)
        elif routing == "zipf":
            self.topk_ids = zipf_ids(_rng(seed, _TAG_IDS), _rng(seed, _TAG_PERM), T, E, K)
        else:
            raise ValueError(routing)
        self.topk_weights = softmax_weights_bf16(_rng(seed, _TAG_W), T, K)
        self._dy = None
        self._W1 = None
        self._W2 = None

    @property
    def dy(self) -> np.ndarray:
        if self._dy is None:
            s = self.shape
            self._dy = normal_bf16(_rng(self.seed, _TAG_DY), (s.T, s.H))
        return self._dy

    def expert_W1(self, e: int) -> np.ndarray:
        """up_proj_weight[e], bf16 bits [H, 2I]."""
        s = self.shape
        return normal_bf16(_rng(self.seed, _TAG_W1, e), (s.H, 2 * s.I), 1.0 / np.sqrt(s.H))

    def expert_W2(self, e: int) -> np.ndarray:
        """down_proj_weight[e], bf16 bits [I, H]."""
        s = self.shape
        return normal_bf16(_rng(self.seed, _TAG_W2, e), (s.I, s.H), 1.0 / np.sqrt(s.I))

    def shared_W1(self) -> np.ndarray:
        """Optional shared expert's up_proj weight, bf16 bits [H, 2I] (drawn like a
        routed expert's, from its own sub-stream)."""
        s = self.shape
        return normal_bf16(_rng(self.seed, _TAG_SW1), (s.H, 2 * s.I), 1.0 / np.sqrt(s.H))

    def shared_W2(self) -> np.ndarray:
        """Optional shared expert's down_proj weight, bf16 bits [I, H]."""
        s = self.shape
        return normal_bf16(_rng(self.seed, _TAG_SW2), (s.I, s.H), 1.0 / np.sqrt(s.I))

    def _all(self, fn, shape_tail):
        s = self.shape
        out = np.empty((s.E,) + shape_tail, np.uint16)

        def one(e):
            out[e] = fn(e)

        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(one, range(s.E)))
        return out

    @property
    def W1(self) -> np.ndarray:
        if self._W1 is None:
            s = self.shape
            self._W1 = self._all(self.expert_W1, (s.H, 2 * s.I))
        return self._W1

    @property
    def W2(self) -> np.ndarray:
        if self._W2 is None:
            s = self.shape
            self._W2 = self._all(self.expert_W2, (s.I, s.H))
        return self._W2


def make(name: str) -> Problem:
    c = CONFIGS[name]
    return Problem(c["shape"], c["seed"], c["routing"])


def make_shape(T: int, H: int, I: int, E: int, K: int, seed: int = 7,
               routing: str = "uniform") -> Problem:
    return Problem(Shape(T, H, I, E, K), seed, routing)

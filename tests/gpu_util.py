"""Helpers shared by the GPU parity tests: device upload of the seeded inputs,
calls through the C ABI (via the thin binding) and the elementwise tolerance

    |gpu - ref| <= 1e-2 + 2e-2 * |ref|

for bf16 storage with fp32 accumulation, against the fp64 oracle."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from types import SimpleNamespace

import numpy as np
import torch

import dispatch_grouped_gemm_gb300 as hmm
import moe_inputs as mi

ATOL, RTOL = 1e-2, 2e-2


def dev():
    return torch.device("cuda", 0)


def bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check(name: str, gpu: np.ndarray, ref: np.ndarray):
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{name}: non-finite values"
    err = np.abs(gpu - ref)
    lim = ATOL + RTOL * np.abs(ref)
    bad = err > lim
    if bad.any():
        idx = np.unravel_index(np.argmax(err / lim), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())}/{bad.size} outside |d| <= {ATOL} + {RTOL}|ref|; worst at "
            f"{idx}: gpu={gpu[idx]!r} ref={ref[idx]!r} ratio={float((err / lim)[idx]):.3f}")
    return float((err / lim).max()) if err.size else 0.0


def problem(T, H, I, E, K, seed=7, ids=None, w=None):
    """Seeded inputs (bf16 bits) with optional explicit routing."""
    p = mi.make_shape(T, H, I, E, K, seed=seed)
    ns = SimpleNamespace(T=T, H=H, I=I, E=E, K=K, x=p.x, ids=p.topk_ids if ids is None else ids,
                         w=p.topk_weights if w is None else w, W1=p.W1, W2=p.W2, dy=p.dy)
    ns.ids = np.ascontiguousarray(ns.ids, dtype=np.int32)
    return ns


def upload(p, weights_dtype="bf16"):
    d = SimpleNamespace()
    d.x = bf16(p.x)
    d.ids = torch.from_numpy(np.ascontiguousarray(p.ids, dtype=np.int32)).to(dev())
    d.w = bf16(p.w)
    if weights_dtype == "f32":
        d.w = d.w.float()
    d.W1 = bf16(p.W1)
    d.W2 = bf16(p.W2)
    d.dy = bf16(p.dy)
    return d


def upload_problem_weights(prob: mi.Problem):
    """Device copies of every expert's weights, drawn per expert on the host
    in parallel and streamed to the device (bounded host memory)."""
    s = prob.shape
    W1 = torch.empty((s.E, s.H, 2 * s.I), dtype=torch.bfloat16, device=dev())
    W2 = torch.empty((s.E, s.I, s.H), dtype=torch.bfloat16, device=dev())
    workers = min(16, os.cpu_count() or 1)

    def gen(e):
        return e, prob.expert_W1(e), prob.expert_W2(e)

    with ThreadPoolExecutor(max_workers=workers) as ex:
        for start in range(0, s.E, workers):
            for e, w1, w2 in ex.map(gen, range(start, min(s.E, start + workers))):
                W1[e].copy_(bf16(w1))
                W2[e].copy_(bf16(w2))
    return W1, W2


class Runner:
    """Calls hmm_forward / hmm_backward through the binding with explicit
    buffers (so tests can reuse and inspect them)."""

    def __init__(self):
        self.ctx = hmm.Context.for_device(dev())

    def shape(self, d):
        return hmm.Context.shape_of(d.x, d.ids, d.w, d.W1, d.W2)

    def forward(self, d, training=True):
        sh = self.shape(d)
        fwd, sv, _ = hmm.hmm_workspace_size(sh, training)
        y = torch.empty_like(d.x)
        ws = torch.empty(max(fwd, 16), dtype=torch.uint8, device=dev())
        saved = torch.empty(max(sv, 16), dtype=torch.uint8, device=dev()) if training else None
        hmm.hmm_forward(self.ctx.handle, sh, d.x, d.ids, d.w, d.W1, d.W2, y, saved, ws)
        return y, saved

    def backward(self, d, saved):
        sh = self.shape(d)
        _, _, bwd = hmm.hmm_workspace_size(sh, True)
        ws = torch.empty(max(bwd, 16), dtype=torch.uint8, device=dev())
        dx = torch.empty_like(d.x)
        dW1 = torch.full_like(d.W1, float("nan"))   # stale values must be overwritten
        dW2 = torch.full_like(d.W2, float("nan"))
        dw = torch.empty_like(d.w)
        hmm.hmm_backward(self.ctx.handle, sh, d.dy, d.w, d.W1, d.W2, saved, dx, dW1, dW2, dw, ws)
        return dx, dW1, dW2, dw

    def status(self):
        return hmm.hmm_status(self.ctx.handle)

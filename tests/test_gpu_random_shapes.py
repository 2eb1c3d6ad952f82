"""Seeded random shapes and routings on the GPU path vs the fp64 oracle.

Each case draws T (1-900 tokens), H (a multiple of 8 up to 512), I (a
multiple of 8 from 64 to 384), E (1-48 experts), K (2-8 slots per token), the
routing (distinct experts per token, or repeats allowed, with some experts
left empty), the routing weights' dtype (bf16 or fp32), the row-mode tiling
(single CTAs, CTA pairs, small token blocks) and sometimes the shared expert;
it then checks the inference forward, the training forward and the backward
elementwise within |gpu - ref| <= 1e-2 + 2e-2 |ref|
[HyperMegaMoE §7.1, §7.2: shapes, dtypes and routings beyond the named
configurations, each against the reference].

A second set (test_random_large_shape_matches_oracle) draws larger shapes: H
up to 1024 and I up to 768, so every tiling runs several weight tiles along
the MMA's M side and several token blocks per expert.

The family is that of the five workloads (K >= 2, I >= 64).  Outside it the
16-bit storage the bound allows for can exceed the bound by itself: with
I = 24 and the shared expert one y element came out at 1.14x (fp64 with only
the SwiGLU output rounded to bf16 reproduces the GPU value to 2e-5), with
K = 1 (unit routing weights) and H / I = 4.8 one weight-gradient element at
1.07x.
"""
import numpy as np
import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import moe_inputs as mi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return gu.Runner()


def _case(i, large=False):
    seed = (9500 if large else 9000) + i
    r = np.random.default_rng(seed)
    if large:
        T = int(r.integers(300, 1201))
        H = 8 * int(r.integers(64, 129))
        I = 8 * int(r.integers(48, 97))
        E = int(r.integers(2, 25))
        K = int(r.integers(2, 7))
    else:
        T = int(r.integers(1, 901))
        H = 8 * int(r.integers(1, 65))
        I = 8 * int(r.integers(8, 49))
        E = int(r.integers(1, 49))
        K = int(r.integers(2, 9))
    repeats = K > E or r.random() < 0.5
    if repeats:
        # a random subset of the experts is used (others stay empty), repeats allowed
        used = r.choice(E, size=int(r.integers(1, E + 1)), replace=False)
        ids = used[r.integers(0, used.size, size=(T, K))].astype(np.int32)
    else:
        ids = None
    p = gu.problem(T, H, I, E, K, seed=seed, ids=ids)
    if ids is not None:
        lg = r.standard_normal((T, K)).astype(np.float32)
        ex = np.exp(lg - lg.max(axis=1, keepdims=True))
        p.w = mi.f32_to_bf16_bits(ex / ex.sum(axis=1, keepdims=True))
    wdt = "f32" if r.random() < 0.3 else "bf16"
    mode = [0, 1, 3][i % 3]
    shared = K < 32 and r.random() < 0.25
    if shared:
        p.Ws1 = mi.normal_bf16(mi._rng(seed, 8), (H, 2 * I), 1.0 / np.sqrt(H))
        p.Ws2 = mi.normal_bf16(mi._rng(seed, 9), (I, H), 1.0 / np.sqrt(I))
    return p, wdt, mode, shared


N_LARGE = 18


def _id(i, large=False):
    p, wdt, mode, shared = _case(i, large)
    return (f"{i}-T{p.T}-H{p.H}-I{p.I}-E{p.E}-K{p.K}-{wdt}-{['cta', 'pair', '', 'small'][mode]}"
            + ("-shared" if shared else ""))


@pytest.mark.parametrize("i", range(N_CASES), ids=_id)
def test_random_shape_matches_oracle(run, i):
    _check(run, *_case(i))


@pytest.mark.parametrize("i", range(N_LARGE), ids=lambda i: _id(i, True))
def test_random_large_shape_matches_oracle(run, i):
    _check(run, *_case(i, True))


def _check(run, p, wdt, mode, shared):
    d = gu.upload(p, weights_dtype=wdt)
    c = run.ctx
    hmm.hmm_set_option(c.handle, hmm.HMM_OPT_PAIR_ROWS, mode)
    try:
        kw = {}
        if shared:
            kw = dict(Ws1=gu.bf16(p.Ws1), Ws2=gu.bf16(p.Ws2))
        y, saved = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=True, **kw)
        yi, _ = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=False, **kw)
        outs = c.backward(d.dy, d.x, d.ids, d.w, d.W1, d.W2, saved, **kw)
        torch.cuda.synchronize()
        # fp32 routing weights are the same bf16 values widened: the oracle reads those
        w_ref = p.w
        ref = oracle.forward(p.x, p.ids, w_ref, p.W1, p.W2)
        rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, w_ref, p.W1, p.W2, p.dy)
        if shared:
            ref = ref + oracle.shared_forward(p.x, p.Ws1, p.Ws2)
            sdx, sdW1, sdW2 = oracle.shared_backward(p.x, p.Ws1, p.Ws2, p.dy)
            rdx = rdx + sdx
        gu.check("y", gu.f64(y), ref)
        gu.check("y (inference)", gu.f64(yi), ref)
        gu.check("dx", gu.f64(outs[0]), rdx)
        gu.check("d_up_proj_weight", gu.f64(outs[1]), rdW1)
        gu.check("d_down_proj_weight", gu.f64(outs[2]), rdW2)
        gu.check("d_topk_weights", gu.f64(outs[3]), rdw)
        if shared:
            gu.check("d_shared_up_proj_weight", gu.f64(outs[4]), sdW1)
            gu.check("d_shared_down_proj_weight", gu.f64(outs[5]), sdW2)
        counts = np.bincount(p.ids.reshape(-1), minlength=p.E)
        for e in np.nonzero(counts == 0)[0]:
            assert not gu.f64(outs[1][e]).any() and not gu.f64(outs[2][e]).any()
        assert run.status() == (0, 0)
    finally:
        hmm.hmm_set_option(c.handle, hmm.HMM_OPT_PAIR_ROWS, 2)

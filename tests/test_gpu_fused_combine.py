"""The combine folded into the GMM2 epilogue (HMM_OPT_FUSED_COMBINE) vs the
separate combine kernel and the fp64 oracle, through the C ABI
[HyperMegaMoE §6.2: permute/unpermute fused into the operator; MoE overlap
explainer §6: per-token completion counts, publish once every branch is in,
deterministic merge order].

- y is bit-identical to the separate combine (the same fp32 operations in the
  same k order, one bf16 rounding), and within the tolerance of the oracle;
- on single CTAs, CTA pairs and small token blocks, training and inference;
- edge cases: empty and hot experts, repeated experts in a token, zero
  routing weights, ragged sizes, one token, fp32 routing weights, and the
  optional shared expert (K + 1 rows per token, fp32 expert outputs);
- repeated calls stay bit-identical (the counters are zeroed every call), and
  a backward after a fused forward is unchanged.
"""
import numpy as np
import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import moe_inputs as mi
import oracle
from tests import gpu_util as gu
from tests.test_gpu_parity import SCEN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return gu.Runner()


@pytest.fixture(params=[0, 1, 3], ids=["cta", "pair", "small"])
def rows_mode(run, request):
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, request.param)
    yield request.param
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, 2)


def _fused(run, on):
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_FUSED_COMBINE, 1 if on else 0)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


CASES = [c for c in SCEN if c[0] in ("multi_tile", "empty_and_hot", "duplicates", "zero_weights",
                                     "one_token", "ragged_small", "single_hot", "tiny_config")]


@pytest.mark.parametrize("training", [True, False])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_fused_combine_bit_identical_and_matches_oracle(run, case, training, rows_mode):
    _, p = case
    d = gu.upload(p)
    try:
        _fused(run, False)
        y_sep, _ = run.forward(d, training=training)
        _fused(run, True)
        y_f, _ = run.forward(d, training=training)
        y_f2, _ = run.forward(d, training=training)
        torch.cuda.synchronize()
    finally:
        _fused(run, False)
    assert torch.equal(_bits(y_f), _bits(y_sep))
    assert torch.equal(_bits(y_f2), _bits(y_sep))
    gu.check("y (fused combine)", gu.f64(y_f), oracle.forward(p.x, p.ids, p.w, p.W1, p.W2))
    assert run.status() == (0, 0)


def test_fused_combine_fp32_weights_and_backward(run):
    p = gu.problem(96, 128, 64, 6, 3, seed=21)
    d = gu.upload(p, weights_dtype="f32")
    try:
        _fused(run, False)
        y_sep, saved_sep = run.forward(d)
        g_sep = run.backward(d, saved_sep)
        _fused(run, True)
        y_f, saved_f = run.forward(d)
        g_f = run.backward(d, saved_f)
        torch.cuda.synchronize()
    finally:
        _fused(run, False)
    assert torch.equal(_bits(y_f), _bits(y_sep))
    for a, b in zip(g_sep, g_f):
        assert torch.equal(_bits(a), _bits(b))
    gu.check("y", gu.f64(y_f), oracle.forward(p.x, p.ids, p.w, p.W1, p.W2))


def _with_shared(p, seed):
    p.Ws1 = mi.normal_bf16(mi._rng(seed, 8), (p.H, 2 * p.I), 1.0 / np.sqrt(p.H))
    p.Ws2 = mi.normal_bf16(mi._rng(seed, 9), (p.I, p.H), 1.0 / np.sqrt(p.I))
    return p


@pytest.mark.parametrize("case", ["multi_tile", "empty_and_hot", "one_token"])
def test_fused_combine_with_shared_expert(run, case, rows_mode):
    p = _with_shared(dict(SCEN)[case], 31)
    d = gu.upload(p)
    Ws1, Ws2 = gu.bf16(p.Ws1), gu.bf16(p.Ws2)
    c = run.ctx
    try:
        _fused(run, False)
        y_sep, _ = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=True, Ws1=Ws1, Ws2=Ws2)
        _fused(run, True)
        y_f, _ = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=True, Ws1=Ws1, Ws2=Ws2)
        yi_f, _ = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=False, Ws1=Ws1, Ws2=Ws2)
        torch.cuda.synchronize()
    finally:
        _fused(run, False)
    assert torch.equal(_bits(y_f), _bits(y_sep))
    assert torch.equal(_bits(yi_f), _bits(y_sep))
    ref = oracle.forward(p.x, p.ids, p.w, p.W1, p.W2) + oracle.shared_forward(p.x, p.Ws1, p.Ws2)
    gu.check("y (fused combine, shared expert)", gu.f64(y_f), ref)
    assert run.status() == (0, 0)

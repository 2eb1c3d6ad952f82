"""GPU path with the optional shared expert [HyperMegaMoE §6.1] vs the fp64
oracle, through the C ABI (hmm_forward_shared / hmm_backward_shared):

- y = routed combine + FFN_s(x) (every token, unit weight);
- dx (routed + shared parts), d_up_proj_weight, d_down_proj_weight,
  d_topk_weights, d_shared_up_proj_weight, d_shared_down_proj_weight;
- elementwise |gpu - ref| <= 1e-2 + 2e-2 |ref|, on single CTAs and on CTA
  pairs, with empty, hot and ragged routings;
- the entry points refuse a shape whose shared flag does not match them.
"""
import numpy as np
import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import moe_inputs as mi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return gu.Runner()


def _with_shared(p, seed):
    p.Ws1 = mi.normal_bf16(mi._rng(seed, 8), (p.H, 2 * p.I), 1.0 / np.sqrt(p.H))
    p.Ws2 = mi.normal_bf16(mi._rng(seed, 9), (p.I, p.H), 1.0 / np.sqrt(p.I))
    return p


def _cases():
    yield "tiny", _with_shared(gu.problem(64, 128, 64, 8, 2, seed=1000), 1000)
    base = gu.problem(300, 264, 200, 10, 3, seed=11)
    yield "ragged", _with_shared(base, 11)
    ids = base.ids.copy()
    ids[np.isin(ids, [2, 5, 7])] = 0          # empty experts, one hot
    for t in range(ids.shape[0]):
        seen = set()
        for k in range(ids.shape[1]):
            if ids[t, k] in seen:
                ids[t, k] = [e for e in (1, 3, 4, 6, 8, 9) if e not in seen][0]
            seen.add(int(ids[t, k]))
    yield "empty_and_hot", _with_shared(gu.problem(300, 264, 200, 10, 3, seed=11, ids=ids), 12)
    g = np.log([5, 3, 2, 1, 1, 0.5]) + np.random.default_rng(15).gumbel(size=(700, 6))
    yield "multi_tile", _with_shared(
        gu.problem(700, 264, 200, 6, 4, seed=14, ids=np.argsort(-g, axis=1)[:, :4].astype(np.int32)), 14)
    yield "one_token", _with_shared(gu.problem(1, 128, 64, 4, 2, seed=12), 13)


CASES = list(_cases())


@pytest.fixture(params=[0, 1, 3], ids=["cta", "pair", "small"])
def rows_mode(run, request):
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, request.param)
    yield request.param
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, 2)


def _upload(p):
    d = gu.upload(p)
    d.Ws1 = gu.bf16(p.Ws1)
    d.Ws2 = gu.bf16(p.Ws2)
    return d


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_shared_forward_backward_match_oracle(run, case, rows_mode):
    _, p = case
    d = _upload(p)
    c = run.ctx
    y, saved = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=True, Ws1=d.Ws1, Ws2=d.Ws2)
    yi, _ = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=False, Ws1=d.Ws1, Ws2=d.Ws2)
    dx, dW1, dW2, dw, dWs1, dWs2 = c.backward(d.dy, d.x, d.ids, d.w, d.W1, d.W2, saved,
                                              Ws1=d.Ws1, Ws2=d.Ws2)
    torch.cuda.synchronize()
    ys = oracle.shared_forward(p.x, p.Ws1, p.Ws2)
    ref = oracle.forward(p.x, p.ids, p.w, p.W1, p.W2) + ys
    gu.check("y", gu.f64(y), ref)
    gu.check("y (inference)", gu.f64(yi), ref)
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    sdx, sdW1, sdW2 = oracle.shared_backward(p.x, p.Ws1, p.Ws2, p.dy)
    gu.check("dx", gu.f64(dx), rdx + sdx)
    gu.check("d_topk_weights", gu.f64(dw), rdw)
    gu.check("d_up_proj_weight", gu.f64(dW1), rdW1)
    gu.check("d_down_proj_weight", gu.f64(dW2), rdW2)
    gu.check("d_shared_up_proj_weight", gu.f64(dWs1), sdW1)
    gu.check("d_shared_down_proj_weight", gu.f64(dWs2), sdW2)
    assert run.status() == (0, 0)


def test_shared_flag_must_match_the_entry_point(run):
    p = CASES[0][1]
    d = _upload(p)
    sh = run.shape(d)                      # shared = 0
    fwd, sv, _ = hmm.hmm_workspace_size(sh, True)
    y = torch.empty_like(d.x)
    ws = torch.empty(fwd, dtype=torch.uint8, device=gu.dev())
    saved = torch.empty(sv, dtype=torch.uint8, device=gu.dev())
    with pytest.raises(hmm.HmmError):
        hmm.hmm_forward_shared(run.ctx.handle, sh, d.x, d.ids, d.w, d.W1, d.W2, d.Ws1, d.Ws2,
                               y, saved, ws)
    sh1 = hmm.make_shape(sh.T, sh.H, sh.I, sh.E, sh.K, sh.weights_dtype, shared=1)
    fwd1, sv1, bwd1 = hmm.hmm_workspace_size(sh1, True)
    assert fwd1 > fwd and sv1 > sv         # the shared expert's rows
    ws1 = torch.empty(fwd1, dtype=torch.uint8, device=gu.dev())
    saved1 = torch.empty(sv1, dtype=torch.uint8, device=gu.dev())
    with pytest.raises(hmm.HmmError):
        hmm.hmm_forward(run.ctx.handle, sh1, d.x, d.ids, d.w, d.W1, d.W2, y, saved1, ws1)
    with pytest.raises(hmm.HmmError):       # the shared weights are required
        hmm.hmm_forward_shared(run.ctx.handle, sh1, d.x, d.ids, d.w, d.W1, d.W2, None, d.Ws2,
                               y, saved1, ws1)
    bw = torch.empty(bwd1, dtype=torch.uint8, device=gu.dev())
    with pytest.raises(hmm.HmmError):       # the split entry points serve shared == 0
        hmm.hmm_backward_dx(run.ctx.handle, sh1, d.dy, d.w, d.W1, d.W2, saved1,
                            torch.empty_like(d.x), None, bw)
    torch.cuda.synchronize()
    assert run.status() == (0, 0)


def test_shared_autograd(run):
    p = CASES[1][1]
    d = _upload(p)
    leaves = [t.clone().requires_grad_(True) for t in (d.x, d.w, d.W1, d.W2, d.Ws1, d.Ws2)]
    x, w, W1, W2, Ws1, Ws2 = leaves
    y = hmm.moe_ffn(x, d.ids, w, W1, W2, shared_up_proj_weight=Ws1, shared_down_proj_weight=Ws2)
    y.backward(d.dy)
    torch.cuda.synchronize()
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    sdx, sdW1, sdW2 = oracle.shared_backward(p.x, p.Ws1, p.Ws2, p.dy)
    gu.check("x.grad", gu.f64(x.grad), rdx + sdx)
    gu.check("w.grad", gu.f64(w.grad), rdw)
    gu.check("Ws1.grad", gu.f64(Ws1.grad), sdW1)
    gu.check("Ws2.grad", gu.f64(Ws2.grad), sdW2)

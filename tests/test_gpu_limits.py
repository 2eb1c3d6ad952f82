"""The GPU path at the documented limits, against the fp64 oracle:
E = 1024 experts and K = 32 slots per token (the routing scan's 1024 threads,
the dispatch warp's 32 slot lanes, the longest schedule), and the same with
the shared expert (E + 1 = 1024, K + 1 = 32).  Small H and I keep the oracle
fast; routing, forward and every gradient are checked."""
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


def _check_all(run, p, shared):
    d = gu.upload(p)
    c = run.ctx
    kw = {}
    if shared:
        d.Ws1, d.Ws2 = gu.bf16(p.Ws1), gu.bf16(p.Ws2)
        kw = dict(Ws1=d.Ws1, Ws2=d.Ws2)
    y, saved = c.forward(d.x, d.ids, d.w, d.W1, d.W2, training=True, **kw)
    grads = c.backward(d.dy, d.x, d.ids, d.w, d.W1, d.W2, saved, **kw)
    torch.cuda.synchronize()
    ref = oracle.forward(p.x, p.ids, p.w, p.W1, p.W2)
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    if shared:
        ref = ref + oracle.shared_forward(p.x, p.Ws1, p.Ws2)
        sdx, sdW1, sdW2 = oracle.shared_backward(p.x, p.Ws1, p.Ws2, p.dy)
        rdx = rdx + sdx
    gu.check("y", gu.f64(y), ref)
    gu.check("dx", gu.f64(grads[0]), rdx)
    gu.check("d_up_proj_weight", gu.f64(grads[1]), rdW1)
    gu.check("d_down_proj_weight", gu.f64(grads[2]), rdW2)
    gu.check("d_topk_weights", gu.f64(grads[3]), rdw)
    if shared:
        gu.check("d_shared_up_proj_weight", gu.f64(grads[4]), sdW1)
        gu.check("d_shared_down_proj_weight", gu.f64(grads[5]), sdW2)
    assert run.status() == (0, 0)


def _limits_problem(E, K, seed):
    T, H, I = 1024, 64, 64
    r = np.random.default_rng(seed)
    ids = np.argsort(r.random((T, E)), axis=1)[:, :K].astype(np.int32)  # K distinct of E
    return gu.problem(T, H, I, E, K, seed=seed, ids=ids)


def test_max_experts_and_slots(run):
    p = _limits_problem(1024, 32, 21)
    counts = np.bincount(p.ids.reshape(-1), minlength=1024)
    assert counts.min() > 0                  # every expert has rows at this size
    got = [t.cpu().numpy() for t in _route(run, p)]
    for name, g, r in zip(("counts", "offsets", "slot2row", "row2slot"), got,
                          oracle.route(p.ids, 1024)):
        np.testing.assert_array_equal(g[: r.size], r, err_msg=name)
    _check_all(run, p, shared=False)


def test_max_experts_and_slots_with_shared_expert(run):
    p = _limits_problem(1023, 31, 22)
    p.Ws1 = mi.normal_bf16(mi._rng(22, 8), (p.H, 2 * p.I), 1.0 / np.sqrt(p.H))
    p.Ws2 = mi.normal_bf16(mi._rng(22, 9), (p.I, p.H), 1.0 / np.sqrt(p.I))
    _check_all(run, p, shared=True)


def test_beyond_limits_refused_on_host(run):
    for E, K, shared in ((1025, 2, 0), (8, 33, 0), (1024, 2, 1), (8, 32, 1)):
        sh = hmm.make_shape(16, 64, 64, E, K, shared=shared)
        with pytest.raises(hmm.HmmError):
            hmm.hmm_workspace_size(sh, True)


def _route(run, p):
    sh = hmm.make_shape(p.T, p.H, p.I, p.E, p.K)
    fwd, _, _ = hmm.hmm_workspace_size(sh, False)
    dev = gu.dev()
    ids = torch.from_numpy(p.ids).to(dev)
    out = (torch.empty(p.E, dtype=torch.int32, device=dev),
           torch.empty(p.E + 1, dtype=torch.int32, device=dev),
           torch.empty(p.T * p.K, dtype=torch.int32, device=dev),
           torch.empty(p.T * p.K, dtype=torch.int32, device=dev))
    ws = torch.empty(fwd, dtype=torch.uint8, device=dev)
    hmm.hmm_route(run.ctx.handle, sh, ids, *out, ws)
    torch.cuda.synchronize()
    return out

"""Forward + backward captured in a CUDA graph and replayed.

A training step that launches the same fixed-shape kernels every iteration
can be captured once and replayed, which takes the host's per-launch work off
the step.  The library's calls qualify: they allocate nothing, synchronise
nothing (with HMM_OPT_VALIDATE and HMM_OPT_PROFILE off), reset their own
counters in every call [HyperMegaMoE §5.3: no stale event state across
iterations], and the backward's second stream (the dx combine beside the
weight gradients) joins the capture through its fork and join events.
The replays must write what eager calls write, bit for bit, including after
the inputs are overwritten in place between replays.
"""
import numpy as np
import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return gu.Runner()


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("pair_rows", [0, 1, 3])
def test_capture_and_replay_fwd_bwd(run, pair_rows):
    h = run.ctx.handle
    hmm.hmm_set_option(h, hmm.HMM_OPT_PAIR_ROWS, pair_rows)
    try:
        p = gu.problem(300, 264, 200, 10, 3, seed=11)
        d = gu.upload(p)
        sh = run.shape(d)
        fwd, sv, bwd = hmm.hmm_workspace_size(sh, True)
        dev = gu.dev()
        ws_f = torch.empty(fwd, dtype=torch.uint8, device=dev)
        saved = torch.empty(sv, dtype=torch.uint8, device=dev)
        ws_b = torch.empty(bwd, dtype=torch.uint8, device=dev)
        y = torch.empty_like(d.x)
        dx = torch.empty_like(d.x)
        dW1 = torch.empty_like(d.W1)
        dW2 = torch.empty_like(d.W2)
        dw = torch.empty_like(d.w)

        def step():
            hmm.hmm_forward(h, sh, d.x, d.ids, d.w, d.W1, d.W2, y, saved, ws_f)
            hmm.hmm_backward(h, sh, d.dy, d.w, d.W1, d.W2, saved, dx, dW1, dW2, dw, ws_b)

        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()                                    # eager, on the capture stream
        torch.cuda.synchronize()
        eager = [t.clone() for t in (y, dx, dW1, dW2, dw)]

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for t in (y, dx, dW1, dW2, dw):
            t.fill_(float("nan"))                     # the replay must write every element
        g.replay()
        torch.cuda.synchronize()
        for name, a, b in zip(("y", "dx", "dW1", "dW2", "d_topk_weights"), eager,
                              (y, dx, dW1, dW2, dw)):
            assert torch.equal(_bits(a), _bits(b)), name

        # new inputs written in place: the replay computes on them
        q = gu.problem(300, 264, 200, 10, 3, seed=12)
        d.x.copy_(gu.bf16(q.x))
        d.ids.copy_(torch.from_numpy(q.ids).to(dev))
        d.w.copy_(gu.bf16(q.w))
        d.dy.copy_(gu.bf16(q.dy))
        g.replay()
        g.replay()                                    # twice: no state carried over
        torch.cuda.synchronize()
        ry = oracle.forward(q.x, q.ids, q.w, p.W1, p.W2)
        rdx, rdW1, rdW2, rdw = oracle.backward(q.x, q.ids, q.w, p.W1, p.W2, q.dy)
        gu.check("y (replay)", gu.f64(y), ry)
        gu.check("dx (replay)", gu.f64(dx), rdx)
        gu.check("d_up_proj_weight (replay)", gu.f64(dW1), rdW1)
        gu.check("d_down_proj_weight (replay)", gu.f64(dW2), rdW2)
        gu.check("d_topk_weights (replay)", gu.f64(dw), rdw)
        del g
        assert run.status() == (0, 0)
    finally:
        hmm.hmm_set_option(h, hmm.HMM_OPT_PAIR_ROWS, 2)

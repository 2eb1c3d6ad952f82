"""Failure detection without a GPU fault: a bounded device wait that runs out.

The fault is injected on the host (HMM_OPT_INJECT_SKIP_READY): the GMM1 tiles
of one forward skip the release of their ready counters, so every GMM2 tile's
acquire-poll runs out of its (shortened) budget.  The kernel must record
HMM_STATUS_TIMEOUT, leave cleanly (no trap, no hang), and the context must be
usable again: the next call gives the oracle's result [HyperMegaMoE §5.3: no
stale event state after failures; §7.3: failures diagnosable, no deadlock]."""
import time

import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_next_call_recovers():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    run = gu.Runner()
    p = gu.problem(300, 264, 200, 10, 3, seed=11)
    d = gu.upload(p)
    run.ctx.set_option(hmm.HMM_OPT_WAIT_BUDGET_NS, 50_000_000)    # 50 ms
    run.ctx.set_option(hmm.HMM_OPT_INJECT_SKIP_READY, 1)
    try:
        t0 = time.perf_counter()
        run.forward(d)
        rc, bits = run.status()
        elapsed = time.perf_counter() - t0
    finally:
        run.ctx.set_option(hmm.HMM_OPT_INJECT_SKIP_READY, 0)
        run.ctx.set_option(hmm.HMM_OPT_WAIT_BUDGET_NS, 2_000_000_000)
    assert rc == hmm.HMM_ERR_TIMEOUT and bits & hmm.HMM_STATUS_TIMEOUT
    assert elapsed < 20.0
    assert run.status() == (0, 0)                  # cleared by the read
    y, saved = run.forward(d)                       # the context still works
    dx, dW1, dW2, dw = run.backward(d, saved)
    torch.cuda.synchronize()
    assert run.status() == (0, 0)
    gu.check("y", gu.f64(y), oracle.forward(p.x, p.ids, p.w, p.W1, p.W2))
    rdx, _, _, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("dx", gu.f64(dx), rdx)
    gu.check("dw", gu.f64(dw), rdw)

"""Failure detection without a GPU fault: a bounded device wait that runs out.

The fault is injected on the host (HMM_OPT_INJECT_SKIP_READY): the producer
tiles of one launch skip the release of their ready counters, so every
consumer tile's acquire-poll runs out of its (shortened) budget.
- forward: GMM1 tiles do not release, GMM2 tiles wait;
- backward: act_grad tiles do not release, input-grad tiles wait (the
  weight-gradient launch after it then sees the timeout bit and leaves early
  too).
Each runs on single CTAs, on CTA pairs (whose teardown drains both CTAs'
copies in flight) and on single CTAs with small token blocks.  The kernels
must record HMM_STATUS_TIMEOUT, leave cleanly (no trap, no hang), and the
context must be usable again: the next calls give the oracle's results
[HyperMegaMoE §5.3: no stale event state after failures; §7.3: failures
diagnosable, no deadlock]."""
import time

import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 3], ids=["cta", "pair", "small"])
@pytest.mark.parametrize("where", ["forward", "backward"])
def test_bounded_wait_times_out_and_next_call_recovers(where, mode):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    run = gu.Runner()
    p = gu.problem(300, 264, 200, 10, 3, seed=11)
    d = gu.upload(p)
    run.ctx.set_option(hmm.HMM_OPT_PAIR_ROWS, mode)
    try:
        saved = None
        if where == "backward":
            y, saved = run.forward(d)
            torch.cuda.synchronize()
            assert run.status() == (0, 0)
        run.ctx.set_option(hmm.HMM_OPT_WAIT_BUDGET_NS, 50_000_000)    # 50 ms
        run.ctx.set_option(hmm.HMM_OPT_INJECT_SKIP_READY, 1 if where == "forward" else 2)
        try:
            t0 = time.perf_counter()
            if where == "forward":
                run.forward(d)
            else:
                run.backward(d, saved)
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
    finally:
        run.ctx.set_option(hmm.HMM_OPT_PAIR_ROWS, 2)
    gu.check("y", gu.f64(y), oracle.forward(p.x, p.ids, p.w, p.W1, p.W2))
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("dx", gu.f64(dx), rdx)
    gu.check("dw", gu.f64(dw), rdw)
    gu.check("dW1", gu.f64(dW1), rdW1)
    gu.check("dW2", gu.f64(dW2), rdW2)


def test_inject_option_range():
    """Host-side validation of the injection option (no device work)."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    run = gu.Runner()
    with pytest.raises(hmm.HmmError):
        run.ctx.set_option(hmm.HMM_OPT_INJECT_SKIP_READY, 3)

"""The per-tile GEMM timeline (hmm_set_trace): records appear for every tile
of the traced launch, time stamps are ordered along the tile's pipeline, and
the results of a traced call are unchanged."""
import numpy as np
import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
from dispatch_grouped_gemm_gb300 import trace as tr
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1, 2])
def test_trace_records_every_tile(which):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    run = gu.Runner()
    p = gu.problem(300, 264, 200, 10, 3, seed=11)
    d = gu.upload(p)
    y0, saved = run.forward(d)
    g0 = run.backward(d, saved)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(sms * 8 * 64, dtype=torch.int64, device=gu.dev())
    hmm.hmm_set_trace(run.ctx.handle, buf, which)
    try:
        y1, saved = run.forward(d)
        g1 = run.backward(d, saved)
        torch.cuda.synchronize()
    finally:
        hmm.hmm_set_trace(run.ctx.handle, None, 0)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    for a, b in zip(g0, g1):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    t = tr.decode(buf.cpu().numpy().view(np.uint64), sms)
    assert t.size > 0
    # tiles that ran the full pipeline: scheduled <= loads <= MMAs <= epilogue
    full = t[(t["kb"] > 0) & (t["epi1"] > 0)]
    assert full.size > 0
    assert (full["sched"] <= full["load0"]).all() and (full["load0"] <= full["load1"]).all()
    assert (full["mma0"] <= full["mma1"]).all() and (full["mma1"] <= full["epi0"]).all()
    assert (full["epi0"] <= full["epi1"]).all()
    s = tr.summarize(t)
    assert s["tiles"] == t.size and s["span_us"] > 0

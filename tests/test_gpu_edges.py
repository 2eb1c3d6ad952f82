"""More degenerate shapes on the GPU path, against the fp64 oracle, on single
CTAs and on CTA pairs: the smallest hidden and intermediate sizes (H = I = 8,
one 16-byte group per row, TMA boxes wider than the tensor), a single expert
with one slot per token (E = 1, K = 1, many 128-row tiles), one slot per token
over many experts, and fp32 routing weights with the shared expert."""
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


@pytest.fixture(params=[0, 1, 3], ids=["cta", "pair", "small"])
def rows_mode(run, request):
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, request.param)
    yield request.param
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, 2)


def _cases():
    yield "H8_I8", gu.problem(300, 8, 8, 5, 3, seed=31)
    yield "E1_K1", gu.problem(700, 136, 72, 1, 1, seed=32)
    r = np.random.default_rng(33)
    yield "K1_E40", gu.problem(500, 64, 40, 40, 1, seed=33,
                               ids=r.integers(0, 40, size=(500, 1)).astype(np.int32))


CASES = list(_cases())


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_edge_shapes_match_oracle(run, case, rows_mode):
    _, p = case
    d = gu.upload(p)
    y, saved = run.forward(d)
    yi, _ = run.forward(d, training=False)
    dx, dW1, dW2, dw = run.backward(d, saved)
    torch.cuda.synchronize()
    ref = oracle.forward(p.x, p.ids, p.w, p.W1, p.W2)
    gu.check("y", gu.f64(y), ref)
    gu.check("y (inference)", gu.f64(yi), ref)
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("dx", gu.f64(dx), rdx)
    gu.check("d_up_proj_weight", gu.f64(dW1), rdW1)
    gu.check("d_down_proj_weight", gu.f64(dW2), rdW2)
    gu.check("d_topk_weights", gu.f64(dw), rdw)
    assert run.status() == (0, 0)


def test_fp32_weights_with_shared_expert(run):
    p = gu.problem(96, 128, 64, 6, 3, seed=34)
    p.Ws1 = mi.normal_bf16(mi._rng(34, 8), (p.H, 2 * p.I), 1.0 / np.sqrt(p.H))
    p.Ws2 = mi.normal_bf16(mi._rng(34, 9), (p.I, p.H), 1.0 / np.sqrt(p.I))
    d = gu.upload(p, weights_dtype="f32")
    Ws1, Ws2 = gu.bf16(p.Ws1), gu.bf16(p.Ws2)
    y, saved = run.ctx.forward(d.x, d.ids, d.w, d.W1, d.W2, training=True, Ws1=Ws1, Ws2=Ws2)
    dx, dW1, dW2, dw, dWs1, dWs2 = run.ctx.backward(d.dy, d.x, d.ids, d.w, d.W1, d.W2, saved,
                                                    Ws1=Ws1, Ws2=Ws2)
    torch.cuda.synchronize()
    assert dw.dtype == torch.float32
    wf = mi.bf16_bits_to_f32(p.w).astype(np.float64)   # the fp32 weights the GPU saw
    x64 = mi.bf16_bits_to_f32(p.x).astype(np.float64)
    W1, W2, dy = (mi.bf16_bits_to_f32(a).astype(np.float64) for a in (p.W1, p.W2, p.dy))
    S1, S2 = (mi.bf16_bits_to_f32(a).astype(np.float64) for a in (p.Ws1, p.Ws2))
    ref = oracle.forward(x64, p.ids, wf, W1, W2) + oracle.shared_forward(x64, S1, S2)
    gu.check("y", gu.f64(y), ref)
    rdx, _, _, rdw = oracle.backward(x64, p.ids, wf, W1, W2, dy)
    sdx, sdW1, sdW2 = oracle.shared_backward(x64, S1, S2, dy)
    gu.check("dx", gu.f64(dx), rdx + sdx)
    gu.check("d_topk_weights", dw.double().cpu().numpy(), rdw)
    gu.check("d_shared_up_proj_weight", gu.f64(dWs1), sdW1)
    gu.check("d_shared_down_proj_weight", gu.f64(dWs2), sdW2)
    assert run.status() == (0, 0)


@pytest.mark.parametrize("pair_rows", [0, 1, 3], ids=["cta", "pair", "small"])
@pytest.mark.parametrize("case", ["multi_tile", "empty_and_hot", "one_token", "duplicates"])
def test_buffers_full_of_nan_bytes(run, case, pair_rows):
    """Workspace and `saved` filled with 0xFF bytes (NaN as bf16 and fp32)
    before every call: the kernels write every byte they later read (the
    padding rows up to each expert's last 64-row block when training, none in
    inference), so the outputs match the oracle and stay finite."""
    from tests.test_gpu_parity import SCEN
    p = dict(SCEN)[case]
    d = gu.upload(p)
    h = run.ctx.handle
    hmm.hmm_set_option(h, hmm.HMM_OPT_PAIR_ROWS, pair_rows)
    try:
        sh = run.shape(d)
        dev = gu.dev()
        ref_y = oracle.forward(p.x, p.ids, p.w, p.W1, p.W2)
        for training in (False, True):
            fwd, sv, bwd = hmm.hmm_workspace_size(sh, training)
            ws = torch.full((max(fwd, 16),), 255, dtype=torch.uint8, device=dev)
            saved = torch.full((max(sv, 16),), 255, dtype=torch.uint8, device=dev) if training else None
            y = torch.empty_like(d.x)
            hmm.hmm_forward(h, sh, d.x, d.ids, d.w, d.W1, d.W2, y, saved, ws)
            torch.cuda.synchronize()
            gu.check(f"y (training={training})", gu.f64(y), ref_y)
        wsb = torch.full((bwd,), 255, dtype=torch.uint8, device=dev)
        dx = torch.empty_like(d.x)
        dW1 = torch.full_like(d.W1, float("nan"))
        dW2 = torch.full_like(d.W2, float("nan"))
        dw = torch.empty_like(d.w)
        hmm.hmm_backward(h, sh, d.dy, d.w, d.W1, d.W2, saved, dx, dW1, dW2, dw, wsb)
        torch.cuda.synchronize()
        rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
        gu.check("dx", gu.f64(dx), rdx)
        gu.check("d_up_proj_weight", gu.f64(dW1), rdW1)
        gu.check("d_down_proj_weight", gu.f64(dW2), rdW2)
        gu.check("d_topk_weights", gu.f64(dw), rdw)
        assert run.status() == (0, 0)
    finally:
        hmm.hmm_set_option(h, hmm.HMM_OPT_PAIR_ROWS, 2)

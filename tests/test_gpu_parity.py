"""GPU path vs the fp64 oracle, through the C ABI.

- routing metadata: bit-exact (counts, offsets, stable permutation, inverse);
- forward y and backward dx, d_up_proj_weight, d_down_proj_weight,
  d_topk_weights: elementwise |gpu - ref| <= 1e-2 + 2e-2 |ref|;
- edge cases the HyperMegaMoE test plan lists (§7.2): empty experts, one hot
  expert, repeated experts inside a token, zero routing weights, ragged token
  counts, tiles not dividing H or I, a single token, fp32 routing weights;
- repeated calls are bit-identical (no stale counters across iterations, §5.3);
- an out-of-range expert id is reported, never clamped (§4.2).
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


def _route_gpu(run, ids_np, E):
    T, K = ids_np.shape
    sh = hmm.make_shape(T, 8, 8, E, K)
    fwd, _, _ = hmm.hmm_workspace_size(sh, False)
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(gu.dev())
    counts = torch.empty(E, dtype=torch.int32, device=gu.dev())
    offsets = torch.empty(E + 1, dtype=torch.int32, device=gu.dev())
    s2r = torch.empty(max(1, T * K), dtype=torch.int32, device=gu.dev())
    r2s = torch.empty(max(1, T * K), dtype=torch.int32, device=gu.dev())
    ws = torch.empty(fwd, dtype=torch.uint8, device=gu.dev())
    hmm.hmm_route(run.ctx.handle, sh, ids, counts, offsets, s2r, r2s, ws)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (counts, offsets, s2r, r2s)]


def _routing_cases():
    r = np.random.default_rng(5)
    yield "tiny", mi.make("tiny").topk_ids, 8
    yield "prefill", mi.make("prefill").topk_ids, 64
    yield "skewed", mi.make("skewed").topk_ids, 32
    yield "decode", mi.make("decode").topk_ids, 256
    yield "repeats", r.integers(0, 5, size=(3001, 7)).astype(np.int32), 5
    ids = r.integers(0, 40, size=(777, 4)).astype(np.int32)
    ids[ids % 3 == 0] = 1           # many empty experts, one hot
    yield "empty_hot", ids, 40
    yield "one_slot", np.array([[3]], np.int32), 4
    yield "E1", np.zeros((100, 1), np.int32), 1
    # the scan inside the rank blocks at its limit (64 chunks x 512 experts),
    # and the separate scan launch past it (E > 512; 157 chunks x 256 experts)
    yield "fused_scan_limit", r.integers(0, 512, size=(8192, 8)).astype(np.int32), 512
    yield "scan_launch_wide_E", r.integers(0, 600, size=(3000, 6)).astype(np.int32), 600
    yield "scan_launch_many_chunks", r.integers(0, 256, size=(20000, 8)).astype(np.int32), 256


@pytest.mark.parametrize("case", list(_routing_cases()), ids=lambda c: c[0])
def test_routing_bit_exact(run, case):
    _, ids, E = case
    got = _route_gpu(run, ids, E)
    ref = oracle.route(ids, E)
    for name, g, r in zip(("counts", "offsets", "slot2row", "row2slot"), got, ref):
        np.testing.assert_array_equal(g[: r.size], r, err_msg=name)


# ---------------------------------------------------------------- forward

def _scenarios():
    T, H, I, E, K = 300, 264, 200, 10, 3
    base = gu.problem(T, H, I, E, K, seed=11)
    yield "uniform", base
    r = np.random.default_rng(3)
    ids = base.ids.copy()
    ids[np.isin(ids, [2, 5, 7])] = 0          # experts 2, 5, 7 empty; expert 0 hot
    for t in range(T):                          # keep K distinct where possible
        seen = set()
        for k in range(K):
            if ids[t, k] in seen:
                ids[t, k] = [e for e in (1, 3, 4, 6, 8, 9) if e not in seen][0]
            seen.add(int(ids[t, k]))
    yield "empty_and_hot", gu.problem(T, H, I, E, K, seed=11, ids=ids)
    hot = base.ids.copy()
    hot[:, 0] = 4                               # every token hits expert 4 (3 m-tiles)
    hot[:, 1] = np.where(hot[:, 1] == 4, 9, hot[:, 1])
    hot[:, 2] = np.where(hot[:, 2] == 4, 8, hot[:, 2])
    yield "single_hot", gu.problem(T, H, I, E, K, seed=11, ids=hot)
    dup = base.ids.copy()
    dup[::3, 1] = dup[::3, 0]                   # repeated expert inside a token
    yield "duplicates", gu.problem(T, H, I, E, K, seed=11, ids=dup)
    w0 = base.w.copy()
    w0[::2, 2] = 0                              # zero routing weights
    yield "zero_weights", gu.problem(T, H, I, E, K, seed=11, w=w0)
    yield "one_token", gu.problem(1, 128, 64, 4, 2, seed=12)
    yield "ragged_small", gu.problem(37, 136, 72, 6, 4, seed=13, ids=r.integers(0, 6, size=(37, 4)))
    yield "tiny_config", gu.problem(64, 128, 64, 8, 2, seed=1000)
    # skewed top-4 of 6 experts (Gumbel top-k): 6, 5, 5, 4, 3 and 2 tiles of 128
    # rows, so CTA pairs with and without an empty second half; K (H = 264)
    # and N (I = 200) ragged
    g = np.log([5, 3, 2, 1, 1, 0.5]) + np.random.default_rng(15).gumbel(size=(700, 6))
    yield "multi_tile", gu.problem(700, 264, 200, 6, 4, seed=14,
                                   ids=np.argsort(-g, axis=1)[:, :4].astype(np.int32))


SCEN = list(_scenarios())


@pytest.fixture(params=[0, 1, 3], ids=["cta", "pair", "small"])
def rows_mode(run, request):
    """Rows-mode GEMMs on single CTAs, on CTA pairs (2-SM MMAs) or on single
    CTAs with token blocks of at most 64 rows."""
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, request.param)
    yield request.param
    hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_PAIR_ROWS, 2)


@pytest.mark.parametrize("training", [True, False])
@pytest.mark.parametrize("case", SCEN, ids=lambda c: c[0])
def test_forward_matches_oracle(run, case, training, rows_mode):
    _, p = case
    d = gu.upload(p)
    y, _ = run.forward(d, training=training)
    torch.cuda.synchronize()
    ref = oracle.forward(p.x, p.ids, p.w, p.W1, p.W2)
    gu.check("y", gu.f64(y), ref)
    assert run.status() == (0, 0)


@pytest.mark.parametrize("case", SCEN, ids=lambda c: c[0])
def test_backward_matches_oracle(run, case, rows_mode):
    _, p = case
    d = gu.upload(p)
    y, saved = run.forward(d)
    dx, dW1, dW2, dw = run.backward(d, saved)
    torch.cuda.synchronize()
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("dx", gu.f64(dx), rdx)
    gu.check("d_topk_weights", gu.f64(dw), rdw)
    gu.check("d_up_proj_weight", gu.f64(dW1), rdW1)
    gu.check("d_down_proj_weight", gu.f64(dW2), rdW2)
    counts = np.bincount(p.ids.reshape(-1), minlength=p.E)
    for e in np.nonzero(counts == 0)[0]:       # empty experts: exact zeros
        assert not gu.f64(dW1[e]).any() and not gu.f64(dW2[e]).any()
    assert run.status() == (0, 0)


def test_fp32_routing_weights(run):
    p = gu.problem(96, 128, 64, 6, 3, seed=21)
    d = gu.upload(p, weights_dtype="f32")
    y, saved = run.forward(d)
    dx, dW1, dW2, dw = run.backward(d, saved)
    torch.cuda.synchronize()
    assert dw.dtype == torch.float32
    gu.check("y", gu.f64(y), oracle.forward(p.x, p.ids, p.w, p.W1, p.W2))
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("dx", gu.f64(dx), rdx)
    gu.check("dw", gu.f64(dw), rdw)


def test_repeated_calls_bit_identical(run, rows_mode):
    p = dict(SCEN)["multi_tile"]
    d = gu.upload(p)
    outs = []
    for _ in range(3):
        y, saved = run.forward(d)
        outs.append([y.clone()] + [t.clone() for t in run.backward(d, saved)])
    torch.cuda.synchronize()
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_overlapped_launches_bit_identical(run):
    """Programmatic dependent launches change when kernels are scheduled,
    never what they compute: forward and backward with and without them agree
    bit for bit."""
    p = dict(SCEN)["multi_tile"]
    d = gu.upload(p)
    outs = []
    try:
        for overlap in (0, 1):
            hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_OVERLAP_LAUNCHES, overlap)
            y, saved = run.forward(d)
            outs.append([y.clone()] + [t.clone() for t in run.backward(d, saved)])
        torch.cuda.synchronize()
    finally:
        hmm.hmm_set_option(run.ctx.handle, hmm.HMM_OPT_OVERLAP_LAUNCHES, 1)
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    assert run.status() == (0, 0)


def test_out_of_range_expert_id_reported(run):
    p = gu.problem(64, 128, 64, 8, 2, seed=3)
    ids = p.ids.copy()
    ids[5, 1] = 8                                 # == E
    p.ids = ids
    d = gu.upload(p)
    run.ctx.set_option(hmm.HMM_OPT_VALIDATE, 1)
    try:
        with pytest.raises(hmm.HmmError) as ei:
            run.forward(d)
        assert ei.value.code == hmm.HMM_ERR_EXPERT_ID
    finally:
        run.ctx.set_option(hmm.HMM_OPT_VALIDATE, 0)
    # without validation the call runs and the status word reports it
    p.ids[5, 1] = -3
    d = gu.upload(p)
    run.forward(d)
    rc, bits = run.status()
    assert rc == hmm.HMM_ERR_EXPERT_ID and bits & hmm.HMM_STATUS_EXPERT_ID
    assert run.status() == (0, 0)                 # cleared


def test_host_boundary_rejections(run):
    p = gu.problem(64, 128, 64, 8, 2, seed=3)
    d = gu.upload(p)
    sh = run.shape(d)
    fwd, sv, _ = hmm.hmm_workspace_size(sh, True)
    y = torch.empty_like(d.x)
    small = torch.empty(fwd - 256, dtype=torch.uint8, device=gu.dev())
    saved = torch.empty(sv, dtype=torch.uint8, device=gu.dev())
    with pytest.raises(hmm.HmmError) as ei:
        hmm.hmm_forward(run.ctx.handle, sh, d.x, d.ids, d.w, d.W1, d.W2, y, saved, small)
    assert ei.value.code == -5
    ws = torch.empty(fwd + 16, dtype=torch.uint8, device=gu.dev())
    with pytest.raises(hmm.HmmError) as ei:   # misaligned x
        hmm.hmm_forward(run.ctx.handle, sh, d.x.data_ptr() + 2, d.ids, d.w, d.W1, d.W2, y,
                        saved, ws)
    assert ei.value.code == -4
    with pytest.raises(TypeError):
        run.forward(gu.SimpleNamespace(x=d.x.float(), ids=d.ids, w=d.w, W1=d.W1, W2=d.W2))
    with pytest.raises(ValueError):
        run.forward(gu.SimpleNamespace(x=d.x, ids=d.ids, w=d.w, W1=d.W1, W2=d.W2[:, :32]))


def test_autograd_and_grad_accumulation(run):
    p = gu.problem(64, 128, 64, 8, 2, seed=1000)
    d = gu.upload(p)
    x = d.x.clone().requires_grad_()
    w = d.w.clone().requires_grad_()
    W1 = d.W1.clone().requires_grad_()
    W2 = d.W2.clone().requires_grad_()
    for _ in range(2):                             # grads accumulate into .grad
        y = hmm.moe_ffn(x, d.ids, w, W1, W2)
        y.backward(d.dy)
    torch.cuda.synchronize()
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("2*dx", gu.f64(x.grad), 2 * rdx)
    gu.check("2*dW1", gu.f64(W1.grad), 2 * rdW1)
    gu.check("2*dW2", gu.f64(W2.grad), 2 * rdW2)
    gu.check("2*dw", gu.f64(w.grad), 2 * rdw)
    with torch.no_grad():
        y2 = hmm.moe_ffn(d.x, d.ids, d.w, d.W1, d.W2)
    assert torch.equal(y2.view(torch.int16), y.detach().view(torch.int16))


def test_backward_split_dx_then_dw_is_bit_identical(run, rows_mode):
    """hmm_backward_dx followed by hmm_backward_dw (the deferred weight
    gradients of the EP overlap issue's W/D split, §2.3) writes what one
    hmm_backward call writes, bit for bit; the weight half can also write
    one of the two weight gradients alone."""
    p = dict(SCEN)["multi_tile"]
    d = gu.upload(p)
    y, saved = run.forward(d)
    dx, dW1, dW2, dw = run.backward(d, saved)
    sh = run.shape(d)
    _, _, bwd = hmm.hmm_workspace_size(sh, True)
    ws = torch.empty(bwd, dtype=torch.uint8, device=gu.dev())
    dx2 = torch.empty_like(dx)
    dw2 = torch.empty_like(dw)
    dW1b = torch.full_like(dW1, float("nan"))
    dW2b = torch.full_like(dW2, float("nan"))
    hmm.hmm_backward_dx(run.ctx.handle, sh, d.dy, d.w, d.W1, d.W2, saved, dx2, dw2, ws)
    torch.cuda.synchronize()
    assert torch.equal(dx.view(torch.int16), dx2.view(torch.int16))
    assert torch.equal(dw.view(torch.int16), dw2.view(torch.int16))
    hmm.hmm_backward_dw(run.ctx.handle, sh, saved, dW1b, dW2b, ws)
    torch.cuda.synchronize()
    assert torch.equal(dW1.view(torch.int16), dW1b.view(torch.int16))
    assert torch.equal(dW2.view(torch.int16), dW2b.view(torch.int16))
    # one weight gradient only
    dW2c = torch.full_like(dW2, float("nan"))
    hmm.hmm_backward_dw(run.ctx.handle, sh, saved, None, dW2c, ws)
    torch.cuda.synchronize()
    assert torch.equal(dW2.view(torch.int16), dW2c.view(torch.int16))
    assert run.status() == (0, 0)


@pytest.mark.parametrize("case", ["multi_tile", "empty_and_hot", "duplicates"])
def test_backward_split_matches_oracle(run, case, rows_mode):
    """The W/D split against the fp64 oracle [EP overlap issue §2.3, §4.5:
    D-only and W-only entry points; HyperMegaMoE §7.2: each optional
    increment gets its own forward, backward and edge cases]: dx and
    d_topk_weights from hmm_backward_dx, then the weight gradients from a
    later hmm_backward_dw (another kernel launched in between on the same
    stream), each elementwise within the tolerance; empty experts exact
    zeros."""
    p = dict(SCEN)[case]
    d = gu.upload(p)
    y, saved = run.forward(d)
    sh = run.shape(d)
    _, _, bwd = hmm.hmm_workspace_size(sh, True)
    ws = torch.empty(bwd, dtype=torch.uint8, device=gu.dev())
    dx = torch.empty_like(d.x)
    dw = torch.empty_like(d.w)
    dW1 = torch.full_like(d.W1, float("nan"))
    dW2 = torch.full_like(d.W2, float("nan"))
    hmm.hmm_backward_dx(run.ctx.handle, sh, d.dy, d.w, d.W1, d.W2, saved, dx, dw, ws)
    other = torch.randn(1 << 20, device=gu.dev()).sum()    # unrelated work in between
    hmm.hmm_backward_dw(run.ctx.handle, sh, saved, dW1, dW2, ws)
    torch.cuda.synchronize()
    del other
    rdx, rdW1, rdW2, rdw = oracle.backward(p.x, p.ids, p.w, p.W1, p.W2, p.dy)
    gu.check("dx (backward_dx)", gu.f64(dx), rdx)
    gu.check("d_topk_weights (backward_dx)", gu.f64(dw), rdw)
    gu.check("d_up_proj_weight (backward_dw)", gu.f64(dW1), rdW1)
    gu.check("d_down_proj_weight (backward_dw)", gu.f64(dW2), rdW2)
    counts = np.bincount(p.ids.reshape(-1), minlength=p.E)
    for e in np.nonzero(counts == 0)[0]:
        assert not gu.f64(dW1[e]).any() and not gu.f64(dW2[e]).any()
    assert run.status() == (0, 0)

"""Pins for the fp64 oracle, each against something other than the oracle.

- routing: brute force by a library sort of (expert, slot) pairs;
- forward: an independent dense formulation (every expert on every token,
  weighted by its summed gate), a library special case (E=1, K=1, w=1 is a
  plain SwiGLU FFN, checked against torch fp64), a closed-form probe with
  unique token values and per-expert signature columns (MoE overlap explainer
  §6 test recipe), and the invariances the method fixes (token-order
  equivariance, expert relabelling, linearity in the routing weights, zero
  weights inert);
- backward: central finite differences of the forward in fp64, the library
  special case through torch autograd, exact zeros for empty experts and the
  exact linearity of y in each routing weight.

Each test would fail for a dropped term, a wrong sign or index, a transposed
operand or swapped gate/up halves somewhere in the oracle.
"""
import math

import numpy as np
import pytest

import moe_inputs as mi
import oracle


def _tiny_f64(T=5, H=6, I=4, E=3, K=2, seed=0, distinct=True):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, H))
    if distinct:
        ids = np.stack([r.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    else:
        ids = r.integers(0, E, size=(T, K)).astype(np.int32)
    w = r.random((T, K))
    W1 = r.standard_normal((E, H, 2 * I)) / math.sqrt(H)
    W2 = r.standard_normal((E, I, H)) / math.sqrt(I)
    dy = r.standard_normal((T, H))
    return x, ids, w, W1, W2, dy


def _dense(x, ids, w, W1, W2):
    """Independent formulation: run every expert on every token and weight it
    by c_e[t] = sum_k w[t,k] [ids[t,k] == e] (handles repeated experts)."""
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    y = np.zeros((T, H))
    for e in range(E):
        c = ((ids == e) * w).sum(axis=1)
        g = x @ W1[e][:, :I]
        u = x @ W1[e][:, I:]
        y += c[:, None] * (((g / (1.0 + np.exp(-g))) * u) @ W2[e])
    return y


# ---------------------------------------------------------------- routing

@pytest.mark.parametrize("T,K,E,seed", [(1, 1, 1, 0), (7, 3, 5, 1), (64, 2, 8, 2),
                                        (300, 6, 64, 3), (50, 4, 3, 4)])
def test_route_brute_force_sort(T, K, E, seed):
    r = np.random.default_rng(seed)
    ids = r.integers(0, E, size=(T, K)).astype(np.int32)  # repeats allowed
    counts, offsets, s2r, r2s = oracle.route(ids, E)
    flat = ids.reshape(-1)
    order = sorted(range(T * K), key=lambda s: (int(flat[s]), s))
    np.testing.assert_array_equal(r2s, np.array(order, np.int32))
    inv = np.empty(T * K, np.int64)
    inv[np.array(order)] = np.arange(T * K)
    np.testing.assert_array_equal(s2r, inv)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert counts.sum() == T * K
    np.testing.assert_array_equal(r2s[s2r], np.arange(T * K))


def test_route_rejects_out_of_range():
    ids = np.array([[0, 3]], np.int32)
    with pytest.raises(oracle.InvalidExpertId):
        oracle.route(ids, 3)
    with pytest.raises(oracle.InvalidExpertId):
        oracle.route(np.array([[-1]], np.int32), 3)


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("distinct", [True, False])
@pytest.mark.parametrize("seed", [0, 1])
def test_forward_matches_dense_formulation(distinct, seed):
    x, ids, w, W1, W2, _ = _tiny_f64(T=9, H=8, I=5, E=4, K=3, seed=seed, distinct=distinct)
    y = oracle.forward(x, ids, w, W1, W2)
    np.testing.assert_allclose(y, _dense(x, ids, w, W1, W2), rtol=1e-12, atol=1e-13)


def test_forward_E1_K1_is_plain_swiglu_ffn_torch():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(5)
    T, H, I = 6, 16, 12
    x = r.standard_normal((T, H))
    W1 = r.standard_normal((1, H, 2 * I)) / 4
    W2 = r.standard_normal((1, I, H)) / 4
    y = oracle.forward(x, np.zeros((T, 1), np.int32), np.ones((T, 1)), W1, W2)
    xt = torch.from_numpy(x)
    Wg = torch.from_numpy(W1[0][:, :I])
    Wu = torch.from_numpy(W1[0][:, I:])
    Wd = torch.from_numpy(W2[0])
    ref = (torch.nn.functional.silu(xt @ Wg) * (xt @ Wu)) @ Wd
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_forward_closed_form_signature_probe():
    """Unique token values, and expert e writes (e+1)*a_t only into column
    1+e: any misrouting, wrong gate or dropped slot changes a column."""
    T, E, K, I = 10, 5, 3, 1
    H = 1 + E
    r = np.random.default_rng(11)
    ids = np.stack([r.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w = r.random((T, K))
    x = np.zeros((T, H))
    x[:, 0] = 0.25 + 0.1 * np.arange(T)           # unique per token
    W1 = np.zeros((E, H, 2 * I))
    W1[:, 0, 0] = 1.0                              # gate = x0
    W1[:, 0, 1] = 2.0                              # up = 2 x0
    W2 = np.zeros((E, I, H))
    for e in range(E):
        W2[e, 0, 1 + e] = e + 1.0
    y = oracle.forward(x, ids, w, W1, W2)
    for t in range(T):
        g = x[t, 0]
        a = g / (1.0 + math.exp(-g)) * (2.0 * g)
        expect = np.zeros(H)
        for k in range(K):
            expect[1 + ids[t, k]] += w[t, k] * (ids[t, k] + 1.0) * a
        np.testing.assert_allclose(y[t], expect, rtol=1e-14, atol=0)
        assert y[t, 0] == 0.0


def test_forward_gate_up_order_matters():
    """Swapping the gate and up halves changes y (silu is not symmetric)."""
    x, ids, w, W1, W2, _ = _tiny_f64(seed=3)
    I = W1.shape[2] // 2
    swapped = np.concatenate([W1[:, :, I:], W1[:, :, :I]], axis=2)
    assert np.abs(oracle.forward(x, ids, w, W1, W2) - oracle.forward(x, ids, w, swapped, W2)).max() > 1e-3


def test_forward_token_permutation_equivariance():
    x, ids, w, W1, W2, _ = _tiny_f64(T=11, seed=4)
    p = np.random.default_rng(0).permutation(x.shape[0])
    y = oracle.forward(x, ids, w, W1, W2)
    yp = oracle.forward(x[p], ids[p], w[p], W1, W2)
    np.testing.assert_array_equal(yp, y[p])


def test_forward_expert_relabelling_invariance():
    x, ids, w, W1, W2, _ = _tiny_f64(T=8, E=5, seed=6)
    q = np.random.default_rng(1).permutation(W1.shape[0])   # new label of expert e is q[e]
    W1n = np.empty_like(W1)
    W2n = np.empty_like(W2)
    W1n[q] = W1
    W2n[q] = W2
    y = oracle.forward(x, ids, w, W1, W2)
    yn = oracle.forward(x, q[ids].astype(np.int32), w, W1n, W2n)
    np.testing.assert_array_equal(yn, y)


@pytest.mark.parametrize("alpha", [2.0, 0.5, 0.0])
def test_forward_linear_in_weights(alpha):
    x, ids, w, W1, W2, _ = _tiny_f64(seed=7)
    np.testing.assert_array_equal(oracle.forward(x, ids, alpha * w, W1, W2),
                                  alpha * oracle.forward(x, ids, w, W1, W2))


def test_forward_zero_weight_slots_inert():
    x, ids, w, W1, W2, _ = _tiny_f64(T=8, E=4, K=2, seed=8)
    w0 = w.copy()
    w0[:, 1] = 0.0
    ids2 = ids.copy()
    ids2[:, 1] = (ids[:, 1] + 1) % 4          # rerouting a zero-weight slot changes nothing
    y_a = oracle.forward(x, ids, w0, W1, W2)
    y_b = oracle.forward(x, ids2, w0, W1, W2)
    y_k1 = oracle.forward(x, ids[:, :1].copy(), w[:, :1].copy(), W1, W2)
    np.testing.assert_array_equal(y_a, y_b)
    np.testing.assert_array_equal(y_a, y_k1)


def test_forward_bf16_inputs_decode_exactly():
    """bf16 and fp64 entry points agree when given the same values."""
    p = mi.make_shape(6, 16, 8, 4, 2, seed=3)
    f = lambda b: mi.bf16_bits_to_f32(b).astype(np.float64)
    y16 = oracle.forward(p.x, p.topk_ids, p.topk_weights, p.W1, p.W2)
    y64 = oracle.forward(f(p.x), p.topk_ids, f(p.topk_weights), f(p.W1), f(p.W2))
    np.testing.assert_array_equal(y16, y64)


def test_expert_ffn_stagewise():
    x, ids, w, W1, W2, _ = _tiny_f64(seed=9)
    I = W1.shape[2] // 2
    h, a, o = oracle.expert_ffn(x[0], W1[1], W2[1])
    np.testing.assert_allclose(h, x[0] @ W1[1], rtol=1e-13, atol=1e-14)
    g, u = h[:I], h[I:]
    np.testing.assert_allclose(a, g / (1 + np.exp(-g)) * u, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o, a @ W2[1], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- backward

def _loss(x, ids, w, W1, W2, dy):
    return float((oracle.forward(x, ids, w, W1, W2) * dy).sum())


def _fd(f, arr, idx, eps=1e-6):
    old = arr[idx]
    arr[idx] = old + eps
    lp = f()
    arr[idx] = old - eps
    lm = f()
    arr[idx] = old
    return (lp - lm) / (2 * eps)


@pytest.mark.parametrize("distinct", [True, False])
def test_backward_finite_differences(distinct):
    x, ids, w, W1, W2, dy = _tiny_f64(T=4, H=5, I=3, E=3, K=2, seed=12, distinct=distinct)
    dx, dW1, dW2, dw = oracle.backward(x, ids, w, W1, W2, dy)
    f = lambda: _loss(x, ids, w, W1, W2, dy)
    rel = lambda a, b: abs(a - b) / max(1e-8, abs(b))
    for idx in np.ndindex(x.shape):
        assert rel(dx[idx], _fd(f, x, idx)) < 1e-6
    for idx in np.ndindex(w.shape):
        assert rel(dw[idx], _fd(f, w, idx)) < 1e-6
    for idx in np.ndindex(W1.shape):
        assert abs(dW1[idx] - _fd(f, W1, idx)) < 1e-6 * max(1.0, abs(dW1[idx]))
    for idx in np.ndindex(W2.shape):
        assert abs(dW2[idx] - _fd(f, W2, idx)) < 1e-6 * max(1.0, abs(dW2[idx]))


def test_backward_E1_K1_torch_autograd():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(21)
    T, H, I = 5, 12, 8
    x = r.standard_normal((T, H))
    W1 = r.standard_normal((1, H, 2 * I)) / 3
    W2 = r.standard_normal((1, I, H)) / 3
    w = r.random((T, 1)) + 0.5
    dy = r.standard_normal((T, H))
    dx, dW1, dW2, dw = oracle.backward(x, np.zeros((T, 1), np.int32), w, W1, W2, dy)
    xt = torch.from_numpy(x).requires_grad_()
    W1t = torch.from_numpy(W1[0]).requires_grad_()
    W2t = torch.from_numpy(W2[0]).requires_grad_()
    wt = torch.from_numpy(w).requires_grad_()
    h = xt @ W1t
    y = wt * ((torch.nn.functional.silu(h[:, :I]) * h[:, I:]) @ W2t)
    (y * torch.from_numpy(dy)).sum().backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dW1[0], W1t.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dW2[0], W2t.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_backward_dw_is_exact_linear_response():
    """y is linear in each routing weight, so y(w + d e_tk) - y(w) = d * o_tk
    and dw[t,k] = <dy_t, o_tk> holds with w = 0 as well."""
    x, ids, w, W1, W2, dy = _tiny_f64(T=6, seed=13)
    w[2, 1] = 0.0
    _, dw = oracle.backward_tokens(x, ids, w, W1, W2, dy)
    for t in range(x.shape[0]):
        for k in range(ids.shape[1]):
            _, _, o = oracle.expert_ffn(x[t], W1[ids[t, k]], W2[ids[t, k]])
            np.testing.assert_allclose(dw[t, k], float(dy[t] @ o), rtol=1e-12, atol=1e-13)
    assert dw[2, 1] != 0.0


def test_backward_empty_expert_weight_grads_exact_zero():
    x, ids, w, W1, W2, dy = _tiny_f64(T=6, E=4, K=2, seed=14)
    ids[ids == 3] = 0
    ids[:, 1] = np.where(ids[:, 0] == ids[:, 1], 1 + (ids[:, 0] % 2), ids[:, 1])
    assert not (ids == 3).any()
    dW1, dW2 = oracle.weight_grad(3, x, ids, w, W1, W2, dy)
    assert not dW1.any() and not dW2.any()


def test_backward_zero_weight_slot_contributes_no_dx_dW():
    x, ids, w, W1, W2, dy = _tiny_f64(T=5, E=3, K=2, seed=15)
    w[:, 1] = 0.0
    dx, dW1, dW2, _ = oracle.backward(x, ids, w, W1, W2, dy)
    dx1, dW1_1, dW2_1, _ = oracle.backward(x, ids[:, :1].copy(), w[:, :1].copy(), W1, W2, dy)
    np.testing.assert_allclose(dx, dx1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dW1, dW1_1, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dW2, dW2_1, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------ shared expert
# [HyperMegaMoE §6.1] optional shared expert, merged at Combine with unit
# weight (the reading: no gate, every token).

def _shared_f64(T=6, H=8, I=5, seed=7):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, H))
    Ws1 = r.standard_normal((H, 2 * I)) / math.sqrt(H)
    Ws2 = r.standard_normal((I, H)) / math.sqrt(I)
    dy = r.standard_normal((T, H))
    return x, Ws1, Ws2, dy


def test_shared_forward_is_a_dense_swiglu_ffn_torch():
    """Library special case: the shared term is silu(x Wg) (x Wu) Wd for
    every token, as torch computes it in fp64."""
    torch = pytest.importorskip("torch")
    x, Ws1, Ws2, _ = _shared_f64()
    I = Ws2.shape[0]
    xt, W1t, W2t = (torch.from_numpy(a) for a in (x, Ws1, Ws2))
    ref = (torch.nn.functional.silu(xt @ W1t[:, :I]) * (xt @ W1t[:, I:])) @ W2t
    np.testing.assert_allclose(oracle.shared_forward(x, Ws1, Ws2), ref.numpy(),
                               rtol=1e-12, atol=1e-12)


def test_shared_backward_matches_torch_autograd():
    """dx_s, dWs1, dWs2 of L = <dy, FFN_s(x)> against torch fp64 autograd."""
    torch = pytest.importorskip("torch")
    x, Ws1, Ws2, dy = _shared_f64()
    I = Ws2.shape[0]
    xt, W1t, W2t = (torch.from_numpy(a).clone().requires_grad_(True) for a in (x, Ws1, Ws2))
    y = (torch.nn.functional.silu(xt @ W1t[:, :I]) * (xt @ W1t[:, I:])) @ W2t
    (y * torch.from_numpy(dy)).sum().backward()
    dxs, dWs1, dWs2 = oracle.shared_backward(x, Ws1, Ws2, dy)
    np.testing.assert_allclose(dxs, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dWs1, W1t.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dWs2, W2t.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_shared_backward_finite_differences():
    """Central differences of L = <dy, FFN_s(x)> in fp64 for sampled entries."""
    x, Ws1, Ws2, dy = _shared_f64(T=4, H=6, I=3, seed=9)
    dxs, dWs1, dWs2 = oracle.shared_backward(x, Ws1, Ws2, dy)
    loss = lambda x_, a_, b_: float((oracle.shared_forward(x_, a_, b_) * dy).sum())
    eps = 1e-6
    r = np.random.default_rng(1)
    for arr, grad, which in ((x, dxs, 0), (Ws1, dWs1, 1), (Ws2, dWs2, 2)):
        for _ in range(6):
            idx = tuple(r.integers(0, n) for n in arr.shape)
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [x, Ws1, Ws2]
            args_m = [x, Ws1, Ws2]
            args_p[which], args_m[which] = p, m
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


def test_shared_expert_equals_a_routed_expert_with_unit_weight():
    """The shared expert is the routed forward/backward of an E=1, K=1 layer
    with every routing weight 1 (the routed oracle is pinned above)."""
    x, Ws1, Ws2, dy = _shared_f64(T=7, seed=11)
    T = x.shape[0]
    ids = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    np.testing.assert_allclose(oracle.shared_forward(x, Ws1, Ws2),
                               oracle.forward(x, ids, w, Ws1[None], Ws2[None]),
                               rtol=1e-13, atol=1e-13)
    dxs, dWs1, dWs2 = oracle.shared_backward(x, Ws1, Ws2, dy)
    rdx, rdW1, rdW2, _ = oracle.backward(x, ids, w, Ws1[None], Ws2[None], dy)
    np.testing.assert_allclose(dxs, rdx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dWs1, rdW1[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dWs2, rdW2[0], rtol=1e-12, atol=1e-12)

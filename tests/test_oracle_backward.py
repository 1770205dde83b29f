"""Pins of the oracle's router-side backward and selection-bias update (CPU only).

The analytic gradient is checked against central finite differences of the forward oracle's own
loss terms (aux_stats_from_counts for P and z, softmax_topk_route for the softmax weights), so a
dropped term, a wrong sign or a transposed product in the backward fails here.  Closed forms
at uniform logits and the feedback direction stated by the pages pin the rest.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O

F64 = np.float64


def _kth_gap(key, k):
    s = -np.sort(-key, axis=1)
    return float(np.min(s[:, k - 1] - s[:, k])) if key.shape[1] > k else np.inf


def _loss_softmax(g, idx, counts, d_w, alpha, beta, renorm, scale):
    """Router-side loss from the forward oracle's functions (selection recomputed and checked)."""
    T, E = g.shape
    st = O.aux_stats_from_counts(g, counts, E, "softmax")
    idx2, w, _ = O.softmax_topk_route(g, idx.shape[1], renorm, scale)
    assert np.array_equal(idx2, idx)
    return alpha * st["l_balance"] + beta * st["z_loss"] + float((d_w * w).sum())


def _loss_sigmoid(g, idx, counts, d_w, alpha, beta, renorm, scale):
    """Same for sigmoid scoring; the weights are the forward's steps 8-10 on the fixed selection
    (the forward rounds s to float32 for the selection, which finite differences cannot see
    through)."""
    T, E = g.shape
    st = O.aux_stats_from_counts(g, counts, E, "sigmoid")
    s = O.sigmoid(g)
    sS = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    w = sS / sS.sum(axis=1, keepdims=True) if renorm else sS
    return alpha * st["l_balance"] + beta * st["z_loss"] + float((d_w * w * scale).sum())


def _fd_grad(fun, g, h=1e-6):
    out = np.zeros_like(g)
    for i in range(g.shape[0]):
        for j in range(g.shape[1]):
            gp = g.copy(); gp[i, j] += h
            gm = g.copy(); gm[i, j] -= h
            out[i, j] = (fun(gp) - fun(gm)) / (2 * h)
    return out


def _counts(idx, E):
    return np.bincount(idx.reshape(-1), minlength=E).astype(F64)


@pytest.mark.parametrize("renorm,scale,k", [(True, 1.0, 2), (True, 2.5, 3), (False, 1.0, 1)])
def test_softmax_backward_matches_finite_differences(renorm, scale, k):
    rng = np.random.default_rng(11 + k)
    T, E = 6, 8
    g = rng.standard_normal((T, E)) * 1.5
    idx = O.topk_desc(g, k)
    assert _kth_gap(g, k) > 1e-3
    counts = _counts(idx, E)
    d_w = rng.standard_normal((T, k))
    alpha, beta = 0.37, 0.21
    dg = O.router_backward(g, idx, d_w, counts / T, alpha, beta, "softmax", renorm, scale)
    fd = _fd_grad(lambda gg: _loss_softmax(gg, idx, counts, d_w, alpha, beta, renorm, scale), g)
    assert np.max(np.abs(dg - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd)))


@pytest.mark.parametrize("groups,renorm", [((1, 1), True), ((4, 2), True), ((1, 1), False)])
def test_sigmoid_backward_matches_finite_differences(groups, renorm):
    rng = np.random.default_rng(5)
    T, E, k = 5, 16, 4
    g = rng.standard_normal((T, E))
    bias = (rng.random(E) - 0.5) * 0.2
    idx, _, _ = O.sigmoid_group_route(g.astype(np.float32), bias, k, groups[0], groups[1], 2.5,
                                      renorm)
    counts = _counts(idx, E)
    d_w = rng.standard_normal((T, k))
    alpha, beta = 0.5, 0.1
    dg = O.router_backward(g, idx, d_w, counts / T, alpha, beta, "sigmoid", renorm, 2.5)
    fd = _fd_grad(lambda gg: _loss_sigmoid(gg, idx, counts, d_w, alpha, beta, renorm, 2.5), g)
    assert np.max(np.abs(dg - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd)))


def test_param_grads_match_finite_differences():
    rng = np.random.default_rng(3)
    T, d, E, k = 5, 6, 4, 2
    x = rng.standard_normal((T, d))
    W = rng.standard_normal((E, d)) * 0.5
    g = x @ W.T
    idx = O.topk_desc(g, k)
    assert _kth_gap(g, k) > 1e-3
    counts = _counts(idx, E)
    d_w = rng.standard_normal((T, k))
    a, b = 0.3, 0.2
    dg = O.router_backward(g, idx, d_w, counts / T, a, b, "softmax", True, 1.0)
    dW, dx = O.router_param_grads(x, W, dg)
    lossW = lambda WW: _loss_softmax(x @ WW.T, idx, counts, d_w, a, b, True, 1.0)
    lossx = lambda xx: _loss_softmax(xx @ W.T, idx, counts, d_w, a, b, True, 1.0)
    assert np.max(np.abs(dW - _fd_grad(lossW, W))) <= 1e-7 * max(1.0, np.abs(dW).max())
    assert np.max(np.abs(dx - _fd_grad(lossx, x))) <= 1e-7 * max(1.0, np.abs(dx).max())


def test_uniform_logits_closed_forms():
    """At g = 0 every p_i = 1/E and lse = log E, so the balance term gives
    (alpha E / T)(f_i - mean f) / E per entry and the z term beta (2/T) log(E) / E."""
    T, E, k = 8, 4, 2
    g = np.zeros((T, E))
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    f = np.array([1.0, 0.75, 0.25, 0.0])
    alpha, beta = 0.7, 0.3
    dg_bal = O.router_backward(g, idx, None, f, alpha, 0.0)
    expect = alpha * E / T * (f - f.mean()) / E
    assert np.allclose(dg_bal, np.tile(expect, (T, 1)), rtol=0, atol=1e-15)
    dg_z = O.router_backward(g, idx, None, None, 0.0, beta)
    assert np.allclose(dg_z, beta * 2.0 / T * np.log(E) / E, rtol=0, atol=1e-15)
    # sigmoid at g = 0: s = 1/2, s(1-s) = 1/4, q = 1/E, sum s = E/2
    dg_sig = O.router_backward(g, idx, None, f, alpha, 0.0, "sigmoid")
    expect_sig = alpha * E / T * (f - f.mean()) / (E / 2) * 0.25
    assert np.allclose(dg_sig, np.tile(expect_sig, (T, 1)), rtol=0, atol=1e-15)


def test_balance_gradient_pushes_overloaded_experts_down():
    """The feedback the pages describe: the more an expert is chosen (larger f_i), the larger
    dL/dP_i, so a descent step lowers that expert's logits relative to the others."""
    rng = np.random.default_rng(9)
    T, E = 64, 8
    g = rng.standard_normal((T, E)) * 0.01
    f = np.array([0.9, 0.5, 0.2, 0.1, 0.1, 0.1, 0.05, 0.05])
    idx = O.topk_desc(g, 2)
    dg = O.router_backward(g, idx, None, f, 1.0, 0.0)
    col = dg.sum(axis=0)
    assert col[0] > 0 and col[-1] < 0
    order = np.argsort(-f, kind="stable")
    strictly = np.diff(f[order]) < 0
    assert np.all(np.diff(col[order])[strictly] < 0)
    # one descent step lowers P of the most chosen expert and raises P of the least chosen
    P0 = O.softmax(g).mean(axis=0)
    P1 = O.softmax(g - 50.0 * dg).mean(axis=0)
    assert P1[0] < P0[0] and P1[-1] > P0[-1]


def test_no_terms_no_gradient():
    g = np.random.default_rng(1).standard_normal((4, 6))
    idx = O.topk_desc(g, 2)
    assert not O.router_backward(g, idx, None, None, 0.0, 0.0).any()


def test_finite_differences_catch_planted_mistakes():
    """Sensitivity of the pin: a flipped z-loss sign, a gradient taken at the wrong route scale,
    or frequencies normalised by T*k instead of T all disagree with the finite differences by
    far more than the tolerance."""
    rng = np.random.default_rng(2)
    T, E, k = 6, 8, 2
    g = rng.standard_normal((T, E))
    idx = O.topk_desc(g, k)
    counts = _counts(idx, E)
    d_w = rng.standard_normal((T, k))
    fd = _fd_grad(lambda gg: _loss_softmax(gg, idx, counts, d_w, 0.5, 0.5, True, 2.5), g)
    tol = 1e-7 * max(1.0, np.abs(fd).max())
    good = O.router_backward(g, idx, d_w, counts / T, 0.5, 0.5, "softmax", True, 2.5)
    assert np.max(np.abs(good - fd)) <= tol
    z_only = O.router_backward(g, idx, None, None, 0.0, 0.5)
    planted = [good - 2 * z_only,
               O.router_backward(g, idx, d_w, counts / T, 0.5, 0.5, "softmax", True, 1.0),
               O.router_backward(g, idx, d_w, counts / (T * k), 0.5, 0.5, "softmax", True, 2.5)]
    for bad in planted:
        assert np.max(np.abs(bad - fd)) > 1e3 * tol


def test_bias_update_hand_example():
    """T=8 tokens, k=2, E=4: mean load 4.  Loads 5, 3, 4, 4 -> -g, +g, unchanged, unchanged."""
    b = np.array([0.0, 0.1, -0.1, 0.25], np.float32)
    out = O.bias_update(b, np.array([5, 3, 4, 4]), T=8, k=2, gamma=0.001)
    assert out.dtype == np.float32
    assert out[0] == np.float32(np.float32(0.0) - np.float32(0.001))
    assert out[1] == np.float32(np.float32(0.1) + np.float32(0.001))
    assert out[2] == b[2] and out[3] == b[3]


def test_bias_update_balances_a_skewed_router():
    """Closing the loop of the DeepSeek-V3 rule on a skewed router (selection on s + b, load =
    selections per expert) brings the busiest expert near the mean load, which an update of the
    wrong sign would drive away from it."""
    rng = np.random.default_rng(4)
    T, E, k = 2048, 16, 2
    g = rng.standard_normal((T, E)).astype(np.float32) + np.linspace(1.0, -1.0, E,
                                                                    dtype=np.float32)
    b = np.zeros(E, np.float32)

    def loads(bias):
        idx, _, _ = O.sigmoid_group_route(g, bias, k, 1, 1, 1.0)
        return np.bincount(idx.reshape(-1), minlength=E)

    ratio0 = loads(b).max() / (T * k / E)
    for _ in range(300):
        b = O.bias_update(b, loads(b), T, k, 0.002)
    ratio1 = loads(b).max() / (T * k / E)
    assert ratio0 > 1.5 and ratio1 < 1.1
    # the wrong sign makes it worse
    bw = np.zeros(E, np.float32)
    for _ in range(50):
        bw = (2 * bw - O.bias_update(bw, loads(bw), T, k, 0.002)).astype(np.float32)
    assert loads(bw).max() / (T * k / E) > ratio0

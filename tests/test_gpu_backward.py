"""GPU parity of the router-side backward and the selection-bias update against the oracle.

Both sides take the same float32 logits (the oracle's), the same selection and the same
frequencies, so the comparison isolates the backward.  Tolerances, derived from the arithmetic:
  * dL/dg is float32 on the device: |err| <= DG_RTOL x S_t, where S_t is the token's scale of
    the terms before they cancel: max_e |dL/dg| + sum_j |d_w w_j| + alpha E max f / T +
    2 beta |lse| / T.  (With renormalised weights the gate term sums to zero over the selected
    experts, so when a token's upstream gradients are nearly equal its dL/dg is much smaller
    than the float32 terms it was computed from);
  * the gradient GEMMs (bf16 configuration) take dL/dg rounded once to bf16 (relative error
    <= 2^-8 per entry) times exact bf16 x or W_gate, accumulated in float32 over K terms, so
    |err| <= sum_t (2^-8 |dg| + 1.01 delta_t) |x| + K 2^-24 sum_t |dg x| elementwise, with
    delta_t = DG_RTOL x S_t the dL/dg allowance of token t;
  * the bias update is one float32 addition: bit-exact.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from gpu_util import config_of, lib
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

DG_RTOL = 2e-5
U_BF16 = 2.0 ** -8
ALPHA, BETA = 0.01, 0.001


def _case(name, **kw):
    return moe_inputs.workload(name, **kw)


SMALL = {
    "tiny_f32": _case("tiny"),
    "mixtral_like": _case("mixtral", T=300, d=256),
    "dsmoe_like_d384": _case("dsmoe16b", T=777, d=384),
    "v3_like_groups": _case("v3", T=200, d=512, E=64),
    "e160_n192": _case("mixtral", T=130, d=256, E=160, k=4),
    "switch_k1": _case("mixtral", T=257, d=256, E=16, k=1, renormalize=False),
    "one_token": _case("mixtral", T=1, d=256),
    "v3_scaled_sigmoid": _case("v3", T=96, d=256, E=256),
}
FULL = {"mixtral": _case("mixtral"), "dsmoe16b": _case("dsmoe16b"), "v3": _case("v3")}


def _reference(wl, T, alpha, beta, with_dw, inp, gi):
    x64 = moe_inputs.to_f64(inp["x"])
    w64 = moe_inputs.to_f64(inp["w_gate"])
    r = O.route(wl, x64, w64, moe_inputs.to_f64(inp["bias"]))
    counts = np.bincount(r["idx"].reshape(-1), minlength=wl.E)
    f32 = (counts / T).astype(np.float32)
    dw = moe_inputs.to_f64(gi["d_topk_w"]) if with_dw else None
    dg = O.router_backward(r["g32"], r["idx"], dw, f32.astype(np.float64), alpha, beta, wl.score,
                           wl.renormalize, wl.route_scale)
    g = r["g32"].astype(np.float64)
    gm = g.max(axis=1)
    lse = gm + np.log(np.exp(g - gm[:, None]).sum(axis=1))
    scale = np.abs(dg).max(axis=1) + alpha * wl.E * f32.max() / T + 2 * beta * np.abs(lse) / T
    if dw is not None:
        scale = scale + (np.abs(dw) * np.abs(r["w"])).sum(axis=1)
    return {"x": x64, "w": w64, "g32": r["g32"], "idx": r["idx"], "f32": f32, "counts": counts,
            "dg": dg, "dg_scale": scale[:, None]}


def _run(wl, T, ref, gi, alpha, beta, with_dw=True, want_dlogits=True, want_dx=True):
    m = lib()
    cfg = config_of(wl, T)
    dev = "cuda"
    inp_x, inp_w = ref["x_dev"], ref["w_dev"]
    logits = torch.from_numpy(ref["g32"]).to(dev)
    idx = torch.from_numpy(ref["idx"]).to(dev)
    f = torch.from_numpy(ref["f32"]).to(dev)
    d_logits = torch.full((T, wl.E), float("nan"), device=dev) if want_dlogits else None
    d_w_gate = torch.full((wl.E, wl.d), float("nan"), device=dev)
    d_x = torch.full((T, wl.d), float("nan"), device=dev) if want_dx else None
    ws = m.router_backward_workspace(cfg)
    m.moe_router_backward(cfg, inp_x, inp_w, logits, idx, gi["d_topk_w"] if with_dw else None, f,
                          alpha, beta, d_logits, d_w_gate, d_x, ws)
    torch.cuda.synchronize()
    st = m.sync_status(ws)
    assert st == 0, m.status_string(st)
    to = lambda t: None if t is None else t.cpu().numpy().astype(np.float64)
    return {"d_logits": to(d_logits), "d_w_gate": to(d_w_gate), "d_x": to(d_x)}


def _check_dg(got, ref):
    dg, scale = ref["dg"], ref["dg_scale"]
    err = np.abs(got - dg)
    assert np.isfinite(got).all()
    assert np.all(err <= DG_RTOL * scale + 1e-30), float((err / (scale + 1e-30)).max())


def _gemm_bound(dg, scale, K, bf16):
    """Elementwise allowance for dg^T other (dW) or dg other (dx), see the module docstring."""
    delta = DG_RTOL * scale
    D = (U_BF16 * np.abs(dg) + 1.01 * delta) if bf16 else np.broadcast_to(delta, dg.shape)
    return D, K * 2.0 ** -24 + (0 if bf16 else 1e-7)


def _check_gemm(got, want, tol, pred2):
    err = np.abs(got - want)
    assert np.isfinite(got).all()
    assert np.all(err <= tol), float((err / tol).max())
    if pred2 is not None:
        # Tight check: rounding errors are independent across the K terms, so the RMS error is
        # close to the root of the summed variances (uniform rounding: (2^-8)^2 / 3 per term);
        # a misplaced operand tile would give errors of the order of the values themselves.
        rms_err = float(np.sqrt(np.mean(err ** 2)))
        rms_pred = float(np.sqrt(np.mean(pred2)))
        assert rms_err <= 3.0 * rms_pred, (rms_err, rms_pred)
        assert rms_pred < 0.05 * float(np.sqrt(np.mean(want ** 2)))


def _check_dW(got, ref, cols, bf16):
    dg, x = ref["dg"], ref["x"][:, cols]
    want = dg.T @ x
    D, gam = _gemm_bound(dg, ref["dg_scale"], dg.shape[0], bf16)
    tol = D.T @ np.abs(x) + gam * (np.abs(dg).T @ np.abs(x)) + 1e-30
    pred2 = None
    if bf16:
        delta = DG_RTOL * ref["dg_scale"]
        pred2 = (U_BF16 ** 2 / 3) * ((dg ** 2).T @ (x ** 2)) + (delta ** 2).T @ (x ** 2)
    _check_gemm(got[:, cols], want, tol, pred2)


def _check_dx(got, ref, rows, bf16):
    dg, W = ref["dg"][rows], ref["w"]
    want = dg @ W
    D, gam = _gemm_bound(dg, ref["dg_scale"][rows], W.shape[0], bf16)
    tol = D @ np.abs(W) + gam * (np.abs(dg) @ np.abs(W)) + 1e-30
    pred2 = None
    if bf16:
        delta = DG_RTOL * ref["dg_scale"][rows]
        pred2 = (U_BF16 ** 2 / 3) * ((dg ** 2) @ (W ** 2)) + (delta ** 2) * (W ** 2).sum(axis=0)
    _check_gemm(got[rows], want, tol, pred2)


def _full_run(wl, T=None, alpha=ALPHA, beta=BETA, with_dw=True, sample=None):
    T = T or wl.T
    inp = moe_inputs.make_router_inputs(wl, 0, "cuda", T)
    gi = moe_inputs.make_grad_inputs(wl, 0, "cuda", T)
    ref = _reference(wl, T, alpha, beta, with_dw, inp, gi)
    ref["x_dev"], ref["w_dev"] = inp["x"], inp["w_gate"]
    got = _run(wl, T, ref, gi, alpha, beta, with_dw)
    bf16 = wl.dtype == "bf16"
    _check_dg(got["d_logits"], ref)
    rng = np.random.default_rng(0)
    if sample is None:
        cols, rows = np.arange(wl.d), np.arange(T)
    else:
        # every column of the first and last 128-column tile, plus a random sample
        edge = np.r_[np.arange(128), np.arange(wl.d - 128, wl.d)]
        cols = np.unique(np.r_[edge, rng.choice(wl.d, sample, replace=False)])
        rows = np.unique(np.r_[np.arange(min(T, 130)), np.arange(max(0, T - 130), T),
                               rng.choice(T, min(T, sample), replace=False)])
    _check_dW(got["d_w_gate"], ref, cols, bf16)
    _check_dx(got["d_x"], ref, rows, bf16)
    return ref, got


@pytest.mark.parametrize("case", list(SMALL))
def test_router_backward_small(case):
    _full_run(SMALL[case])


@pytest.mark.parametrize("case", list(FULL))
def test_router_backward_full_size(case):
    _full_run(FULL[case], sample=256)


def test_router_backward_term_selection_and_optional_outputs():
    """Each loss term alone, and the optional outputs left out."""
    wl = _case("v3", T=160, d=256, E=64)
    T = wl.T
    inp = moe_inputs.make_router_inputs(wl, 0, "cuda", T)
    gi = moe_inputs.make_grad_inputs(wl, 0, "cuda", T)
    for alpha, beta, with_dw in [(0.3, 0.0, False), (0.0, 0.2, False), (0.0, 0.0, True)]:
        ref = _reference(wl, T, alpha, beta, with_dw, inp, gi)
        ref["x_dev"], ref["w_dev"] = inp["x"], inp["w_gate"]
        got = _run(wl, T, ref, gi, alpha, beta, with_dw)
        _check_dg(got["d_logits"], ref)
        _check_dW(got["d_w_gate"], ref, np.arange(wl.d), True)
    only_dw = _run(wl, T, ref, gi, 0.0, 0.0, True, want_dlogits=False, want_dx=False)
    _check_dW(only_dw["d_w_gate"], ref, np.arange(wl.d), True)


def test_router_backward_is_deterministic():
    wl = _case("v3", T=1000, d=512, E=256)
    inp = moe_inputs.make_router_inputs(wl, 0, "cuda")
    gi = moe_inputs.make_grad_inputs(wl, 0, "cuda")
    ref = _reference(wl, wl.T, ALPHA, BETA, True, inp, gi)
    ref["x_dev"], ref["w_dev"] = inp["x"], inp["w_gate"]
    a = _run(wl, wl.T, ref, gi, ALPHA, BETA)
    b = _run(wl, wl.T, ref, gi, ALPHA, BETA)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_router_backward_bad_index_is_reported_not_faulted():
    m = lib()
    wl = _case("mixtral", T=64, d=256)
    cfg = config_of(wl)
    inp = moe_inputs.make_router_inputs(wl, 0, "cuda")
    idx = torch.zeros((wl.T, wl.k), dtype=torch.int32, device="cuda")
    idx[:, 1] = 1
    idx[5, 0] = wl.E + 3
    logits = torch.zeros((wl.T, wl.E), device="cuda")
    dw = torch.ones((wl.T, wl.k), device="cuda")
    dW = torch.empty((wl.E, wl.d), device="cuda")
    ws = m.router_backward_workspace(cfg)
    m.moe_router_backward(cfg, inp["x"], inp["w_gate"], logits, idx, dw, None, 0.0, 0.0, None, dW,
                          None, ws)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == -1
    assert m.sync_status(ws) == 0          # the status word is cleared once read


@pytest.mark.parametrize("T,k,E", [(4096, 2, 8), (3000, 6, 64), (777, 8, 256)])
def test_bias_update_bitexact(T, k, E):
    m = lib()
    wl = _case("v3" if E == 256 else "dsmoe16b" if E == 64 else "mixtral", T=T, d=256, E=E, k=k)
    cfg = config_of(wl)
    rng = np.random.default_rng(T)
    counts = rng.multinomial(T * k, np.full(E, 1.0 / E))
    if (T * k) % E == 0:
        # place loads exactly at the mean, one above and one below
        mean = T * k // E
        counts = np.full(E, mean)
        counts[0] += 5
        counts[1] -= 5
        counts[2] += 1
        counts[3] -= 1
    f32 = (counts / T).astype(np.float32)
    b0 = moe_inputs.make_grad_inputs(wl, 0, "cuda")["bias_state"]
    want = O.bias_update(b0.cpu().numpy(), counts, T, k, 0.001)
    b = b0.clone()
    m.moe_bias_update(cfg, torch.from_numpy(f32).cuda(), b, 0.001)
    torch.cuda.synchronize()
    got = b.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    if (T * k) % E == 0:
        assert got[4] == b0[4].item() and got[0] < b0[0].item() and got[1] > b0[1].item()

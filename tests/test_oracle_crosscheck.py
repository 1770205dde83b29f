"""The C++ oracle against an independent restatement of the same equations in numpy
(oracle/moe_oracle_np.py, written separately, matrix products through numpy), and the sampled
token-by-token forward against the whole-layer forward.  CPU only.

Two implementations that share no code agreeing on random layers of every routing mode is a
cross-check, not a pin by itself: the pins are in test_oracle*.py.  The sampled forward is the
expected value of every full-size GPU output check, so it is pinned here against the layer
forward it must reproduce: with and without shared experts, with capacity drops, and with the
expert weights fetched one expert at a time."""
import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from oracle import moe_oracle_np as N


def _host(inp):
    return {k: moe_inputs.to_f64(v) for k, v in inp.items()}


LAYERS = {
    "softmax_cap": dict(name="mixtral", T=300, d=64, E=8, k=2, F=96, capacity_factor=1.0),
    "collapsed_cap": dict(name="mixtral_collapsed", T=200, d=64, E=8, k=2, F=64,
                          capacity_factor=1.25),
    "switch": dict(name="mixtral", T=150, d=64, E=8, k=1, F=64, renormalize=False,
                   capacity_factor=1.0),
    "v3_like": dict(name="v3", T=120, d=64, E=32, k=4, F=64, F_shared=64),
    "dsmoe_like": dict(name="dsmoe16b", T=160, d=64, E=16, k=3, F=64, F_shared=32),
    "tiny_f32": dict(name="tiny"),
}


@pytest.mark.parametrize("case", sorted(LAYERS))
def test_layer_matches_numpy_restatement(case):
    spec = dict(LAYERS[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    h = _host(moe_inputs.make_inputs(wl))
    a = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    b = N.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    assert np.array_equal(a["g32"], b["g32"])
    assert np.array_equal(a["idx"], b["idx"])
    assert np.abs(a["w"] - b["w"]).max() < 1e-14
    for key in ("counts", "kept", "offsets", "pos", "row_of", "perm"):
        assert np.array_equal(a["disp"][key], b["disp"][key]), key
    assert a["disp"]["n_dropped"] == b["disp"]["n_dropped"]
    scale = np.sqrt(np.mean(b["out"] ** 2))
    assert np.abs(a["out"] - b["out"]).max() < 1e-12 * scale
    for key in ("f", "P"):
        assert np.abs(a["stats"][key] - b["stats"][key]).max() < 1e-13
    for key in ("l_balance", "z_loss", "l_balance_per_k"):
        assert a["stats"][key] == pytest.approx(b["stats"][key], rel=1e-13)


def test_expert_choice_matches_numpy_restatement():
    wl = moe_inputs.workload("dsmoe16b_ec", T=192, d=64, E=8, k=2, F=32, F_shared=32)
    h = _host(moe_inputs.make_inputs(wl))
    a = O.moe_forward_expert_choice(wl, h["x"], h["w_gate"], h["w13"], h["w2"], h["ws13"],
                                    h["ws2"])
    b = N.moe_forward_expert_choice(wl, h["x"], h["w_gate"], h["w13"], h["w2"], h["ws13"],
                                    h["ws2"])
    assert np.array_equal(a["tokens"], b["tokens"])
    assert np.abs(a["weights"] - b["weights"]).max() < 1e-15
    for key in ("ptr", "rows", "experts"):
        assert np.array_equal(a["csr"][key], b["csr"][key]), key
    assert np.abs(a["out"] - b["out"]).max() < 1e-12 * np.sqrt(np.mean(b["out"] ** 2))


def test_backward_and_fp8_match_numpy_restatement():
    rng = np.random.default_rng(3)
    g = rng.standard_normal((40, 16)) * 2
    idx = N.topk_desc(g, 3)
    assert np.array_equal(O.topk_desc(g, 3), idx)
    dw = rng.standard_normal((40, 3))
    f = np.bincount(idx.reshape(-1), minlength=16) / 40.0
    for score in ("softmax", "sigmoid"):
        a = O.router_backward(g, idx, dw, f, 0.01, 0.001, score, True, 2.5)
        b = N.router_backward(g, idx, dw, f, 0.01, 0.001, score, True, 2.5)
        assert np.abs(a - b).max() < 1e-15
    x = rng.standard_normal((40, 24))
    wg = rng.standard_normal((16, 24))
    for u, v in zip(O.router_param_grads(x, wg, g), N.router_param_grads(x, wg, g)):
        assert np.abs(u - v).max() < 1e-12
    V = (rng.standard_normal((30, 50)) * 10.0 ** rng.uniform(-4, 3, (30, 1))).astype(np.float32)
    ca, sa = O.quantize_rows_fp8(V)
    cb, sb = N.quantize_rows_fp8(V)
    assert np.array_equal(ca, cb) and np.array_equal(sa, sb)


# ---------------------------------------------------------------------------------------------
# the sampled forward (expected value of the full-size GPU checks) against the layer forward
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["softmax_cap", "collapsed_cap", "v3_like", "dsmoe_like"])
@pytest.mark.parametrize("source", ["float64", "bf16_tensors"])
def test_sampled_forward_equals_layer_forward(case, source):
    spec = dict(LAYERS[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    inp = moe_inputs.make_inputs(wl)
    h = _host(inp)
    res = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                        h["ws2"])
    row_of = res["disp"]["row_of"]
    if wl.capacity_factor:
        assert res["disp"]["n_dropped"] > 0          # some sampled pairs are dropped
    calls = []
    src = h if source == "float64" else inp          # bf16 torch tensors straight through

    def fetch(e):
        calls.append(e)
        return src["w13"][e], src["w2"][e]

    def shared():
        return None if src["ws13"] is None else (src["ws13"], src["ws2"])

    tokens = np.array([0, 7, wl.T // 2, wl.T - 1] + list(range(10, wl.T, 37)))
    got = O.moe_forward_sampled(src["x"], res["idx"], res["w"], row_of, fetch, shared, tokens)
    want = res["out"][tokens]
    assert np.abs(got - want).max() <= 1e-12 * np.sqrt(np.mean(res["out"] ** 2))
    # each needed expert is fetched exactly once, and only those
    need = {int(e) for e in np.unique(res["idx"][tokens][row_of[tokens] >= 0])}
    assert sorted(calls) == sorted(need)


def test_sampled_forward_catches_a_slot_slip():
    # the same selection with the weights of a token's two choices swapped must give a
    # different answer: the sampled forward reads w[t, j] for the slot j of idx[t, j]
    wl = moe_inputs.workload("mixtral", T=64, d=64, E=8, k=2, F=64)
    h = _host(moe_inputs.make_inputs(wl))
    res = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"])
    w_bad = res["w"][:, ::-1].copy()
    tok = np.arange(8)
    good = O.moe_forward_sampled(h["x"], res["idx"], res["w"], res["disp"]["row_of"],
                                 lambda e: (h["w13"][e], h["w2"][e]), None, tok)
    bad = O.moe_forward_sampled(h["x"], res["idx"], w_bad, res["disp"]["row_of"],
                                lambda e: (h["w13"][e], h["w2"][e]), None, tok)
    assert np.abs(good - res["out"][tok]).max() < 1e-12
    assert np.abs(bad - res["out"][tok]).max() > 1e-3


def test_bf16_bits_are_widened_exactly():
    # a bf16 tensor passed as its 16 bits and the same values as float64 give identical logits
    wl = moe_inputs.workload("v3", T=50, d=64, E=32, F=64, F_shared=64)
    inp = moe_inputs.make_router_inputs(wl)
    assert inp["x"].dtype == torch.bfloat16
    a = O.router_logits(inp["x"], inp["w_gate"])
    b = O.router_logits(moe_inputs.to_f64(inp["x"]), moe_inputs.to_f64(inp["w_gate"]))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])

"""Pins of the oracle's FP8 (E4M3) quantisation and FP8 layer (CPU only).

The E4M3 rounding is checked against torch's float8_e4m3fn conversion (a library routine,
independent of the oracle) on the whole grid, on every tie point and on random values; the
per-row quantiser against its defining properties; the FP8 layer against the pinned bf16 layer,
exactly when the quantisation is made the identity and statistically otherwise.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O


def _grid():
    """Every finite E4M3 value, from all 256 byte patterns (NaN patterns dropped)."""
    b = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    return np.unique(b[np.isfinite(b)].astype(np.float64))


def test_grid_matches_the_format():
    g = _grid()
    pos = g[g > 0]
    assert g.max() == 448.0 and g.min() == -448.0
    assert pos.min() == 2.0 ** -9                      # smallest subnormal
    assert len(pos) == 126                             # 7 subnormals + 15 binades x 8 - 1 NaN
    assert np.array_equal(O.e4m3_round(g.astype(np.float32)), g)


def test_rounding_matches_torch_on_ties_and_random_values():
    g = _grid()
    pos = g[g >= 0]
    mids = (pos[:-1] + pos[1:]) / 2                    # exact ties between neighbours
    nudged = np.concatenate([mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    rng = np.random.default_rng(0)
    rand = rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))
    v = np.concatenate([mids, -mids, nudged, -nudged, rand]).astype(np.float32)
    v = v[np.abs(v) <= 464.0]                          # torch does not saturate beyond 464
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = O.e4m3_round(v)
    assert np.array_equal(got, want)


def test_saturation():
    got = O.e4m3_round(np.array([465.0, 1e6, -500.0, 3.4e38], np.float32))
    assert got.tolist() == [448.0, 448.0, -448.0, 448.0]


def test_row_quantiser_properties():
    rng = np.random.default_rng(1)
    V = rng.standard_normal((64, 300)).astype(np.float32) * np.exp(rng.uniform(-8, 8, (64, 1)))
    V[3] = 0.0
    c, s = O.quantize_rows_fp8(V)
    assert s[3] == 0 and not c[3].any()
    amax_at = np.argmax(np.abs(V), axis=1)
    rows = np.arange(64) != 3
    assert np.all(np.abs(c[rows, amax_at[rows]]) == 448.0)
    # relative error 2^-4 in the normal range, absolute 2^-10 x scale below it
    deq = c * s[:, None]
    err = np.abs(deq - V.astype(np.float64))
    assert np.all(err <= 2.0 ** -4 * np.abs(V) + 2.0 ** -10 * s[:, None] + 1e-300)
    # an exactly representable row (grid values times a power of two) is kept exactly
    g = _grid()
    row = rng.choice(g, 50)
    row[7] = 448.0
    Vx = (row * 2.0 ** -5).astype(np.float32)[None, :]
    cx, sx = O.quantize_rows_fp8(Vx)
    assert np.array_equal(cx[0] * sx[0], Vx[0].astype(np.float64)) and sx[0] == 2.0 ** -5


def _small(name, **kw):
    wl = moe_inputs.workload(name, **kw)
    inp = moe_inputs.make_inputs(wl)
    h = {k: moe_inputs.to_f64(v) for k, v in inp.items()}
    return wl, h


@pytest.mark.parametrize("case", [dict(name="v3", T=24, d=128, E=16, F=128, F_shared=128),
                                  dict(name="mixtral", T=20, d=128, E=8, F=256)])
def test_fp8_layer_with_identity_quantisation_is_the_bf16_layer(case):
    wl, h = _small(**case)
    want = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                         h["ws2"])["out"]
    with O.fp8_identity_quantisation():
        wq = O.fp8_expert_weights(h["w13"], h["w2"], h["ws13"], h["ws2"])
        got, _ = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq)
        # the same with the weights quantised inside the sampled path
        disp = O.dispatch(*_route_disp(wl, h))
        r = O.route(wl, h["x"], h["w_gate"], h["bias"])
        part = O.moe_forward_fp8_sampled(h["x"], r["idx"], r["w"], disp["row_of"],
                                         lambda e: (h["w13"][e], h["w2"][e]),
                                         lambda: (h["ws13"], h["ws2"]) if h["ws13"] is not None
                                         else None, [0, 5, wl.T - 1])
    # identical up to float64 rounding (h goes through float32 in the fp8 path)
    scale = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(got - want)) <= 1e-6 * scale
    assert np.max(np.abs(part - want[[0, 5, wl.T - 1]])) <= 1e-6 * scale
    # outside the context the quantiser is E4M3 again
    assert np.max(np.abs(O.fp8_expert_weights(h["w13"], h["w2"])["w2"] - h["w2"])) > 0


def _route_disp(wl, h):
    r = O.route(wl, h["x"], h["w_gate"], h["bias"])
    return r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E)


@pytest.mark.parametrize("case", [dict(name="v3", T=24, d=256, E=16, F=256, F_shared=256),
                                  dict(name="mixtral", T=20, d=256, E=8, F=512)])
def test_fp8_layer_error_against_bf16_layer(case):
    """E4M3 keeps 4 significant bits: a value with significand m in [1, 2) is rounded by up to
    2^-4/m relative, an RMS of about 2^-4 sqrt(E[1/m^2]/3) ~ 2.5% per operand.  Four operands
    (x, W1|W3, h, W2) give ~5-6% of the output RMS: clearly nonzero and far below the size of
    any structural mistake."""
    wl, h = _small(**case)
    want = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                         h["ws2"])["out"]
    wq = O.fp8_expert_weights(h["w13"], h["w2"], h["ws13"], h["ws2"])
    got, _ = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq)
    rel = np.sqrt(np.mean((got - want) ** 2)) / np.sqrt(np.mean(want ** 2))
    assert 0.01 < rel < 0.10, rel


@pytest.mark.parametrize("case", [dict(name="v3", T=24, d=128, E=16, F=128, F_shared=128),
                                  dict(name="mixtral", T=20, d=128, E=8, F=256,
                                       capacity_factor=1.0)])
def test_fp8_layer_is_the_layer_on_dequantised_operands(case):
    """The FP8 layer is the plain layer evaluated on dequantised operands: x quantised per
    token, every weight row per row, h (rounded to float32) per row before the down product.
    Composed here with numpy products from the row quantiser alone (pinned above against
    torch's E4M3 conversion), so a scale applied twice, or to the wrong axis, or an operand
    left unquantised, moves the output by whole quantisation steps."""
    wl, h = _small(**case)
    wq = O.fp8_expert_weights(h["w13"], h["w2"], h["ws13"], h["ws2"])
    got, r = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq)
    xc, xs = O.quantize_rows_fp8(h["x"].astype(np.float32))
    xq = xc * xs[:, None]

    def ffn(rows, W13, W2):
        F = W13.shape[0] // 2
        a, b = rows @ W13[:F].T, rows @ W13[F:].T
        hh = (a / (1.0 + np.exp(-a)) * b).astype(np.float32)
        hc, hs = O.quantize_rows_fp8(hh)
        return (hc * hs[:, None]) @ W2.T

    disp = O.dispatch(r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E))
    want = np.zeros_like(got) if wq["ws13"] is None else ffn(xq, wq["ws13"], wq["ws2"])
    n_routed = 0
    for t in range(wl.T):
        for j in range(wl.k):
            if disp["row_of"][t, j] >= 0:
                e = int(r["idx"][t, j])
                want[t] += r["w"][t, j] * ffn(xq[t:t + 1], wq["w13"][e], wq["w2"][e])[0]
                n_routed += 1
    assert n_routed > 0
    if wl.capacity_factor:
        assert disp["n_dropped"] > 0 or n_routed == wl.T * wl.k
    scale = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(got - want)) <= 1e-9 * scale
    # and it is not the unquantised layer: the comparison above resolves quantisation steps
    plain = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                          h["ws2"])["out"]
    assert np.max(np.abs(plain - want)) > 1e-3 * scale


def test_fp8_layer_token_subset_matches_full():
    wl, h = _small("v3", T=24, d=128, E=16, F=128, F_shared=128)
    wq = O.fp8_expert_weights(h["w13"], h["w2"], h["ws13"], h["ws2"])
    full, _ = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq)
    part, _ = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq, tokens=[3, 17, 0])
    assert np.allclose(part, full[[3, 17, 0]], rtol=0, atol=1e-12)


def test_fp8_sampled_matches_full():
    wl, h = _small("v3", T=24, d=128, E=16, F=128, F_shared=128)
    wq = O.fp8_expert_weights(h["w13"], h["w2"], h["ws13"], h["ws2"])
    full, r = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq)
    disp = O.dispatch(r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E))
    toks = [5, 0, 23]
    part = O.moe_forward_fp8_sampled(h["x"], r["idx"], r["w"], disp["row_of"],
                                     lambda e: (h["w13"][e], h["w2"][e]),
                                     lambda: (h["ws13"], h["ws2"]), toks)
    assert np.allclose(part, full[toks], rtol=0, atol=1e-12)

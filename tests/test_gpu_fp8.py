"""GPU parity of the FP8 (E4M3) expert path against the oracle's quantised layer.

Both sides quantise per row with float32 decisions, so the weight and token codes and scales
are bit-exact.  h is formed from float32 accumulations on the device and from float64 products
in the oracle, so an h value within rounding distance of an E4M3 tie may take the neighbouring
code; such a flip moves the outputs of its token row by about 2^-3 |h| |W2| w.  The bars:
  * routing, dispatch and statistics as in the bf16 layer (the same bf16 router);
  * output max |err| <= 2e-2 x RMS (the layer bar);
  * median |err| <= 1e-4 x RMS: away from the rare flips the device computes the quantised
    layer up to float32 accumulation.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = "cuda"
FP8_OUT_TOL = 2e-2
FP8_OUT_MEDIAN = 1e-4


def _decode(codes):
    return codes.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def test_quantize_rows_bitexact():
    m = U.lib()
    g = torch.Generator(device="cpu").manual_seed(7)
    rows, cols = 300, 256
    v = torch.randn(rows, cols, generator=g) * torch.exp(torch.empty(rows, 1).uniform_(-20, 20,
                                                                                 generator=g))
    v[5] = 0.0
    v[7] = torch.randn(cols, generator=g) * 1e-4       # quantised into the subnormal codes too
    v[9, :] = 0.0
    v[9, 3] = -2.5                                     # a single nonzero entry
    vb = v.to(torch.bfloat16).to(DEV)
    for src in (vb, vb.reshape(3, 100, cols)):
        codes, scales = m.quantize_fp8(src)
        torch.cuda.synchronize()
        want_c, want_s = O.quantize_rows_fp8(moe_inputs.to_f64(src).reshape(-1, cols))
        assert np.array_equal(_decode(codes).reshape(-1, cols), want_c)
        got_s = scales.cpu().numpy()
        assert np.array_equal(got_s.view(np.uint32), want_s.astype(np.float32).view(np.uint32))


def _quantize_weights(inp):
    m = U.lib()
    q = {}
    for key in ("w13", "w2", "ws13", "ws2"):
        q[key] = m.quantize_fp8(inp[key]) if inp[key] is not None else (None, None)
    return q


def _run_fp8(wl, inp, q, T=None):
    m = U.lib()
    cfg = U.config_of(wl, T)
    T, E, k = cfg.T, cfg.E, cfg.k
    out = torch.empty((T, wl.d), dtype=torch.float32, device=DEV)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    w = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    f = torch.zeros(E, dtype=torch.float32, device=DEV)
    P = torch.zeros(E, dtype=torch.float32, device=DEV)
    lb = torch.zeros(1, dtype=torch.float32, device=DEV)
    z = torch.zeros(1, dtype=torch.float32, device=DEV)
    nd = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    ws = m.fp8_workspace(cfg)
    m.moe_forward_fp8(cfg, inp["x"], inp["w_gate"], inp["bias"], *q["w13"], *q["w2"], *q["ws13"],
                      *q["ws2"], out, idx, w, f, P, lb, z, nd, ws)
    torch.cuda.synchronize()
    st = m.sync_status(ws)
    assert st == 0, m.status_string(st)
    return {"out": out.cpu().numpy().astype(np.float64), "idx": idx.cpu().numpy(),
            "w": w.cpu().numpy().astype(np.float64), "f": f.cpu().numpy(),
            "P": P.cpu().numpy(), "l_balance": float(lb.item()), "z_loss": float(z.item()),
            "n_dropped": int(nd.item())}


def _compare_out(got, ref, report):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(got - ref)
    report["max_over_rms"] = float(err.max()) / rms
    report["median_over_rms"] = float(np.median(err)) / rms
    assert err.max() <= FP8_OUT_TOL * rms, report
    assert np.median(err) <= FP8_OUT_MEDIAN * rms, report


SMALL = {
    "v3_b1": dict(name="v3", T=1, d=256, E=64, F=256, F_shared=256),
    "v3_b8": dict(name="v3", T=8, d=512, E=64, F=256, F_shared=384),
    "v3_b64": dict(name="v3", T=64, d=256, E=64, F=384, F_shared=256),
    "mixtral_b32": dict(name="mixtral", T=32, d=256, E=8, F=512),
    "mixtral_b300_chunks": dict(name="mixtral", T=300, d=256, E=8, F=256),
    "dsmoe_b100_two_shared": dict(name="dsmoe16b", T=100, d=256, E=64, F=256, F_shared=256),
    "collapsed_b256_cap": dict(name="mixtral_collapsed", T=256, d=256, F=256,
                               capacity_factor=1.0),
}


@pytest.mark.parametrize("case", list(SMALL))
def test_fp8_forward_small(case):
    wl = moe_inputs.workload(**SMALL[case])
    inp = moe_inputs.make_inputs(wl, device=DEV)
    h = U.host(inp)
    q = _quantize_weights(inp)
    # the weight codes are the oracle's
    c13, s13 = O.quantize_rows_fp8(h["w13"].reshape(-1, wl.d))
    assert np.array_equal(_decode(q["w13"][0]).reshape(-1, wl.d), c13)
    assert np.array_equal(q["w13"][1].cpu().numpy(), s13.astype(np.float32))
    gpu = _run_fp8(wl, inp, q)
    wq = O.fp8_expert_weights(h["w13"], h["w2"], h["ws13"], h["ws2"])
    ref_out, r = O.moe_forward_fp8(wl, h["x"], h["w_gate"], h["bias"], wq)
    report = {}
    ok = U.compare_routing(wl, gpu, r, h["bias"], report)
    if ok.all():
        U.compare_stats(gpu, O.aux_stats(r["g32"], r["idx"], wl.E, wl.score), report)
        disp = O.dispatch(r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E))
        assert gpu["n_dropped"] == disp["n_dropped"]
    _compare_out(gpu["out"][ok], ref_out[ok], report)
    # and FP8 approximates the bf16 layer to the expected few percent
    bf16 = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                         h["ws2"])["out"]
    rel = np.sqrt(np.mean((gpu["out"] - bf16) ** 2)) / np.sqrt(np.mean(bf16 ** 2))
    assert 0.01 < rel < 0.10, rel


FULL = {"v3_b1": ("v3", 1, 1), "v3_b8": ("v3", 8, 4), "v3_b64": ("v3", 64, 4),
        "v3_b256": ("v3", 256, 6), "mixtral_b32": ("mixtral", 32, 6)}


@pytest.mark.parametrize("case", list(FULL))
def test_fp8_forward_full_size(case):
    """Full-size expert weights at a decode batch: routing on every token, outputs on sampled
    tokens (the oracle quantises only the experts those tokens use)."""
    name, B, n_sample = FULL[case]
    wl = moe_inputs.workload(name, T=B)
    inp = moe_inputs.make_inputs(wl, device=DEV)
    q = _quantize_weights(inp)
    gpu = _run_fp8(wl, inp, q)
    x64 = moe_inputs.to_f64(inp["x"])
    w64 = moe_inputs.to_f64(inp["w_gate"])
    bias = moe_inputs.to_f64(inp["bias"])
    r = O.route(wl, x64, w64, bias)
    report = {}
    ok = U.compare_routing(wl, gpu, r, bias, report)
    disp = O.dispatch(r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E))
    toks = np.nonzero(ok)[0][np.linspace(0, ok.sum() - 1, n_sample).astype(int)]
    ref = O.moe_forward_fp8_sampled(x64, r["idx"], r["w"], disp["row_of"],
                                    U.expert_weight_fetcher(inp), U.shared_fetcher(inp), toks)
    _compare_out(gpu["out"][toks], ref, report)

"""Seeded random layer configurations against the oracle (GPU).

Each case draws a valid configuration from the whole space the C ABI accepts: expert counts,
k, group limits with sigmoid scoring, expert choice, capacity factors (including ones that drop
pairs), renormalisation, route scale, shared experts, odd token counts, and the float32 path.
The library then picks its own kernels for the case (prefill or decode, single-CTA or pair, the
GEMM's combine or the combine pass).  Every case is held to the same bars as the named cases:
selections bit-exact outside near ties, statistics within 1e-5 relative, the output within
2e-2 (bf16) or 1e-4 (float32) of its RMS.
"""
import numpy as np
import pytest

import moe_inputs
from oracle import moe_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

N_CASES = 24


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    f32 = rng.random() < 0.15
    d = int(rng.choice([64, 96]) if f32 else rng.choice([128, 256, 384, 512]))
    F = int(rng.choice([64, 128]) if f32 else rng.choice([128, 256, 384]))
    E = int(rng.choice([1, 2, 4, 6, 8, 16, 32, 48, 64]))
    k = int(rng.integers(1, min(8, E) + 1))
    T = int(rng.choice([1, 3, 17, 64, 100, 255, 256, 257, 511, 600]))
    score, routing, n_groups, topk_groups = "softmax", "token_choice", 1, 1
    r = rng.random()
    if r < 0.35:
        score = "sigmoid"
        divisors = [g for g in (2, 4, 8) if E % g == 0 and E // g >= 2]
        if divisors and rng.random() < 0.7:
            n_groups = int(rng.choice(divisors))
            per = E // n_groups
            lo = max(1, -(-k // per))
            topk_groups = int(rng.integers(lo, n_groups + 1))
    elif r < 0.5 and T * k // E >= 1:
        routing = "expert_choice"
    shared = 0 if rng.random() < 0.5 else int(rng.choice([64, 128]) if f32 else
                                              rng.choice([128, 256]))
    cf = float(rng.choice([0.0, 0.0, 1.0, 1.25, 2.0])) if routing == "token_choice" else 0.0
    renorm = bool(rng.random() < 0.8) if routing == "token_choice" else True
    scale = float(rng.choice([1.0, 2.5])) if routing == "token_choice" else 1.0
    bias = 0.1 if score == "sigmoid" and rng.random() < 0.7 else 0.0
    return moe_inputs.Workload(
        f"random{i}", T=T, d=d, E=E, k=k, F=F, n_shared=1 if shared else 0, F_shared=shared,
        score=score, routing=routing, n_groups=n_groups, topk_groups=topk_groups,
        renormalize=renorm, route_scale=scale, capacity_factor=cf,
        dtype="f32" if f32 else "bf16", bias_range=bias)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(i):
    wl = _draw(i)
    m = U.lib()
    assert m.check_config(U.config_of(wl)) == 0, wl
    inp = moe_inputs.make_inputs(wl, device="cuda")
    h = U.host(inp)
    gpu = U.run_forward(wl, inp)
    tol = U.OUT_TOL_F32 if wl.dtype == "f32" else U.OUT_TOL_BF16
    report = {"case": str(wl)}
    if wl.routing == "expert_choice":
        ref = O.moe_forward_expert_choice(wl, h["x"], h["w_gate"], h["w13"], h["w2"], h["ws13"],
                                          h["ws2"])
        U.compare_stats(gpu, ref["stats"], report)
        U.compare_out(gpu["out"].float().cpu().numpy(), ref["out"], tol, report)
        return
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                        h["ws2"])
    ok = U.compare_routing(wl, gpu, ref, h["bias"], report)
    if ok.all():
        U.compare_stats(gpu, ref["stats"], report)
        assert gpu["n_dropped"] == ref["disp"]["n_dropped"], report
    U.compare_out(gpu["out"].float().cpu().numpy()[ok], ref["out"][ok], tol, report)

"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and compare it with the
oracle under the stated tolerances."""
import numpy as np
import torch

import moe_inputs
from oracle import moe_oracle as O

# tolerances (stated once, used by every parity test)
STATS_RTOL = 1e-5          # f_i, P_i, L_balance, z-loss: relative
WEIGHT_ATOL = 1e-5         # gate weights (fp32 on both sides)
OUT_TOL_BF16 = 2e-2        # max-abs error <= 2e-2 x RMS of the oracle's output (bf16 path)
OUT_TOL_F32 = 1e-4         # same rule for the float32 path
TIE_REL = 1e-6             # near-tie window on the deciding scores


def lib():
    import top_routing_expert_scoring_b300 as m
    return m


def config_of(wl, T=None, out_dtype="f32"):
    return lib().make_config(T or wl.T, wl.d, wl.E, wl.k, wl.F, wl.F_sh, wl.score, wl.routing,
                             wl.n_groups, wl.topk_groups, wl.renormalize, wl.route_scale,
                             wl.capacity_factor, wl.dtype, out_dtype)


def host(inp):
    return {k: moe_inputs.to_f64(v) for k, v in inp.items()}


def run_forward(wl, inp, cfg=None):
    """moe_forward through the C ABI; returns the outputs on the host plus the workspace."""
    m = lib()
    cfg = cfg or config_of(wl)
    dev = inp["x"].device
    T, E, k = cfg.T, cfg.E, cfg.k
    out_dt = torch.float32 if cfg.out_dtype == 1 else torch.bfloat16
    out = torch.empty((T, wl.d), dtype=out_dt, device=dev)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    w = torch.zeros((T, k), dtype=torch.float32, device=dev)
    f = torch.zeros(E, dtype=torch.float32, device=dev)
    P = torch.zeros(E, dtype=torch.float32, device=dev)
    lb = torch.zeros(1, dtype=torch.float32, device=dev)
    z = torch.zeros(1, dtype=torch.float32, device=dev)
    nd = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ws = m.workspace(cfg, dev)
    m.moe_forward(cfg, inp["x"], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"], inp["ws13"],
                  inp["ws2"], out, idx, w, f, P, lb, z, nd, ws)
    torch.cuda.synchronize()
    st = m.sync_status(ws)
    assert st == 0, m.status_string(st)
    return {"out": out, "idx": idx.cpu().numpy(), "w": w.cpu().numpy().astype(np.float64),
            "f": f.cpu().numpy(), "P": P.cpu().numpy(), "l_balance": float(lb.item()),
            "z_loss": float(z.item()), "n_dropped": int(nd.item()), "ws": ws, "cfg": cfg}


def deciding_gaps(wl, r, bias):
    """Relative gap between the k-th and (k+1)-th selection keys (and, with a group limit, the
    kept and first dropped group scores) of every token, from the oracle's float32 keys."""
    g32 = r["g32"]
    T, E = g32.shape
    if wl.score == "softmax":
        keys = g32.astype(np.float64)
        gaps = []
    else:
        s32 = O.sigmoid(g32).astype(np.float32)
        sb = (s32 + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
        gaps = []
        if wl.n_groups > 1 and wl.topk_groups < wl.n_groups:
            per = E // wl.n_groups
            top2 = -np.sort(-sb.reshape(T, wl.n_groups, per), axis=-1)[..., :2]
            gs = np.sort((top2[..., 0] + top2[..., 1]).astype(np.float32), axis=1)[:, ::-1]
            a, b = gs[:, wl.topk_groups - 1].astype(np.float64), gs[:, wl.topk_groups].astype(np.float64)
            gaps.append((a - b) / np.maximum(np.abs(a), 1e-30))
            keep = O.topk_desc(top2[..., 0] + top2[..., 1], wl.topk_groups)
            mask = np.ones((T, wl.n_groups), bool)
            np.put_along_axis(mask, keep.astype(np.int64), False, axis=1)
            sb = np.where(np.repeat(mask, per, axis=1), -np.inf, sb)
        keys = sb.astype(np.float64)
    if wl.k < E:
        srt = -np.sort(-keys, axis=1)
        a, b = srt[:, wl.k - 1], srt[:, wl.k]
        with np.errstate(invalid="ignore"):
            gaps.append(np.where(np.isfinite(b), (a - b) / np.maximum(np.abs(a), 1e-30), np.inf))
    if not gaps:
        return np.full(T, np.inf)
    return np.min(np.stack(gaps), axis=0)


def compare_routing(wl, gpu, r, bias, report):
    """Indices bit-exact except reported near-tie tokens; weights within WEIGHT_ATOL.
    Returns the mask of tokens whose selection is compared (and matched)."""
    gaps = deciding_gaps(wl, r, bias)
    near = gaps < TIE_REL
    mism = (gpu["idx"] != r["idx"]).any(axis=1)
    report["near_tie_tokens"] = int(near.sum())
    report["excused_mismatches"] = int((mism & near).sum())
    bad = np.nonzero(mism & ~near)[0]
    assert len(bad) == 0, f"index mismatch outside the near-tie window at tokens {bad[:10]} " \
                          f"(gaps {gaps[bad[:10]]})"
    ok = ~mism
    werr = np.abs(gpu["w"][ok] - r["w"][ok]).max() if ok.any() else 0.0
    report["weight_max_abs_err"] = float(werr)
    assert werr <= WEIGHT_ATOL, werr
    return ok


def compare_stats(gpu, st, report):
    for key in ("f", "P"):
        ref = st[key]
        err = np.abs(gpu[key] - ref).max() / max(np.abs(ref).max(), 1e-30)
        report[f"{key}_rel_err"] = float(err)
        assert err <= STATS_RTOL, (key, err)
    for key in ("l_balance", "z_loss"):
        err = abs(gpu[key] - st[key]) / max(abs(st[key]), 1e-30)
        report[f"{key}_rel_err"] = float(err)
        assert err <= STATS_RTOL, (key, err)


def compare_out(got, ref, tol, report, key="out", bf16_rounded=False):
    """max |got - ref| <= tol * RMS(ref).  When `got` was rounded to bf16 at the end, each
    element may also carry that rounding, up to 2^-8 |ref| (8-bit significand): the bound is
    then tol * RMS + 2^-8 |ref| element by element."""
    got = np.asarray(got, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    diff = np.abs(got - ref)
    err = float(diff.max())
    report[f"{key}_max_abs_err_over_rms"] = err / rms
    if bf16_rounded:
        excess = diff - 2.0 ** -8 * np.abs(ref)
        report[f"{key}_max_err_beyond_rounding_over_rms"] = float(excess.max()) / rms
        assert (excess <= tol * rms).all(), (float(excess.max()) / rms)
    else:
        assert err <= tol * rms, (err, rms, err / rms)


def expert_weight_fetcher(inp):
    """Per-expert host copies of the routed weights in their own dtype (the oracle widens bf16
    exactly), copied from wherever they live."""
    def fetch(e):
        return inp["w13"][e].to("cpu"), inp["w2"][e].to("cpu")
    return fetch


def shared_fetcher(inp):
    def fetch():
        if inp["ws13"] is None:
            return None
        return inp["ws13"].to("cpu"), inp["ws2"].to("cpu")
    return fetch


def coverage_tokens(offsets, perm, k, T, rng, n_random):
    """Tokens whose rows cover every expert's first and last row -- so every expert, its first
    M tile and its last (ragged) M tile are looked at -- plus n_random tokens drawn at random.
    offsets [E+1] and perm [T*k] describe the expert-ordered rows."""
    toks = set()
    E = len(offsets) - 1
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            toks.add(int(perm[lo]) // k)
            toks.add(int(perm[hi - 1]) // k)
    toks |= {int(t) for t in rng.choice(T, size=min(n_random, T), replace=False)}
    return np.array(sorted(toks), dtype=np.int64)

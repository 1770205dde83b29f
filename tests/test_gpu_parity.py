"""GPU-vs-oracle parity of the whole layer and of each stage, through the C ABI.

Bars: selected expert indices, counts, offsets, positions, permutation and drop set
bit-exact (tokens whose deciding scores differ by less than 1e-6 relative are reported and
excluded); statistics within 1e-5 relative; layer output max-abs error <= 2e-2 x RMS (bf16) or
1e-4 x RMS (float32 path).  Small cases span several tiles with ragged tails; the full-size
cases (the benchmark's launch configuration) compare routing and dispatch on every token and
the output on sampled tokens."""
import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(wl, device=DEV, seed=0):
    return moe_inputs.make_inputs(wl, seed=seed, device=device)


def _full_check(wl, inp, report, out_tol):
    """Whole-layer parity on a case small enough for the oracle's full forward."""
    h = U.host(inp)
    gpu = U.run_forward(wl, inp)
    if wl.routing == "expert_choice":
        ref = O.moe_forward_expert_choice(wl, h["x"], h["w_gate"], h["w13"], h["w2"], h["ws13"],
                                          h["ws2"])
        U.compare_stats(gpu, ref["stats"], report)
        U.compare_out(gpu["out"].float().cpu().numpy(), ref["out"], out_tol, report)
        return gpu, ref
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    ok = U.compare_routing(wl, gpu, ref, h["bias"], report)
    if ok.all():
        U.compare_stats(gpu, ref["stats"], report)
        assert gpu["n_dropped"] == ref["disp"]["n_dropped"]
        m = U.lib()
        _, row_of_p, offsets_p, _, _ = m.moe_workspace_views(gpu["cfg"], gpu["ws"])
        row_of = _read_i32(row_of_p, wl.T * wl.k).reshape(wl.T, wl.k)
        offsets = _read_i32(offsets_p, wl.E + 1)
        assert (row_of == ref["disp"]["row_of"]).all()
        assert (offsets == ref["disp"]["offsets"]).all()
    got = gpu["out"].float().cpu().numpy()
    U.compare_out(got[ok], ref["out"][ok], out_tol, report)
    return gpu, ref


class _DevArray:
    """Zero-copy view of n int32 values at a raw device address (the workspace views)."""
    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False),
                                         "version": 3, "strides": None}


def _read_i32(ptr, n):
    torch.cuda.synchronize()
    return torch.as_tensor(_DevArray(ptr, n), device=DEV).cpu().numpy()


# ---------------------------------------------------------------------------------------------
# small cases: full oracle forward
# ---------------------------------------------------------------------------------------------
SMALL = {
    # float32 path
    "tiny": dict(name="tiny"),
    "tiny_dense": dict(name="tiny_dense"),
    "tiny_uniform": dict(name="tiny_uniform"),
    # bf16: ragged M tiles, capacity drops, 3 N tiles in the gate/up GEMM
    "softmax_cap": dict(name="mixtral", T=700, d=256, F=384, capacity_factor=1.25),
    "softmax_collapsed_cap": dict(name="mixtral_collapsed", T=600, d=256, F=256,
                                  capacity_factor=1.0),
    # Switch routing: k = 1, the weight is the probability itself (no renormalisation)
    "switch_k1": dict(name="mixtral", T=500, d=256, F=256, k=1, renormalize=False,
                      capacity_factor=1.0),
    # bf16 DeepSeek-V3-like gate: sigmoid + bias, 8 groups keep 4, top-8, scale 2.5, shared
    "v3_like": dict(name="v3", T=333, d=256, E=64, F=256, F_shared=256),
    # bf16 DeepSeekMoE-like: 2 shared experts, d not a multiple of 256 (N=128 down tiles)
    "dsmoe_like": dict(name="dsmoe16b", T=1000, d=384, E=16, F=256, F_shared=128),
    # expert choice
    "ec_like": dict(name="dsmoe16b_ec", T=512, d=256, E=16, k=4, F=256, F_shared=128),
    # decode-sized batches (<= 64 rows per expert on average): swap-AB decode kernel, shared
    # experts folded into the same tile list
    "decode_b1": dict(name="v3", T=1, d=256, E=64, F=256, F_shared=256),
    "decode_b8": dict(name="v3", T=8, d=512, E=64, F=256, F_shared=384),
    "decode_b64": dict(name="v3", T=64, d=256, E=64, F=384, F_shared=256),
    "decode_mixtral_b32": dict(name="mixtral", T=32, d=512, F=384),
    "decode_collapsed_b256": dict(name="mixtral_collapsed", T=256, d=256, F=256),
    "decode_dsmoe_b100": dict(name="dsmoe16b", T=100, d=256, E=64, F=128, F_shared=128),
    # E = 256: router logits from the K-sliced decode kernel (4 and 2 slices); Top-k one CTA
    # per token (T <= 64) or one warp per token
    "decode_e256_b40": dict(name="v3", T=40, d=512, E=256, F=128, F_shared=128),
    # one-CTA-per-token Top-k with E not a multiple of 32 (idle threads in the last warp) and
    # with groups of 25 and 24 experts that straddle warps
    "topk_cta_e40": dict(name="mixtral", T=30, d=256, E=40, k=5, F=128),
    "topk_cta_e200_groups25": dict(name="v3", T=50, d=256, E=200, k=7, F=128, F_shared=128),
    "topk_cta_e96_groups24": dict(name="v3", T=37, d=256, E=96, k=8, F=128, n_shared=0,
                                  F_shared=0, n_groups=4, topk_groups=3),
    "decode_e256_b100": dict(name="v3", T=100, d=1024, E=256, F=128, F_shared=128),
    # prefill batches of a wide router (E % 32 == 0, T > 512): scoring, group limit, Top-k and
    # statistics terms in the router GEMM's epilogue, one thread per token
    "router_fused_softmax_e64": dict(name="mixtral", T=1000, d=256, E=64, k=6, F=128),
    "router_fused_v3_e256": dict(name="v3", T=700, d=256, E=256, F=128, F_shared=128),
    "router_fused_groups_of_64": dict(name="v3", T=600, d=256, E=128, k=6, F=128,
                                      F_shared=128, n_groups=2, topk_groups=1),
    # E = 96 (three 32-expert chunks) with a last tile of 20 tokens (M = 64 accumulator layout)
    "router_fused_e96_tail": dict(name="mixtral", T=1300, d=256, E=96, k=5, F=128),
    "router_fused_switch_e32": dict(name="mixtral", T=777, d=256, E=32, k=1, F=128,
                                    renormalize=False),
    "router_fused_sigmoid_one_group": dict(name="v3", T=900, d=256, E=64, k=6, F=128,
                                           F_shared=128, n_groups=1, topk_groups=1),
    # 153 tiles of 128 tokens on 148 CTAs: some CTAs route two tiles (double-buffered
    # accumulators, epilogue state reused), and the last tile has 44 rows
    "router_fused_two_tiles_per_cta": dict(name="v3", T=19500, d=128, E=64, k=4, F=128,
                                           F_shared=128, n_groups=2, topk_groups=1),
    "one_expert": dict(name="mixtral", T=130, d=128, E=1, k=1, F=128),
    # prefill path with E = 1, k = 1 and d = 256 (decode regime needs <= 64 rows per expert)
    "one_expert_d256": dict(name="mixtral", T=300, d=256, E=1, k=1, F=128),
}


def _router_env(case, monkeypatch):
    """The router_fused_* cases take the router GEMM with the routing epilogue whatever their E
    (by default only routers of >= 128 experts do)."""
    if case.startswith("router_fused_"):
        monkeypatch.setenv("MOE_B300_ROUTER", "fused")


@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_layer_parity(case, monkeypatch):
    _router_env(case, monkeypatch)
    spec = dict(SMALL[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    inp = _inputs(wl)
    report = {}
    tol = U.OUT_TOL_F32 if wl.dtype == "f32" else U.OUT_TOL_BF16
    _full_check(wl, inp, report, tol)
    print(case, report)


@pytest.mark.parametrize("case,ks1,ks2", [("decode_b8", 3, 3), ("decode_b8", 8, 1),
                                         ("decode_b1", 5, 3), ("decode_collapsed_b256", 3, 3)])
def test_decode_forced_k_slices(case, ks1, ks2, monkeypatch):
    """The decode GEMMs with K cut into slice counts the cost model may not pick (uneven
    slices of the K blocks, and a count above the K blocks, clamped), partials summed in slice
    order: the layer against the oracle under the same bar."""
    monkeypatch.setenv("MOE_B300_KSPLIT1", str(ks1))
    monkeypatch.setenv("MOE_B300_KSPLIT2", str(ks2))
    spec = dict(SMALL[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    inp = _inputs(wl)
    report = {}
    _full_check(wl, inp, report, U.OUT_TOL_BF16)
    print(case, ks1, ks2, report)


@pytest.mark.parametrize("case", ["v3_like", "softmax_cap"])
def test_bf16_output(case, monkeypatch):
    # the layer output rounded once to bf16: the bound adds that rounding (2^-8 |out|).  The
    # bf16 mode rounds the combine pass's float32 sum, so the float32 reference run below uses
    # that pass too (a k <= 2 float32 layer would otherwise add its terms in the down GEMM)
    monkeypatch.setenv("MOE_B300_COMBINE", "separate")
    spec = dict(SMALL[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    inp = _inputs(wl)
    cfg = U.config_of(wl, out_dtype="bf16")
    gpu = U.run_forward(wl, inp, cfg)
    assert gpu["out"].dtype == torch.bfloat16
    h = U.host(inp)
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    report = {}
    ok = U.compare_routing(wl, gpu, ref, h["bias"], report)
    U.compare_out(gpu["out"].float().cpu().numpy()[ok], ref["out"][ok], U.OUT_TOL_BF16, report,
                  bf16_rounded=True)
    f32 = U.run_forward(wl, inp)
    # the bf16 output is the float32 output rounded to nearest
    assert torch.equal(f32["out"].to(torch.bfloat16), gpu["out"])
    print(case, report)


def test_uniform_router_exact_ties():
    # W_gate = 0: every logit is exactly 0 on both sides, the tie rule alone decides
    wl = moe_inputs.workload("tiny_uniform")
    gpu = U.run_forward(wl, _inputs(wl))
    assert (gpu["idx"] == np.arange(wl.k)[None, :]).all()
    assert np.abs(gpu["w"] - 1.0 / wl.k).max() == 0
    assert gpu["l_balance"] == pytest.approx(wl.k, rel=1e-7)
    assert gpu["z_loss"] == pytest.approx(np.log(wl.E) ** 2, rel=1e-6)
    assert gpu["n_dropped"] == wl.T * wl.k - 160


def test_forward_is_deterministic():
    wl = moe_inputs.workload("v3", T=400, d=256, E=64, F=256, F_shared=256)
    inp = _inputs(wl)
    a = U.run_forward(wl, inp)
    b = U.run_forward(wl, inp)
    assert torch.equal(a["out"], b["out"])
    assert (a["idx"] == b["idx"]).all() and (a["w"] == b["w"]).all()
    assert (a["f"] == b["f"]).all() and (a["P"] == b["P"]).all()
    assert a["l_balance"] == b["l_balance"] and a["z_loss"] == b["z_loss"]


# ---------------------------------------------------------------------------------------------
# stage entry points
# ---------------------------------------------------------------------------------------------
def test_stage_entry_points():
    m = U.lib()
    wl = moe_inputs.workload("v3", T=700, d=256, E=64, F=256, F_shared=256, capacity_factor=1.25)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    h = U.host(inp)
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    T, E, k, d = wl.T, wl.E, wl.k, wl.d
    ws = m.workspace(cfg)
    i32 = dict(dtype=torch.int32, device=DEV)
    f32 = dict(dtype=torch.float32, device=DEV)
    logits = torch.empty((T, E), **f32)
    idx = torch.empty((T, k), **i32)
    w = torch.empty((T, k), **f32)
    m.moe_router_topk(cfg, inp["x"], inp["w_gate"], inp["bias"], logits, idx, w, ws)
    g = logits.cpu().numpy()
    # logits: fp32 accumulation vs the correctly rounded exact value
    assert np.abs(g - ref["g"]).max() <= 1e-5 * np.abs(ref["g"]).max()
    report = {}
    ok = U.compare_routing(wl, {"idx": idx.cpu().numpy(),
                                "w": w.cpu().numpy().astype(np.float64)}, ref, h["bias"], report)
    assert ok.all()
    f = torch.empty(E, **f32)
    P = torch.empty(E, **f32)
    lb = torch.empty(1, **f32)
    z = torch.empty(1, **f32)
    m.moe_aux_stats(cfg, logits, idx, f, P, lb, z, ws)
    U.compare_stats({"f": f.cpu().numpy(), "P": P.cpu().numpy(), "l_balance": lb.item(),
                     "z_loss": z.item()}, ref["stats"], report)
    # dispatch fed the oracle's indices: bit-exact
    oidx = torch.from_numpy(ref["idx"].astype(np.int32)).to(DEV)
    counts, kept = torch.empty(E, **i32), torch.empty(E, **i32)
    offsets = torch.empty(E + 1, **i32)
    pos, row_of = torch.empty((T, k), **i32), torch.empty((T, k), **i32)
    perm, nd = torch.empty(T * k, **i32), torch.empty(1, **i32)
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV)
    m.moe_dispatch(cfg, oidx, inp["x"], counts, kept, offsets, pos, row_of, perm, x_perm, nd, ws)
    D = ref["disp"]
    for name, t in [("counts", counts), ("kept", kept), ("offsets", offsets), ("pos", pos),
                    ("row_of", row_of), ("perm", perm)]:
        assert (t.cpu().numpy() == D[name]).all(), name
    assert nd.item() == D["n_dropped"] > 0
    nk = int(D["offsets"][-1])
    src = D["perm"][:nk] // k
    assert torch.equal(x_perm[:nk].cpu(), inp["x"].cpu()[torch.from_numpy(src.astype(np.int64))])
    # routed experts on the dispatched rows
    y_perm = torch.zeros((T * k, d), dtype=torch.float32, device=DEV)
    m.moe_expert_ffn(cfg, x_perm, offsets, inp["w13"], inp["w2"], y_perm, ws)
    U.compare_out(y_perm[:nk].float().cpu().numpy(), ref["y_rows"], U.OUT_TOL_BF16, report, "y")
    shared = torch.empty((T, d), dtype=torch.float32, device=DEV)
    m.moe_shared_ffn(cfg, inp["x"], inp["ws13"], inp["ws2"], shared, ws)
    U.compare_out(shared.float().cpu().numpy(), ref["shared"], U.OUT_TOL_BF16, report, "shared")
    out = torch.empty((T, d), dtype=torch.float32, device=DEV)
    ow = torch.from_numpy(ref["w"].astype(np.float32)).to(DEV)
    m.moe_combine(cfg, y_perm, row_of, ow, shared, out)
    U.compare_out(out.float().cpu().numpy(), ref["out"], U.OUT_TOL_BF16, report)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    print(report)


def test_expert_choice_entry_point():
    m = U.lib()
    wl = moe_inputs.workload("dsmoe16b_ec", T=777, d=256, E=16, k=4, F=256, F_shared=128)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    h = U.host(inp)
    g, g32 = O.router_logits(h["x"], h["w_gate"])
    ws = m.workspace(cfg)
    C = wl.T * wl.k // wl.E
    logits = torch.from_numpy(g32).to(DEV)
    tok = torch.empty((wl.E, C), dtype=torch.int32, device=DEV)
    tw = torch.empty((wl.E, C), dtype=torch.float32, device=DEV)
    ptr = torch.empty(wl.T + 1, dtype=torch.int32, device=DEV)
    rows = torch.empty(wl.E * C, dtype=torch.int32, device=DEV)
    m.moe_expert_choice(cfg, logits, tok, tw, ptr, rows, ws)
    tokens, weights, _ = O.expert_choice_route(g32, wl.k)
    csr = O.expert_choice_csr(tokens, wl.T)
    assert (tok.cpu().numpy() == tokens).all()
    assert np.abs(tw.cpu().numpy() - weights).max() <= U.WEIGHT_ATOL
    assert (ptr.cpu().numpy() == csr["ptr"]).all()
    assert (rows.cpu().numpy() == csr["rows"]).all()


@pytest.mark.parametrize("T,E,k", [(777, 16, 2), (50000, 16, 2), (4096, 256, 8), (300, 96, 5)])
@pytest.mark.parametrize("kind", ["normal", "few_levels"])
def test_expert_choice_selection_on_given_logits(T, E, k, kind):
    # the selection alone, bit for bit against the oracle: T = 777 keeps the expert's keys in
    # shared memory, T = 50000 reads them from global memory in every radix pass; E = 256 and
    # E = 96 (C not a multiple of anything in particular) run many CTAs; "few_levels"
    # logits take 7 values only, so each expert's C-th key is tied with thousands of tokens and
    # the lowest token indices must win
    m = U.lib()
    wl = moe_inputs.workload("dsmoe16b_ec", T=T, d=256, E=E, k=k, F=256, F_shared=128)
    cfg = U.config_of(wl)
    rng = np.random.default_rng(11 + T)
    if kind == "normal":
        g32 = rng.standard_normal((T, E)).astype(np.float32)
    else:
        g32 = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
    C = T * k // E
    ws = m.workspace(cfg)
    logits = torch.from_numpy(g32).to(DEV)
    tok = torch.empty((E, C), dtype=torch.int32, device=DEV)
    tw = torch.empty((E, C), dtype=torch.float32, device=DEV)
    ptr = torch.empty(T + 1, dtype=torch.int32, device=DEV)
    rows = torch.empty(E * C, dtype=torch.int32, device=DEV)
    m.moe_expert_choice(cfg, logits, tok, tw, ptr, rows, ws)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    tokens, weights, _ = O.expert_choice_route(g32, k)
    csr = O.expert_choice_csr(tokens, T)
    assert (tok.cpu().numpy() == tokens).all()
    assert np.abs(tw.cpu().numpy() - weights).max() <= U.WEIGHT_ATOL
    assert (ptr.cpu().numpy() == csr["ptr"]).all()
    assert (rows.cpu().numpy() == csr["rows"]).all()


# ---------------------------------------------------------------------------------------------
# failure paths (no fault: bounded waits and argument checks)
# ---------------------------------------------------------------------------------------------
def test_bounded_wait_reports_timeout_and_context_survives():
    m = U.lib()
    wl = moe_inputs.workload("tiny")
    cfg = U.config_of(wl)
    ws = m.workspace(cfg)
    m.moe_selftest_timeout(ws, 2000)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == -6
    assert m.sync_status(ws) == 0          # cleared by the read
    _full_check(wl, _inputs(wl), {}, U.OUT_TOL_F32)


def test_bad_expert_index_is_reported_not_faulted():
    m = U.lib()
    wl = moe_inputs.workload("tiny")
    cfg = U.config_of(wl)
    ws = m.workspace(cfg)
    T, E, k = wl.T, wl.E, wl.k
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    idx[:, 1] = 1
    idx[5, 1] = E            # out of range
    idx[9, 1] = 0            # expert chosen twice
    i32 = dict(dtype=torch.int32, device=DEV)
    bufs = [torch.empty(E, **i32), torch.empty(E, **i32), torch.empty(E + 1, **i32),
            torch.empty((T, k), **i32), torch.empty((T, k), **i32), torch.empty(T * k, **i32)]
    nd = torch.empty(1, **i32)
    m.moe_dispatch(cfg, idx, None, *bufs, None, nd, ws)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == -1


# ---------------------------------------------------------------------------------------------
# full size: routing/dispatch on every token, output on sampled tokens
# ---------------------------------------------------------------------------------------------
FULL = {
    "mixtral": dict(name="mixtral"),
    "mixtral_collapsed": dict(name="mixtral_collapsed"),
    "mixtral_cf1.0": dict(name="mixtral", capacity_factor=1.0),
    "mixtral_collapsed_cf1.25": dict(name="mixtral_collapsed", capacity_factor=1.25),
    "dsmoe16b": dict(name="dsmoe16b"),
    "dsmoe16b_ec": dict(name="dsmoe16b_ec"),
    "v3": dict(name="v3"),
    # decode batches of the full-size layers (the K-split cost model picks the slice counts
    # these sizes reach, which small cases do not)
    "v3_b1": dict(name="v3", T=1),
    "v3_b8": dict(name="v3", T=8),
    "v3_b64": dict(name="v3", T=64),
    "v3_b256": dict(name="v3", T=256),
    "mixtral_b1": dict(name="mixtral", T=1),
    "mixtral_b8": dict(name="mixtral", T=8),
    "mixtral_b64": dict(name="mixtral", T=64),
    "mixtral_b256": dict(name="mixtral", T=256),
}


def _check_dispatch_of(gpu, wl, idx):
    """The forward's own dispatch (row_of, offsets, dropped count) against the oracle's
    dispatch of the very indices the GPU selected -- bit-exact whatever the near ties did."""
    m = U.lib()
    _, row_of_p, offsets_p, _, _ = m.moe_workspace_views(gpu["cfg"], gpu["ws"])
    D = O.dispatch(idx, wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E))
    assert (_read_i32(offsets_p, wl.E + 1) == D["offsets"]).all()
    assert (_read_i32(row_of_p, wl.T * wl.k).reshape(wl.T, wl.k) == D["row_of"]).all()
    assert gpu["n_dropped"] == D["n_dropped"]
    return D


def _full_expert_choice(wl, inp, gpu, report):
    """Expert choice at full size: the forward's logits, its [E, C] token lists, weights and
    per-token CSR against the oracle, then the output on tokens covering every expert."""
    m = U.lib()
    g, g32 = O.router_logits(inp["x"], inp["w_gate"])
    logits_p, _, _, _, _ = m.moe_workspace_views(gpu["cfg"], gpu["ws"])
    gl = torch.as_tensor(_DevF32(logits_p, wl.T * wl.E), device=DEV).cpu().numpy().reshape(wl.T, wl.E)
    assert np.abs(gl - g).max() <= 1e-5 * np.abs(g).max()
    tokens, weights, _ = O.expert_choice_route(g32, wl.k)
    E, C = tokens.shape
    csr = O.expert_choice_csr(tokens, wl.T)
    tok_p, w_p, ptr_p, rows_p = m.moe_workspace_views_ec(gpu["cfg"], gpu["ws"])
    gtok = _read_i32(tok_p, E * C).reshape(E, C)
    gw = torch.as_tensor(_DevF32(w_p, E * C), device=DEV).cpu().numpy().reshape(E, C)
    # near ties: an expert whose C-th and (C+1)-th logits (oracle's float32) differ by < 1e-6
    # relative is reported and left out of the list check
    col = -np.sort(-g32.astype(np.float64), axis=0)
    a, b = col[C - 1], col[C]
    near = (a - b) / np.maximum(np.abs(a), 1e-30) < U.TIE_REL
    report["near_tie_experts"] = int(near.sum())
    same = (gtok == tokens).all(axis=1)
    assert (same | near).all(), np.nonzero(~same & ~near)[0][:10]
    assert np.abs(gw[same] - weights[same]).max() <= U.WEIGHT_ATOL
    if same.all():
        assert (_read_i32(ptr_p, wl.T + 1) == csr["ptr"]).all()
        assert (_read_i32(rows_p, E * C) == csr["rows"]).all()
    st = O.aux_stats_from_counts(g32, csr["counts"], wl.E)
    U.compare_stats(gpu, st, report)
    # per-token selection as a padded (idx, w, row) table, on tokens covering every expert's
    # first and last chosen token plus random ones
    rng = np.random.default_rng(0)
    pick = set(rng.choice(wl.T, 16, replace=False).tolist())
    for e in range(E):
        pick |= {int(tokens[e, 0]), int(tokens[e, -1])}
    sample = np.array(sorted(pick))
    kmax = max(int(np.diff(csr["ptr"]).max()), 1)
    idx = np.zeros((wl.T, kmax), np.int64)
    w = np.zeros((wl.T, kmax))
    row_of = -np.ones((wl.T, kmax), np.int64)
    for t in sample:
        for n, r in enumerate(csr["rows"][csr["ptr"][t]:csr["ptr"][t + 1]]):
            e, i = divmod(int(r), C)
            idx[t, n], w[t, n], row_of[t, n] = e, weights[e, i], r
    return sample, idx, w, row_of


@pytest.mark.parametrize("case", list(FULL))
def test_full_size_parity(case):
    spec = dict(FULL[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    inp = moe_inputs.make_inputs(wl, device=DEV)
    report = {}
    gpu = U.run_forward(wl, inp)
    hx = {"x": inp["x"].cpu(), "w_gate": inp["w_gate"].cpu(), "bias": inp["bias"].cpu()}
    rng = np.random.default_rng(0)
    if wl.routing == "expert_choice":
        sample, idx, w, row_of = _full_expert_choice(wl, hx, gpu, report)
        ok_tokens = sample
    else:
        r = O.route(wl, hx["x"], hx["w_gate"], hx["bias"])
        ok = U.compare_routing(wl, gpu, r, moe_inputs.to_f64(inp["bias"]), report)
        # dispatch of the GPU's own indices, always (near ties or not)
        Dg = _check_dispatch_of(gpu, wl, gpu["idx"])
        # statistics: counts from the GPU's selection, probabilities from the oracle's logits
        U.compare_stats(gpu, O.aux_stats(r["g32"], gpu["idx"], wl.E, wl.score), report)
        disp = O.dispatch(r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, wl.T, wl.E))
        if ok.all():
            for key in ("offsets", "row_of", "perm"):
                assert (Dg[key] == disp[key]).all(), key
        idx, w, row_of = r["idx"], r["w"], disp["row_of"]
        sample = U.coverage_tokens(disp["offsets"], disp["perm"], wl.k, wl.T, rng,
                                   16 if wl.E > 8 else 32)
        ok_tokens = sample[ok[sample]]
        report["drop_rate"] = disp["n_dropped"] / (wl.T * wl.k)
        report["f0"] = float(O.aux_stats(r["g32"], r["idx"], wl.E)["f"][0])
    report["sampled_tokens"] = int(len(ok_tokens))
    ref = O.moe_forward_sampled(hx["x"], idx, w, row_of, U.expert_weight_fetcher(inp),
                                U.shared_fetcher(inp), ok_tokens)
    got = gpu["out"][torch.from_numpy(ok_tokens).to(DEV)].float().cpu().numpy()
    U.compare_out(got, ref, U.OUT_TOL_BF16, report)
    print(case, report)
    del inp, gpu
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------------
# both tensor-core GEMM kernels (single CTA, CTA pair) on the same dispatched rows
# ---------------------------------------------------------------------------------------------
PAIR_CASES = {
    # ~1024 rows per expert, ragged: odd and even numbers of 128-row blocks
    "rows1024": dict(name="mixtral", T=2048, d=256, E=4, k=2, F=384),
    # few rows per expert (pairs with an empty half), several N tiles in both GEMMs
    "rows_small": dict(name="mixtral", T=300, d=512, E=8, k=2, F=256),
    # ~256 rows per expert under the selection bias: last pair tiles of <= 128 rows (M = 128
    # pair MMAs) beside ones of 129..255 rows (M = 256, padded)
    "rows256": dict(name="v3", T=512, d=256, E=16, k=8, F=256, n_shared=0),
}


@pytest.mark.parametrize("kernel", ["single", "pair", "pair_m256_only"])
@pytest.mark.parametrize("case", sorted(PAIR_CASES))
def test_expert_gemm_kernels(case, kernel, monkeypatch):
    monkeypatch.setenv("MOE_B300_GEMM", "single" if kernel == "single" else "pair")
    monkeypatch.setenv("MOE_B300_PAIR_HALF", "0" if kernel == "pair_m256_only" else "1")
    m = U.lib()
    spec = dict(PAIR_CASES[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    h = U.host(inp)
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"], h["ws2"])
    D = ref["disp"]
    T, k, d = wl.T, wl.k, wl.d
    nk = int(D["offsets"][-1])
    x_perm = torch.zeros((T * k, d), dtype=torch.bfloat16, device=DEV)
    src = torch.from_numpy((D["perm"][:nk] // k).astype(np.int64))
    x_perm[:nk] = inp["x"].cpu()[src].to(DEV)
    offsets = torch.from_numpy(D["offsets"].astype(np.int32)).to(DEV)
    y = torch.full((T * k, d), float("nan"), dtype=torch.float32, device=DEV)
    ws = m.workspace(cfg)
    m.moe_expert_ffn(cfg, x_perm, offsets, inp["w13"], inp["w2"], y, ws)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    report = {}
    U.compare_out(y[:nk].cpu().numpy(), ref["y_rows"], U.OUT_TOL_BF16, report, "y")
    assert torch.isnan(y[nk:]).all()          # rows past the last expert are never written
    print(case, kernel, report)


def test_shared_expert_on_pair_kernel(monkeypatch):
    monkeypatch.setenv("MOE_B300_GEMM", "pair")
    m = U.lib()
    wl = moe_inputs.workload("dsmoe16b", T=777, d=256, E=8, k=2, F=128, F_shared=256)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    h = U.host(inp)
    ws = m.workspace(cfg)
    shared = torch.empty((wl.T, wl.d), dtype=torch.float32, device=DEV)
    m.moe_shared_ffn(cfg, inp["x"], inp["ws13"], inp["ws2"], shared, ws)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    U.compare_out(shared.cpu().numpy(), O.shared_out(h["x"], h["ws13"], h["ws2"]),
                  U.OUT_TOL_BF16, {}, "shared")


@pytest.mark.parametrize("T", [1, 100, 256, 257, 700])
def test_dispatch_oracle_indices_bitexact(T):
    # T <= 256 takes the single-CTA dispatch, larger T the three-kernel path; both must give
    # the oracle's counts, positions, rows, permutation and drops bit for bit
    m = U.lib()
    wl = moe_inputs.workload("mixtral_collapsed", T=T, d=256, F=128, capacity_factor=1.0)
    cfg = U.config_of(wl)
    inp = moe_inputs.make_router_inputs(wl, device=DEV)
    h = {k: moe_inputs.to_f64(v) for k, v in inp.items()}
    r = O.route(wl, h["x"], h["w_gate"], h["bias"])
    D = O.dispatch(r["idx"], wl.E, O.capacity(wl.capacity_factor, wl.k, T, wl.E))
    E, k, d = wl.E, wl.k, wl.d
    i32 = dict(dtype=torch.int32, device=DEV)
    outs = {n: torch.full(sh, -9, **i32) for n, sh in
            [("counts", (E,)), ("kept", (E,)), ("offsets", (E + 1,)), ("pos", (T, k)),
             ("row_of", (T, k)), ("perm", (T * k,))]}
    nd = torch.full((1,), -9, **i32)
    x_perm = torch.zeros((T * k, d), dtype=torch.bfloat16, device=DEV)
    ws = m.workspace(cfg)
    oidx = torch.from_numpy(r["idx"].astype(np.int32)).to(DEV)
    m.moe_dispatch(cfg, oidx, inp["x"], outs["counts"], outs["kept"], outs["offsets"],
                   outs["pos"], outs["row_of"], outs["perm"], x_perm, nd, ws)
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    for n, t in outs.items():
        assert (t.cpu().numpy() == D[n]).all(), n
    assert nd.item() == D["n_dropped"]
    nk = int(D["offsets"][-1])
    src = torch.from_numpy((D["perm"][:nk] // k).astype(np.int64))
    assert torch.equal(x_perm[:nk].cpu(), inp["x"].cpu()[src])


GRAPH_CASES = {
    "decode_b16": dict(name="v3", T=16, d=256, E=64, F=256, F_shared=256),
    # prefill with shared experts: their GEMMs fork onto the side stream and join back
    "prefill_shared_side": dict(name="v3", T=700, d=256, E=64, F=256, F_shared=256),
    "expert_choice_shared_side": dict(name="dsmoe16b_ec", T=512, d=256, E=16, k=4, F=128,
                                      F_shared=256),
}


@pytest.mark.parametrize("case", list(GRAPH_CASES))
def test_forward_replays_in_a_cuda_graph(case):
    # every launch of moe_forward is stream-ordered and allocation-free (a side stream forked
    # from the caller's and joined back is captured with it), so a captured forward replays
    # with identical results
    m = U.lib()
    spec = dict(GRAPH_CASES[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    ws = m.workspace(cfg)
    out = torch.empty((wl.T, wl.d), dtype=torch.float32, device=DEV)

    def fwd():
        m.moe_forward(cfg, inp["x"], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"],
                      inp["ws13"], inp["ws2"], out, ws=ws)
    fwd()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    assert torch.equal(out, eager)


def test_first_forward_captured_in_a_new_thread():
    """A host thread whose first prefill forward with shared experts is captured into a graph:
    the side stream is not created during the capture, so the shared experts run on the
    captured stream, and the replay equals the eager forward bit for bit."""
    import threading
    m = U.lib()
    wl = moe_inputs.workload("v3", T=700, d=256, E=64, F=256, F_shared=256)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    ws = m.workspace(cfg)
    out = torch.empty((wl.T, wl.d), dtype=torch.float32, device=DEV)

    def fwd():
        m.moe_forward(cfg, inp["x"], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"],
                      inp["ws13"], inp["ws2"], out, ws=ws)
    fwd()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    torch.cuda.synchronize()
    box = {}
    dev_index = torch.cuda.current_device()

    def worker():
        try:
            torch.cuda.set_device(dev_index)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fwd()
            g.replay()
            torch.cuda.synchronize()
        except Exception as exc:      # reported on the test's thread
            box["err"] = exc
    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "err" not in box, box.get("err")
    assert m.sync_status(ws) == 0
    assert torch.equal(out, eager)


@pytest.mark.parametrize("spec", [
    dict(name="v3", T=700, d=256, E=64, F=256, F_shared=256, capacity_factor=1.25),
    dict(name="dsmoe16b", T=1500, d=256, E=64, F=128, F_shared=256),
    dict(name="dsmoe16b_ec", T=512, d=256, E=16, k=4, F=128, F_shared=256),
    dict(name="v3", T=8192, d=512, E=256, F=128, F_shared=256),
])
def test_shared_side_stream_equals_serial(monkeypatch, spec):
    """Prefill shared experts on the side stream (forked before the router, joined before the
    routed GEMMs) run the same kernels on the same operands as the serial order: the layer's
    outputs and statistics are bit-identical."""
    wl = moe_inputs.workload(**spec)
    inp = _inputs(wl)
    monkeypatch.setenv("MOE_B300_SHARED", "serial")
    a = U.run_forward(wl, inp)
    monkeypatch.delenv("MOE_B300_SHARED")
    b = U.run_forward(wl, inp)
    assert torch.equal(a["out"], b["out"])
    assert (a["idx"] == b["idx"]).all() and (a["w"] == b["w"]).all()
    for key in ("f", "P"):
        assert (a[key] == b[key]).all(), key
    assert a["l_balance"] == b["l_balance"] and a["z_loss"] == b["z_loss"]


@pytest.mark.parametrize("case", ["v3_like", "softmax_cap", "decode_b8", "router_fused_v3_e256",
                                  "router_fused_e96_tail", "router_fused_two_tiles_per_cta"])
def test_forward_timed_and_fused_statistics(case, monkeypatch):
    # moe_forward_timed runs moe_forward's kernels (identical output) and brackets the expert
    # GEMMs with the caller's events; the statistics moe_forward fuses into its Top-k pass
    # equal moe_aux_stats on the same logits and selection bit for bit
    _router_env(case, monkeypatch)
    m = U.lib()
    spec = dict(SMALL[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    cfg = U.config_of(wl)
    inp = _inputs(wl)
    a = U.run_forward(wl, inp, cfg)
    ws = m.workspace(cfg)
    out = torch.empty_like(a["out"])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for e in ev:
        e.record()
    m.moe_forward_timed(cfg, inp["x"], inp["w_gate"], inp["bias"], inp["w13"], inp["w2"],
                        inp["ws13"], inp["ws2"], out, ws=ws, ev_begin=ev[0], ev_end=ev[1])
    torch.cuda.synchronize()
    assert m.sync_status(ws) == 0
    assert torch.equal(out, a["out"])
    assert ev[0].elapsed_time(ev[1]) > 0
    logits_p, _, _, _, _ = m.moe_workspace_views(a["cfg"], a["ws"])
    logits = torch.as_tensor(_DevF32(logits_p, wl.T * wl.E), device=DEV).reshape(wl.T, wl.E)
    idx = torch.from_numpy(a["idx"]).to(DEV)
    f = torch.empty(wl.E, dtype=torch.float32, device=DEV)
    P = torch.empty(wl.E, dtype=torch.float32, device=DEV)
    lb = torch.empty(1, dtype=torch.float32, device=DEV)
    z = torch.empty(1, dtype=torch.float32, device=DEV)
    m.moe_aux_stats(cfg, logits.contiguous(), idx, f, P, lb, z, ws)
    torch.cuda.synchronize()
    assert (f.cpu().numpy() == a["f"]).all() and (P.cpu().numpy() == a["P"]).all()
    assert lb.item() == a["l_balance"] and z.item() == a["z_loss"]


class _DevF32:
    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<f4", "data": (ptr, False),
                                         "version": 3, "strides": None}


@pytest.mark.parametrize("spec", [
    dict(name="mixtral", T=700, d=256, F=384, capacity_factor=1.25),
    dict(name="mixtral_collapsed", T=600, d=256, F=256, capacity_factor=1.0),
    dict(name="dsmoe16b", T=3000, d=256, E=64, F=256, F_shared=256),
    dict(name="v3", T=1500, d=512, E=64, F=256, F_shared=256),
])
def test_fused_gather_matches_materialised_rows(monkeypatch, spec):
    """The gate/up GEMM reading its rows straight from x (cp.async gather) computes on the very
    same bf16 operands as the TMA path over the materialised rows: outputs bit-identical; and
    the fused path's output against the oracle's layer under the layer bar."""
    wl = moe_inputs.workload(**spec)
    inp = _inputs(wl)
    monkeypatch.setenv("MOE_B300_PATH", "prefill")
    monkeypatch.setenv("MOE_B300_GEMM", "single")
    monkeypatch.setenv("MOE_B300_GATHER", "separate")
    a = U.run_forward(wl, inp)
    monkeypatch.setenv("MOE_B300_GATHER", "fused")
    b = U.run_forward(wl, inp)
    assert torch.equal(a["out"], b["out"])
    assert (a["idx"] == b["idx"]).all()
    h = U.host(inp)
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"], h["ws13"],
                        h["ws2"])
    report = {}
    ok = U.compare_routing(wl, b, ref, h["bias"], report)
    U.compare_out(b["out"].float().cpu().numpy()[ok], ref["out"][ok], U.OUT_TOL_BF16, report)


@pytest.mark.parametrize("spec", [
    dict(name="mixtral", T=700, d=256, F=384, capacity_factor=1.25),
    dict(name="mixtral", T=513, d=256, E=16, k=1, F=256, renormalize=False),
])
def test_fused_combine_is_deterministic_and_matches_the_combine_pass(monkeypatch, spec):
    """With k <= 2 and no shared experts the down GEMM adds w * y into the zeroed output itself:
    a token gets at most two addends, so the result is the same whatever order they land in.
    The separate combine pass reads y back rounded to bf16 (half an ulp: at most 2^-8 of |y|),
    so per element the two differ by at most 2^-8 * sum_j |w_j| |y_j|, plus a few float32
    roundings.  |y_j| is bounded by the oracle's expert row plus the parity tolerance on y
    (2e-2 of the rows' RMS)."""
    wl = moe_inputs.workload(**spec)
    inp = _inputs(wl)
    monkeypatch.setenv("MOE_B300_PATH", "prefill")
    monkeypatch.setenv("MOE_B300_GEMM", "single")
    monkeypatch.delenv("MOE_B300_COMBINE", raising=False)
    a = U.run_forward(wl, inp)
    b = U.run_forward(wl, inp)
    assert torch.equal(a["out"], b["out"])
    monkeypatch.setenv("MOE_B300_COMBINE", "separate")
    c = U.run_forward(wl, inp)
    fa, fc = a["out"].double().cpu().numpy(), c["out"].double().cpu().numpy()
    rms = np.sqrt(np.mean(fc ** 2))
    h = U.host(inp)
    ref = O.moe_forward(wl, h["x"], h["w_gate"], h["bias"], h["w13"], h["w2"])
    same = (a["idx"] == ref["idx"]).all(axis=1)
    assert same.mean() > 0.99
    row_of = ref["disp"]["row_of"]
    y_abs = np.abs(ref["y_rows"]) + U.OUT_TOL_BF16 * np.sqrt(np.mean(ref["y_rows"] ** 2))
    bound = np.zeros_like(fa)
    for j in range(wl.k):
        rows = row_of[:, j]
        live = rows >= 0
        bound[live] += np.abs(a["w"][live, j])[:, None] * y_abs[rows[live]]
    err = np.abs(fa - fc)[same]
    assert (err <= 2.0 ** -8 * bound[same] + 1e-5 * rms).all()


@pytest.mark.parametrize("case", ["router_fused_v3_e256", "router_fused_e96_tail",
                                  "router_fused_groups_of_64"])
def test_router_epilogue_matches_separate_passes(case, monkeypatch):
    """The router GEMM with the routing in its epilogue against the separate logits GEMM and
    Top-k pass on the same inputs: the same logits (1e-6 relative), the same selection (near
    ties excepted, as against the oracle) and weights within the weight bar; and the stage entry
    point moe_router_topk gives the fused forward's selection."""
    m = U.lib()
    spec = dict(SMALL[case])
    wl = moe_inputs.workload(spec.pop("name"), **spec)
    inp = _inputs(wl)
    cfg = U.config_of(wl)
    T, E, k = wl.T, wl.E, wl.k
    runs = {}
    for mode in ("fused", "separate"):
        monkeypatch.setenv("MOE_B300_ROUTER", mode)
        ws = m.workspace(cfg)
        logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
        idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        m.moe_router_topk(cfg, inp["x"], inp["w_gate"], inp["bias"], logits, idx, w, ws)
        torch.cuda.synchronize()
        assert m.sync_status(ws) == 0
        runs[mode] = (logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
    gf, i_f, w_f = runs["fused"]
    gs, i_s, w_s = runs["separate"]
    assert np.abs(gf - gs).max() <= 1e-6 * np.abs(gs).max()
    h = U.host(inp)
    r = O.route(wl, h["x"], h["w_gate"], h["bias"])
    near = U.deciding_gaps(wl, r, h["bias"]) < U.TIE_REL
    same = (i_f == i_s).all(axis=1)
    assert (same | near).all()
    assert np.abs(w_f[same] - w_s[same]).max() <= U.WEIGHT_ATOL
    monkeypatch.setenv("MOE_B300_ROUTER", "fused")
    fwd = U.run_forward(wl, inp, cfg)
    assert (fwd["idx"] == i_f).all() and (fwd["w"] == w_f.astype(np.float64)).all()


"""Host-side checks of the C ABI that need no GPU: the library loads, exports every entry point
include/moe_b300.h declares, validates configurations, and computes capacity and workspace
sizes.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

import moe_inputs
from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    import top_routing_expert_scoring_b300 as m
    return m


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "moe_b300.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    m = _lib()
    names = declared_entry_points()
    assert len(names) >= 15
    for n in names:
        assert hasattr(m.lib, n), n
        assert n in m.EXPORTED, n
    assert m.version().startswith("moe_b300")


def config_of(wl, T=None):
    m = _lib()
    return m.make_config(T or wl.T, wl.d, wl.E, wl.k, wl.F, wl.F_sh, wl.score, wl.routing,
                         wl.n_groups, wl.topk_groups, wl.renormalize, wl.route_scale,
                         wl.capacity_factor, wl.dtype)


@pytest.mark.parametrize("name", sorted(moe_inputs.WORKLOADS))
def test_workload_configs_are_valid(name):
    m = _lib()
    cfg = config_of(moe_inputs.workload(name))
    assert m.check_config(cfg) == 0
    assert m.workspace_size(cfg) > 0


@pytest.mark.parametrize("field,value,status", [
    ("T", 0, -2), ("E", 0, -2), ("E", 257, -2), ("k", 9, -2), ("k", 0, -2),
    ("d_model", 100, -2), ("d_ff", 1000, -2), ("score", 5, -1), ("dtype", 7, -1),
    ("n_groups", 3, -2), ("renormalize", 2, -1), ("routing", 9, -1), ("out_dtype", 4, -1),
])
def test_config_rejections(field, value, status):
    m = _lib()
    cfg = config_of(moe_inputs.workload("mixtral"))
    setattr(cfg, field, value)
    assert m.check_config(cfg) == status


def test_group_limit_needs_enough_experts():
    m = _lib()
    cfg = config_of(moe_inputs.workload("v3"))
    cfg.topk_groups = 1          # 32 experts in one group >= k = 8: fine
    assert m.check_config(cfg) == 0
    cfg.E, cfg.n_groups, cfg.topk_groups = 64, 32, 2   # 2 groups x 2 experts < 8
    assert m.check_config(cfg) == -2
    cfg = config_of(moe_inputs.workload("mixtral"))
    cfg.n_groups, cfg.topk_groups = 4, 2                 # group limit with softmax scoring
    assert m.check_config(cfg) == -3


@pytest.mark.parametrize("cf,k,T,E", [(1.25, 2, 2048, 16), (1.0, 2, 4096, 8), (1.25, 2, 4096, 8),
                                      (1.1, 2, 4096, 8), (1.5, 8, 8192, 256), (0.3, 6, 333, 64),
                                      (0.0, 2, 256, 8), (-1.0, 2, 256, 8), (1.25, 2, 100, 8)])
def test_capacity_matches_oracle(cf, k, T, E):
    m = _lib()
    cfg = m.make_config(T, 128, E, k, 128, capacity_factor=cf)
    want = O.capacity(cf, k, T, E)
    assert m.capacity(cfg) == (T * k if want is None else min(want, T * k))


def test_status_strings():
    m = _lib()
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert m.status_string(s) and "unknown" not in m.status_string(s)


def test_null_arguments_rejected_before_any_launch():
    m = _lib()
    cfg = config_of(moe_inputs.workload("tiny"))
    P = ctypes.c_void_p
    assert m.lib.moe_forward(ctypes.byref(cfg), *([None] * 17)) == -1
    # workspace checks: NULL and misaligned workspaces are refused
    fake = P(0x1000)
    assert m.lib.moe_router_topk(ctypes.byref(cfg), fake, fake, None, None, fake, fake, None,
                                 None) == -4
    assert m.lib.moe_router_topk(ctypes.byref(cfg), fake, fake, None, None, fake, fake,
                                 P(0x1001), None) == -4
    assert m.lib.moe_sync_status(None, None) == -4
    assert m.lib.moe_selftest_timeout(P(0x1000), 0, None) == -1
    assert m.lib.moe_check_config(None) == -1


def test_workspace_grows_with_tokens():
    m = _lib()
    wl = moe_inputs.workload("mixtral")
    assert m.workspace_size(config_of(wl, T=8192)) > m.workspace_size(config_of(wl, T=4096))


def test_router_backward_rejections_before_any_launch():
    m = _lib()
    P = ctypes.c_void_p
    fake, ws = P(0x1000), P(0x100000)
    f = ctypes.c_float
    cfg = config_of(moe_inputs.workload("mixtral"), T=64)
    bw = m.lib.moe_router_backward
    args = lambda **kw: [kw.get(n, fake) for n in ("x", "w", "g", "idx", "dw", "f")] + [
        f(kw.get("alpha", 0.01)), f(kw.get("beta", 0.001))] + [
        kw.get(n, fake) for n in ("dlog", "dW", "dx", "ws")] + [None]
    assert bw(ctypes.byref(cfg), *args(x=None, ws=ws)) == -1
    assert bw(ctypes.byref(cfg), *args(dW=None, ws=ws)) == -1
    assert bw(ctypes.byref(cfg), *args(f=None, ws=ws)) == -1           # alpha != 0 needs f
    assert bw(ctypes.byref(cfg), *args(idx=None, ws=ws)) == -1         # d_topk_w needs idx
    assert bw(ctypes.byref(cfg), *args(alpha=float("nan"), ws=ws)) == -1
    assert bw(ctypes.byref(cfg), *args(ws=None)) == -4
    assert bw(ctypes.byref(cfg), *args(ws=P(0x100001))) == -4
    ec = config_of(moe_inputs.workload("dsmoe16b_ec"), T=64)
    assert bw(ctypes.byref(ec), *args(ws=ws)) == -3
    ub = m.lib.moe_bias_update
    assert ub(ctypes.byref(cfg), None, fake, f(0.001), None) == -1
    assert ub(ctypes.byref(cfg), fake, fake, f(float("inf")), None) == -1
    big = config_of(moe_inputs.workload("mixtral"), T=1 << 20)
    big.k = 8
    assert ub(ctypes.byref(big), fake, fake, f(0.001), None) == -2


def test_router_backward_workspace_sizes():
    m = _lib()
    wl = moe_inputs.workload("v3")
    small = m.router_backward_workspace_size(config_of(wl, T=1024))
    large = m.router_backward_workspace_size(config_of(wl, T=8192))
    # at least the two bf16 copies of dL/dg ([T, E64] and [E64, T64])
    assert large >= 2 * 8192 * 256 * 2 and large > small
    tiny = moe_inputs.workload("tiny")
    assert m.router_backward_workspace_size(config_of(tiny)) >= tiny.T * tiny.E * 4


def test_fp8_rejections_before_any_launch():
    m = _lib()
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert m.lib.moe_quantize_fp8(4, 64, None, fake, fake, None) == -1
    assert m.lib.moe_quantize_fp8(4, 40, fake, fake, fake, None) == -2    # cols % 16
    assert m.lib.moe_quantize_fp8(0, 64, fake, fake, fake, None) == -2
    n = ctypes.c_size_t()
    tiny = config_of(moe_inputs.workload("tiny"))                         # float32 activations
    assert m.lib.moe_fp8_workspace_size(ctypes.byref(tiny), ctypes.byref(n)) == -3
    d384 = config_of(moe_inputs.workload("mixtral", d=384), T=8)          # d % 256 != 0
    assert m.lib.moe_fp8_workspace_size(ctypes.byref(d384), ctypes.byref(n)) == -2
    ec = config_of(moe_inputs.workload("dsmoe16b_ec"), T=64)
    assert m.lib.moe_fp8_workspace_size(ctypes.byref(ec), ctypes.byref(n)) == -3
    v3 = config_of(moe_inputs.workload("v3"), T=64)
    assert m.lib.moe_forward_fp8(ctypes.byref(v3), *([None] * 21)) == -1
    # the shared expert's codes are required when the layer has one
    args = [fake] * 21
    args[7] = None
    assert m.lib.moe_forward_fp8(ctypes.byref(v3), *args) == -1
    assert m.fp8_workspace_size(v3) > m.workspace_size(v3)


def test_group_limit_needs_two_experts_per_group():
    m = _lib()
    wl = moe_inputs.workload("v3", T=16, d=256, E=8, n_groups=8, topk_groups=5, k=2)
    assert m.check_config(config_of(wl)) == -2
    ok = moe_inputs.workload("v3", T=16, d=256, E=8, n_groups=4, topk_groups=2, k=2)
    assert m.check_config(config_of(ok)) == 0


def test_binding_rejects_host_tensors_before_any_call():
    # the binding hands the library device pointers only: a CPU tensor is refused in Python,
    # before the C call, so no host address ever reaches a kernel
    import torch
    m = _lib()
    wl = moe_inputs.workload("mixtral", T=8, d=256, F=256)
    cfg = config_of(wl)
    x = torch.zeros(8, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        m.moe_forward(cfg, x, x, None, x, x, None, None, x, ws=x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        m.quantize_fp8(x)

"""CPU oracle for the single-GPU MoE layer forward.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline and reference legs may import
this module.  The product path (the CUDA library and its Python binding) never imports, links
or runs it, and this module shares no code with that path.

The arithmetic lives in plain C++ (moe_oracle.cpp, built here into libmoe_oracle.so with the
host compiler: plain loops, double accumulation, std::thread over independent rows).  This
module only marshals arrays: it converts inputs to contiguous host arrays, calls the C entry
point of the same step and wraps the outputs.  Each function cites, through its C counterpart,
the passage of the pages it follows; the pages are

  [R]   "MoE 路由数学"  (jerryiiii.gitbook.io, llm-review, math_dictionary/moe-routing-math)
  [A]   "Mixture of Experts 架构：稀疏激活如何重塑大语言模型的效率与规模"  (x7peeps.com)
  [G]   "MoE混合专家模型深度解析：路由机制与负载均衡"  (guijiagi.com)
  [L17] "第 17 讲 · Systems for Mixture-of-Experts Models"  (semidirectx.com, cmu11-868 lecture17)
  [I]   "MoE 推理优化深入"  (jerryiiii.gitbook.io, notes/distributed/moe-inference-deep)

Inputs may be numpy arrays (float64 or float32) or CPU torch tensors (bfloat16 is passed as its
16 bits and widened exactly by the C++ side).  Parity unpinned: the sigmoid-scoring P_i and the
expert-choice weights (readings of silent pages, see moe_oracle.cpp).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

F64 = np.float64
F32 = np.float32
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    """Compiles moe_oracle.cpp into libmoe_oracle.so (host C++ compiler) when it is missing or
    older than its source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.{os.getpid()}.tmp"
    cxx = os.environ.get("CXX", "g++")
    r = subprocess.run([cxx, *CXXFLAGS, "-o", tmp, _SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


_L = ctypes.CDLL(build())
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_D = ctypes.c_double
_SIGS = {
    "orc_set_threads": ([_I32], None),
    "orc_threads": ([], _I32),
    "orc_router_logits": ([_I64, _I64, _I64, _P, _I32, _P, _I32, _P, _P], None),
    "orc_topk_desc": ([_I64, _I64, _I64, _P, _P], None),
    "orc_softmax": ([_I64, _I64, _P, _P], None),
    "orc_softmax_topk_route": ([_I64, _I64, _I64, _P, _I32, _D, _P, _P, _P], None),
    "orc_sigmoid": ([_I64, _P, _P], None),
    "orc_count_selections": ([_I64, _I64, _I64, _P, _P], None),
    "orc_expected_distinct_experts": ([_I64, _I64, _I64], _D),
    "orc_sigmoid_group_route": ([_I64, _I64, _I64, _P, _P, _I64, _I64, _D, _I32, _P, _P, _P],
                                _I32),
    "orc_groups_of": ([_I64, _I64, _P, _I64, _I64, _P], None),
    "orc_capacity": ([ctypes.c_float, _I64, _I64, _I64], _I64),
    "orc_dispatch": ([_I64, _I64, _I64, _P, _I64] + [_P] * 7, _I32),
    "orc_expert_choice_route": ([_I64, _I64, _I64, _P, _P, _P, _P], None),
    "orc_expert_choice_csr": ([_I64, _I64, _I64, _P, _P, _P, _P], None),
    "orc_silu": ([_I64, _P, _P], None),
    "orc_expert_hidden": ([_I64, _P, _I64, _I64, _P, _I32, _P, _I32, _P], None),
    "orc_swiglu": ([_I64, _P, _I64, _I64, _P, _I32, _P, _I32, _P, _I32, _P], None),
    "orc_combine": ([_I64, _I64, _I64, _P, _P, _P, _P, _P], None),
    "orc_balance_loss": ([_I64, _P, _P], _D),
    "orc_aux_stats_from_counts": ([_I64, _I64, _P, _P, _I32, _P, _P, _P], None),
    "orc_router_backward": ([_I64, _I64, _I64, _P, _P, _P, _P, _D, _D, _I32, _I32, _D, _P],
                            None),
    "orc_router_param_grads": ([_I64, _I64, _I64, _P, _I32, _P, _I32, _P, _P, _P], None),
    "orc_bias_update": ([_I64, _P, _P, _I64, _I64, ctypes.c_float, _P], None),
    "orc_e4m3_round": ([_I64, _P, _P], None),
    "orc_set_fp8_identity": ([_I32], None),
    "orc_quantize_rows_fp8": ([_I64, _I64, _P, _P, _P], None),
    "orc_dequantized_fp8": ([_I64, _I64, _P, _I32, _P], None),
    "orc_fp8_ffn": ([_I64, _I64, _I64, _P, _P, _P, _P], None),
    "orc_forward_tokens": ([_I64, _P, _I64, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P,
                            _I32, _P, _P, _P], None),
    "orc_forward_tokens_fp8": ([_I64, _P, _I64, _I64, _I64, _I64, _I64, _P, _I32, _P, _P, _P,
                                _P, _P, _I32, _P, _P, _I32, _P], None),
    "orc_route": ([_P, _P, _I32, _P, _I32, _P, _P, _P, _P, _P, _P], _I32),
    "orc_moe_forward": ([_P, _P, _I32, _P, _I32, _P, _P, _P, _I32, _P, _P] + [_P] * 18, _I32),
    "orc_moe_forward_expert_choice": ([_P, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P]
                                      + [_P] * 11, None),
}
for _n, (_a, _r) in _SIGS.items():
    _fn = getattr(_L, _n)
    _fn.argtypes = _a
    _fn.restype = _r

BF16, FP32, FP64 = 0, 1, 2


class _Cfg(ctypes.Structure):
    _fields_ = [("T", _I64), ("d", _I64), ("E", _I64), ("k", _I64), ("F", _I64), ("Fs", _I64),
                ("score", _I32), ("n_groups", _I32), ("topk_groups", _I32),
                ("renormalize", _I32), ("route_scale", _D), ("capacity_factor", ctypes.c_float)]


# ----------------------------------------------------------------------------------------------
# marshalling helpers (no arithmetic)
# ----------------------------------------------------------------------------------------------
def threads() -> int:
    """Host threads the oracle's loops use (MOE_ORACLE_THREADS, else all cores)."""
    return int(_L.orc_threads())


def set_threads(n: int) -> None:
    _L.orc_set_threads(int(n))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _out(shape, dtype=F64):
    return np.zeros(shape, dtype=dtype)


class _Src:
    """A host array the C side reads element by element: pointer, element code, the array kept
    alive.  torch bfloat16 tensors pass their 16 bits; float32 and float64 pass as they are;
    anything else is converted to float64."""

    def __init__(self, a):
        try:
            import torch
        except ImportError:           # pragma: no cover - torch is part of the image
            torch = None
        if torch is not None and isinstance(a, torch.Tensor):
            a = a.detach()
            if a.device.type != "cpu":
                a = a.to("cpu")
            a = a.contiguous()
            if a.dtype == torch.bfloat16:
                self.arr, self.code = a.view(torch.int16).numpy(), BF16
            elif a.dtype == torch.float32:
                self.arr, self.code = a.numpy(), FP32
            else:
                self.arr, self.code = a.to(torch.float64).numpy(), FP64
        else:
            a = np.asarray(a)
            if a.dtype == F32:
                self.arr, self.code = np.ascontiguousarray(a), FP32
            else:
                self.arr, self.code = np.ascontiguousarray(a, dtype=F64), FP64
        self.shape = tuple(self.arr.shape)
        self.ptr = ctypes.c_void_p(self.arr.ctypes.data)

    def slab(self, e):
        """Pointer to entry e of the leading axis (one expert of a stacked [E, ...] array)."""
        step = self.arr.strides[0]
        return ctypes.c_void_p(self.arr.ctypes.data + e * step)


def _expert_ptrs(src: _Src, E: int):
    arr = (ctypes.c_void_p * E)()
    for e in range(E):
        arr[e] = src.slab(e)
    return arr


class _Experts:
    """Routed expert weights, either stacked ([E, ...] arrays) or a list with one array per
    expert (None for an expert the caller knows is never selected; the C side never reads it).
    Holds the per-expert pointers, the element code and d_ff."""

    def __init__(self, w13, w2, E):
        if isinstance(w13, (list, tuple)):
            self.srcs = [(None, None) if a is None else (_Src(a), _Src(b))
                         for a, b in zip(w13, w2)]
            self.p13, self.p2 = (ctypes.c_void_p * E)(), (ctypes.c_void_p * E)()
            live = [(e, s) for e, s in enumerate(self.srcs) if s[0] is not None]
            for e, (a, b) in live:
                self.p13[e], self.p2[e] = a.ptr, b.ptr
            flat = [x for _, pair in live for x in pair]
            self.F = live[0][1][0].shape[0] // 2 if live else 0
        else:
            a, b = _Src(w13), _Src(w2)
            self.srcs = [(a, b)]
            self.p13, self.p2 = _expert_ptrs(a, E), _expert_ptrs(b, E)
            flat = [a, b]
            self.F = a.shape[1] // 2
        self.flat = flat


def _same_code(*srcs):
    codes = {s.code for s in srcs if s is not None}
    if len(codes) > 1:
        raise TypeError("the expert weights must all have one element type")
    return codes.pop() if codes else FP64


# ----------------------------------------------------------------------------------------------
# Router logits, scoring, Top-k ([R] §2.1; [A] moe_forward code block; [L17] §2.1, §5.3)
# ----------------------------------------------------------------------------------------------
def router_logits(x, w_gate):
    """g[t, e] = sum_c x[t, c] W_gate[e, c] in double, g32 = float32(g) (moe_oracle.cpp
    orc_router_logits).  Returns (g, g32)."""
    xs, ws = _Src(x), _Src(w_gate)
    T, d = xs.shape
    E = ws.shape[0]
    g, g32 = _out((T, E)), _out((T, E), F32)
    _L.orc_router_logits(T, d, E, xs.ptr, xs.code, ws.ptr, ws.code, _p(g), _p(g32))
    return g, g32


def topk_desc(key, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, descending; equal keys rank by lower index;
    -0.0 equals +0.0 (orc_topk_desc)."""
    key = np.asarray(key)
    n = key.shape[-1]
    flat = _c(key.reshape(-1, n), F64)
    out = _out((flat.shape[0], k), np.int32)
    _L.orc_topk_desc(flat.shape[0], n, k, _p(flat), _p(out))
    return out.reshape(key.shape[:-1] + (k,))


def softmax(g) -> np.ndarray:
    """p = softmax(g) over the last axis ([R] §2.1), in double (orc_softmax)."""
    g = np.asarray(g)
    n = g.shape[-1]
    flat = _c(g.reshape(-1, n), F64)
    p = _out(flat.shape)
    _L.orc_softmax(flat.shape[0], n, _p(flat), _p(p))
    return p.reshape(g.shape)


def sigmoid(g) -> np.ndarray:
    g = np.asarray(g)
    flat = _c(g.reshape(-1), F64)
    s = _out(flat.shape)
    _L.orc_sigmoid(flat.size, _p(flat), _p(s))
    return s.reshape(g.shape)


def softmax_topk_route(g32, k: int, renormalize: bool = True, route_scale: float = 1.0):
    """Softmax scoring, Top-k on the logits, renormalisation ([R] §2.1; orc_softmax_topk_route).
    Returns (idx [T,k] int32, w [T,k] f64, p [T,E] f64)."""
    g = _c(g32, F64)
    T, E = g.shape
    idx, w, p = _out((T, k), np.int32), _out((T, k)), _out((T, E))
    _L.orc_softmax_topk_route(T, E, k, _p(g), int(bool(renormalize)), float(route_scale),
                              _p(idx), _p(w), _p(p))
    return idx, w, p


def sigmoid_group_route(g32, bias, k: int, n_groups: int, topk_groups: int, route_scale: float,
                        renormalize: bool = True):
    """DeepSeek-V3 gate in the ten steps of [L17] §5.3 (orc_sigmoid_group_route).  Returns
    (idx [T,k] int32, w [T,k] f64, s [T,E] f64 = sigmoid(g32) unrounded)."""
    g = _c(g32, F64)
    T, E = g.shape
    b = _c(bias, F32)
    idx, w, s = _out((T, k), np.int32), _out((T, k)), _out((T, E))
    st = _L.orc_sigmoid_group_route(T, E, k, _p(g), _p(b), n_groups, topk_groups,
                                    float(route_scale), int(bool(renormalize)), _p(idx), _p(w),
                                    _p(s))
    if st != 0:
        raise ValueError("a group score is the sum of the group's two largest scores: "
                         "a group needs at least two experts")
    return idx, w, s


def groups_of(idx, E: int, n_groups: int) -> np.ndarray:
    """Number of distinct expert groups each token's selection touches ([L17] §4.3)."""
    idx = _c(idx, np.int32)
    out = _out(idx.shape[0], np.int64)
    _L.orc_groups_of(idx.shape[0], idx.shape[1], _p(idx), E, n_groups, _p(out))
    return out


# ----------------------------------------------------------------------------------------------
# Capacity and dispatch ([L17] §2.2, §2.4)
# ----------------------------------------------------------------------------------------------
def capacity(cf: float, k: int, T: int, E: int):
    """C = ceil(cf * k * T / E) ([L17] §2.4); None when cf <= 0 (orc_capacity)."""
    C = int(_L.orc_capacity(float(np.float32(cf)), k, T, E))
    return None if C < 0 else C


def dispatch(idx, E: int, C):
    """Token-order grouping by expert with the capacity limit (orc_dispatch).  Returns counts,
    kept, offsets, pos, row_of, perm, n_dropped and capacity."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts, kept = _out(E, np.int32), _out(E, np.int32)
    offsets = _out(E + 1, np.int32)
    pos, row_of = _out((T, k), np.int32), _out((T, k), np.int32)
    perm = _out(T * k, np.int32)
    nd = ctypes.c_int64()
    st = _L.orc_dispatch(T, k, E, _p(idx), -1 if C is None else int(C), _p(counts), _p(kept),
                         _p(offsets), _p(pos), _p(row_of), _p(perm), ctypes.byref(nd))
    assert st == 0, "a token selected an expert twice (or an index is out of range)"
    return {"counts": counts, "kept": kept, "offsets": offsets, "pos": pos, "row_of": row_of,
            "perm": perm, "n_dropped": int(nd.value), "capacity": T * k if C is None else C}


def expert_choice_route(g32, k: int):
    """Expert choice ([G] §2.2; orc_expert_choice_route): tokens [E, C] ascending, weights
    [E, C] = p[t, e], p [T, E]."""
    g = _c(g32, F64)
    T, E = g.shape
    C = (T * k) // E
    tokens, weights, p = _out((E, C), np.int32), _out((E, C)), _out((T, E))
    _L.orc_expert_choice_route(T, E, k, _p(g), _p(tokens), _p(weights), _p(p))
    return tokens, weights, p


def expert_choice_csr(tokens, T: int):
    """Per-token view of an expert-choice selection (orc_expert_choice_csr)."""
    tokens = _c(tokens, np.int32)
    E, C = tokens.shape
    ptr = _out(T + 1, np.int32)
    rows, experts = _out(E * C, np.int32), _out(E * C, np.int32)
    _L.orc_expert_choice_csr(E, C, T, _p(tokens), _p(ptr), _p(rows), _p(experts))
    return {"ptr": ptr, "rows": rows, "experts": experts, "counts": np.full(E, C, np.int64)}


# ----------------------------------------------------------------------------------------------
# Expert FFN, shared experts, combine ([L17] §5.2, [R] §2.1 and §2.2, [L17] §2.2 step 4)
# ----------------------------------------------------------------------------------------------
def silu(a) -> np.ndarray:
    a = np.asarray(a)
    flat = _c(a.reshape(-1), F64)
    out = _out(flat.shape)
    _L.orc_silu(flat.size, _p(flat), _p(out))
    return out.reshape(a.shape)


def swiglu_expert(x, w13, w2) -> np.ndarray:
    """Expert(x) = (SiLU(x W1^T) * (x W3^T)) W2^T, w13 = [W1; W3] [2F, d], w2 [d, F]
    (orc_swiglu)."""
    xs, a, b = _Src(x), _Src(w13), _Src(w2)
    n, d = xs.shape
    F = a.shape[0] // 2
    y = _out((n, d))
    _L.orc_swiglu(n, None, d, F, xs.ptr, xs.code, a.ptr, a.code, b.ptr, b.code, _p(y))
    return y


def expert_hidden(x, w13) -> np.ndarray:
    """h = SiLU(x W1^T) * (x W3^T) (orc_expert_hidden)."""
    xs, a = _Src(x), _Src(w13)
    n, d = xs.shape
    F = a.shape[0] // 2
    h = _out((n, F))
    _L.orc_expert_hidden(n, None, d, F, xs.ptr, xs.code, a.ptr, a.code, _p(h))
    return h


def shared_out(x, ws13, ws2):
    """Sum of the always-on experts for every token ([R] §2.2), given concatenated as one
    expert of width n_shared * F_shared."""
    if ws13 is None:
        return np.zeros(tuple(x.shape), F64)
    return swiglu_expert(x, ws13, ws2)


def combine(T: int, d: int, idx, w, row_of, y_rows, shared=None):
    """out[t] = shared[t] + sum_{j : row_of[t,j] >= 0} w[t,j] y_rows[row_of[t,j]]
    (orc_combine)."""
    k = np.asarray(idx).shape[1]
    w, row_of = _c(w, F64), _c(row_of, np.int32)
    y = _c(y_rows, F64)
    sh = None if shared is None else _c(shared, F64)
    out = _out((T, d))
    _L.orc_combine(T, d, k, _p(w), _p(row_of), _p(y), _p(sh), _p(out))
    return out


def expert_rows(x, idx, disp, w13, w2):
    """y_rows[row] = Expert_e(x[t]) for every kept pair (row = row_of[t, j], e = idx[t, j])."""
    xs, a, b = _Src(x), _Src(w13), _Src(w2)
    k = np.asarray(idx).shape[1]
    offsets = disp["offsets"]
    d = xs.shape[1]
    F = a.shape[1] // 2
    y = _out((int(offsets[-1]), d))
    for e in range(a.shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        toks = _c(disp["perm"][lo:hi] // k, np.int32)
        ye = _out((hi - lo, d))
        _L.orc_swiglu(hi - lo, _p(toks), d, F, xs.ptr, xs.code, a.slab(e), a.code, b.slab(e),
                      b.code, _p(ye))
        y[lo:hi] = ye
    return y


# ----------------------------------------------------------------------------------------------
# Load-balance statistics ([R] §3.2; [A] load_balancing_loss and router_z_loss code blocks;
# [G] §3.1, §3.2)
# ----------------------------------------------------------------------------------------------
def balance_loss(f, P) -> float:
    """L_balance = E sum_i f_i P_i ([R] §3.2 boxed equation; orc_balance_loss)."""
    f, P = _c(f, F64), _c(P, F64)
    return float(_L.orc_balance_loss(len(f), _p(f), _p(P)))


def aux_stats(g32, idx, E: int, score: str = "softmax"):
    """Statistics of a token-choice selection idx [T, k] (see aux_stats_from_counts)."""
    idx = _c(idx, np.int32)
    counts = _out(E)
    _L.orc_count_selections(idx.shape[0], idx.shape[1], E, _p(idx), _p(counts))
    return aux_stats_from_counts(g32, counts, E, score)


def aux_stats_from_counts(g32, counts, E: int, score: str = "softmax"):
    """f_i = counts_i / T, P_i = mean_t prob[t, i], L = E sum f_i P_i, z = mean_t lse_t^2
    (orc_aux_stats_from_counts)."""
    g = _c(g32, F64)
    T = g.shape[0]
    counts = _c(counts, F64)
    f, P, out4 = _out(E), _out(E), _out(4)
    _L.orc_aux_stats_from_counts(T, E, _p(g), _p(counts), 0 if score == "softmax" else 1, _p(f),
                                 _p(P), _p(out4))
    return {"f": f, "P": P, "l_balance": float(out4[0]), "l_balance_per_k": float(out4[1]),
            "z_loss": float(out4[2]), "counts": counts.astype(np.int64)}


# ----------------------------------------------------------------------------------------------
# Router-side backward and the bias update ([R] §3.4; [L17] §3.2, §3.4; [A] code blocks)
# ----------------------------------------------------------------------------------------------
def router_backward(g32, idx, d_w, f, alpha: float, beta: float, score: str = "softmax",
                    renormalize: bool = True, route_scale: float = 1.0):
    """dL/dg [T, E] of alpha L_balance + beta z + <d_w, w> with f and the selection fixed
    (orc_router_backward)."""
    g = _c(g32, F64)
    T, E = g.shape
    idx = _c(idx, np.int32)
    dw = None if d_w is None else _c(d_w, F64)
    ff = None if f is None else _c(f, F64)
    dg = _out((T, E))
    _L.orc_router_backward(T, E, idx.shape[1], _p(g), _p(idx), _p(dw), _p(ff), float(alpha),
                           float(beta), 0 if score == "softmax" else 1, int(bool(renormalize)),
                           float(route_scale), _p(dg))
    return dg


def router_param_grads(x, w_gate, dg):
    """With g = x W_gate^T: (dL/dW_gate = dg^T x [E, d], dL/dx = dg W_gate [T, d])."""
    xs, ws = _Src(x), _Src(w_gate)
    T, d = xs.shape
    E = ws.shape[0]
    dg = _c(dg, F64)
    dW, dx = _out((E, d)), _out((T, d))
    _L.orc_router_param_grads(T, d, E, xs.ptr, xs.code, ws.ptr, ws.code, _p(dg), _p(dW), _p(dx))
    return dW, dx


def bias_update(bias, counts, T: int, k: int, gamma: float):
    """One step of the loss-free balancing bias rule ([L17] §3.4; orc_bias_update)."""
    b = _c(bias, F32)
    counts = _c(counts, np.int64)
    out = _out(len(b), F32)
    _L.orc_bias_update(len(b), _p(b), _p(counts), T, k, float(np.float32(gamma)), _p(out))
    return out


# ----------------------------------------------------------------------------------------------
# FP8 (E4M3) expert weights and activations ([L17] §1.4; [I] §4.2)
# ----------------------------------------------------------------------------------------------
E4M3_MAX = 448.0


class fp8_identity_quantisation:
    """Context manager for tests: inside it the oracle's row quantiser is the identity (codes =
    float32 values, scale 1), so the FP8 layer must reduce to the bf16 layer."""

    def __enter__(self):
        _L.orc_set_fp8_identity(1)
        return self

    def __exit__(self, *exc):
        _L.orc_set_fp8_identity(0)
        return False


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value of float32 inputs, ties to even, saturating (orc_e4m3_round)."""
    v = np.asarray(v)
    flat = _c(v.reshape(-1), F32)
    out = _out(flat.shape)
    _L.orc_e4m3_round(flat.size, _p(flat), _p(out))
    return out.reshape(v.shape)


def quantize_rows_fp8(V):
    """Per-row E4M3 quantisation with float32 decisions (orc_quantize_rows_fp8).  Returns
    (codes as float64 values [rows, cols], scales float64 [rows])."""
    V = _c(V, F32)
    rows, cols = V.shape
    codes, scales = _out((rows, cols)), _out(rows)
    _L.orc_quantize_rows_fp8(rows, cols, _p(V), _p(codes), _p(scales))
    return codes, scales


def dequantized_fp8(W) -> np.ndarray:
    """codes * scale of the per-row quantisation of a weight tensor (last axis = row)."""
    src = _Src(W)
    cols = src.shape[-1]
    rows = int(np.prod(src.shape[:-1]))
    out = _out((rows, cols))
    _L.orc_dequantized_fp8(rows, cols, src.ptr, src.code, _p(out))
    return out.reshape(src.shape)


def fp8_expert_weights(w13, w2, ws13=None, ws2=None):
    """Dequantised per-row E4M3 expert weights (float64 arrays of the same shapes)."""
    out = {"w13": dequantized_fp8(w13), "w2": dequantized_fp8(w2), "ws13": None, "ws2": None}
    if ws13 is not None:
        out["ws13"] = dequantized_fp8(ws13)
        out["ws2"] = dequantized_fp8(ws2)
    return out


def fp8_ffn(xd, W13, W2):
    """One SwiGLU expert on dequantised E4M3 rows with dequantised weights (orc_fp8_ffn)."""
    xd, W13, W2 = _c(xd, F64), _c(W13, F64), _c(W2, F64)
    n, d = xd.shape
    F = W13.shape[0] // 2
    y = _out((n, d))
    _L.orc_fp8_ffn(n, d, F, _p(xd), _p(W13), _p(W2), _p(y))
    return y


def _tokens_fp8(x, idx, w, row_of, tokens, E, w13_ptrs, w2_ptrs, wcode, ws13, ws2, F, Fs,
                quantize):
    xs = _Src(x)
    d = xs.shape[1]
    idx, row_of = _c(idx, np.int32), _c(row_of, np.int32)
    w = _c(w, F64)
    tok = _c(tokens, np.int32)
    out = _out((len(tok), d))
    _L.orc_forward_tokens_fp8(len(tok), _p(tok), d, idx.shape[1], F, Fs, E, xs.ptr, xs.code,
                              _p(idx), _p(w), _p(row_of), w13_ptrs, w2_ptrs, wcode,
                              None if ws13 is None else ws13.ptr,
                              None if ws2 is None else ws2.ptr, int(quantize), _p(out))
    return out


def moe_forward_fp8(wl, x, w_gate, bias, wq, tokens=None):
    """The layer with FP8 expert weights (wq: dequantised, from fp8_expert_weights) and FP8
    activations (orc_forward_tokens_fp8).  Routing, weights and statistics are those of the
    bf16 layer.  tokens: evaluate only these tokens' outputs (routing still over all T).
    Returns (out rows, route dict)."""
    r = route(wl, x, w_gate, bias)
    T, E = r["g32"].shape
    disp = dispatch(r["idx"], E, capacity(wl.capacity_factor, wl.k, T, E))
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    a, b = _Src(wq["w13"]), _Src(wq["w2"])
    sa = None if wq["ws13"] is None else _Src(wq["ws13"])
    sb = None if wq["ws2"] is None else _Src(wq["ws2"])
    out = _tokens_fp8(x, r["idx"], r["w"], disp["row_of"], toks, E, _expert_ptrs(a, E),
                      _expert_ptrs(b, E), _same_code(a, b, sa, sb), sa, sb, a.shape[1] // 2,
                      0 if sa is None else sa.shape[0] // 2, quantize=False)
    return out, r


def moe_forward_fp8_sampled(x, idx, w, row_of, expert_weights, shared_weights=None, tokens=None):
    """moe_forward_fp8 for the sampled tokens from a given selection, the bf16 expert weights
    fetched one expert at a time (expert_weights(e) -> (w13 [2F,d], w2 [d,F]), shared_weights()
    -> (ws13, ws2) or None) and quantised by the C side."""
    tokens = np.asarray(tokens)
    idx_a, row_a = np.asarray(idx), np.asarray(row_of)
    need = sorted({int(e) for e in np.unique(idx_a[tokens][row_a[tokens] >= 0])})
    E = int(idx_a.max()) + 1
    held, F = {}, 0
    w13p, w2p = (ctypes.c_void_p * E)(), (ctypes.c_void_p * E)()
    for e in need:
        pa, pb = expert_weights(e)
        a, b = _Src(pa), _Src(pb)
        held[e] = (a, b)
        w13p[e], w2p[e] = a.ptr, b.ptr
        F = a.shape[0] // 2
    sw = shared_weights() if shared_weights is not None else None
    sa = sb = None
    if sw is not None:
        sa, sb = _Src(sw[0]), _Src(sw[1])
    codes = [s for pair in held.values() for s in pair] + [sa, sb]
    return _tokens_fp8(x, idx, w, row_of, tokens, E, w13p, w2p, _same_code(*codes), sa, sb,
                       F, 0 if sa is None else sa.shape[0] // 2, quantize=True)


def expected_distinct_experts(E: int, k: int, B: int) -> float:
    """E (1 - (1 - k/E)^B) ([L17] §1.4; orc_expected_distinct_experts)."""
    return float(_L.orc_expected_distinct_experts(E, k, B))


# ----------------------------------------------------------------------------------------------
# The whole layer
# ----------------------------------------------------------------------------------------------
def _cfg(wl, T, d, F, Fs):
    return _Cfg(T, d, wl.E, wl.k, F, Fs, 0 if wl.score == "softmax" else 1, wl.n_groups,
                wl.topk_groups, int(bool(wl.renormalize)), float(wl.route_scale),
                float(wl.capacity_factor))


def route(wl, x, w_gate, bias):
    """Routing for a workload (orc_route): returns dict with g, g32, idx, w, prob."""
    xs, gs = _Src(x), _Src(w_gate)
    T, d = xs.shape
    cfg = _cfg(wl, T, d, 0, 0)
    E, k = wl.E, wl.k
    b = None if bias is None else _c(bias, F32)
    g, g32 = _out((T, E)), _out((T, E), F32)
    idx, w, prob = _out((T, k), np.int32), _out((T, k)), _out((T, E))
    st = _L.orc_route(ctypes.byref(cfg), xs.ptr, xs.code, gs.ptr, gs.code, _p(b), _p(g), _p(g32),
                      _p(idx), _p(w), _p(prob))
    if st != 0:
        raise ValueError("a group score is the sum of the group's two largest scores: "
                         "a group needs at least two experts")
    return {"g": g, "g32": g32, "idx": idx, "w": w, "prob": prob}


def moe_forward(wl, x, w_gate, bias, w13, w2, ws13=None, ws2=None):
    """Token-choice MoE layer forward ([R] §2.1, §2.2; [L17] §2.2 steps 1-4, §5.2) by
    orc_moe_forward: route, dispatch with capacity, SwiGLU experts, shared experts, weighted
    combine and the load-balance statistics.  w13/w2: stacked [E, ...] arrays, or lists with
    one array per expert (None for experts the tokens do not select)."""
    xs, gs = _Src(x), _Src(w_gate)
    E, k = wl.E, wl.k
    ex = _Experts(w13, w2, E)
    sa = None if ws13 is None else _Src(ws13)
    sb = None if ws2 is None else _Src(ws2)
    T, d = xs.shape
    F = ex.F
    Fs = 0 if sa is None else sa.shape[0] // 2
    cfg = _cfg(wl, T, d, F, Fs)
    bias_a = None if bias is None else _c(bias, F32)
    g, g32 = _out((T, E)), _out((T, E), F32)
    idx, w, prob = _out((T, k), np.int32), _out((T, k)), _out((T, E))
    counts, kept = _out(E, np.int32), _out(E, np.int32)
    offsets = _out(E + 1, np.int32)
    pos, row_of, perm = _out((T, k), np.int32), _out((T, k), np.int32), _out(T * k, np.int32)
    nd = ctypes.c_int64()
    y = _out((T * k, d))
    sh = _out((T, d)) if Fs else None
    out = _out((T, d))
    f, P, st4 = _out(E), _out(E), _out(4)
    st = _L.orc_moe_forward(ctypes.byref(cfg), xs.ptr, xs.code, gs.ptr, gs.code, _p(bias_a),
                            ex.p13, ex.p2, _same_code(*ex.flat, sa, sb),
                            None if sa is None else sa.ptr, None if sb is None else sb.ptr,
                            _p(g), _p(g32), _p(idx), _p(w), _p(prob), _p(counts), _p(kept),
                            _p(offsets), _p(pos), _p(row_of), _p(perm), ctypes.byref(nd), _p(y),
                            _p(sh), _p(out), _p(f), _p(P), _p(st4))
    if st != 0:
        raise ValueError(f"oracle forward refused the layer (code {st})")
    C = capacity(wl.capacity_factor, k, T, E)
    disp = {"counts": counts, "kept": kept, "offsets": offsets, "pos": pos, "row_of": row_of,
            "perm": perm, "n_dropped": int(nd.value), "capacity": T * k if C is None else C}
    stats = {"f": f, "P": P, "l_balance": float(st4[0]), "l_balance_per_k": float(st4[1]),
             "z_loss": float(st4[2]), "counts": counts.astype(np.int64)}
    return {"g": g, "g32": g32, "idx": idx, "w": w, "prob": prob, "disp": disp,
            "y_rows": y[:int(offsets[-1])], "shared": sh, "out": out, "stats": stats}


def moe_forward_tokens(wl, x, idx, w, row_of, w13, w2, ws13=None, ws2=None, tokens=None):
    """out[t] for a subset of tokens, each from that token's own selection
    (orc_forward_tokens)."""
    xs = _Src(x)
    a, b = _Src(w13), _Src(w2)
    sa = None if ws13 is None else _Src(ws13)
    sb = None if ws2 is None else _Src(ws2)
    E = a.shape[0]
    return _forward_tokens(xs, idx, w, row_of, _expert_ptrs(a, E), _expert_ptrs(b, E),
                           _same_code(a, b, sa, sb), sa, sb, a.shape[1] // 2,
                           np.arange(xs.shape[0]) if tokens is None else tokens)


def _forward_tokens(xs, idx, w, row_of, w13p, w2p, wcode, sa, sb, F, tokens):
    idx, row_of = _c(idx, np.int32), _c(row_of, np.int32)
    w = _c(w, F64)
    tok = _c(tokens, np.int32)
    d = xs.shape[1]
    out = _out((len(tok), d))
    Fs = 0 if sa is None else sa.shape[0] // 2
    _L.orc_forward_tokens(len(tok), _p(tok), d, idx.shape[1], F, Fs, xs.ptr, xs.code, _p(idx),
                          _p(w), _p(row_of), w13p, w2p, wcode, None if sa is None else sa.ptr,
                          None if sb is None else sb.ptr, _p(out))
    return out


def moe_forward_sampled(x, idx, w, row_of, expert_weights, shared_weights=None, tokens=None):
    """out[t] for the sampled tokens from a given selection (idx, w, row_of):
    out[t] = Shared(x_t) + sum_{j : row_of[t,j] >= 0} w[t,j] Expert_{idx[t,j]}(x_t).
    expert_weights(e) -> (w13 [2F,d], w2 [d,F]) is called once per expert the sampled tokens
    select (so that full-size layers need not be held in host memory at once);
    shared_weights() -> (ws13, ws2) or None.  Same C entry point as moe_forward_tokens."""
    tokens = np.asarray(tokens)
    idx_a, row_a = np.asarray(idx), np.asarray(row_of)
    need = sorted({int(e) for e in np.unique(idx_a[tokens][row_a[tokens] >= 0])})
    E = int(idx_a.max()) + 1
    w13p, w2p = (ctypes.c_void_p * E)(), (ctypes.c_void_p * E)()
    held, F = [], 0
    for e in need:
        pa, pb = expert_weights(e)
        a, b = _Src(pa), _Src(pb)
        held += [a, b]
        w13p[e], w2p[e] = a.ptr, b.ptr
        F = a.shape[0] // 2
    sw = shared_weights() if shared_weights is not None else None
    sa = sb = None
    if sw is not None:
        sa, sb = _Src(sw[0]), _Src(sw[1])
    return _forward_tokens(_Src(x), idx, w, row_of, w13p, w2p, _same_code(*held, sa, sb), sa, sb,
                           F, tokens)


def moe_forward_expert_choice(wl, x, w_gate, w13, w2, ws13=None, ws2=None):
    """Expert-choice layer ([G] §2.2; orc_moe_forward_expert_choice):
    out[t] = shared[t] + sum_{e chose t} p[t,e] Expert_e(x_t)."""
    xs, gs = _Src(x), _Src(w_gate)
    E, k = wl.E, wl.k
    ex = _Experts(w13, w2, E)
    sa = None if ws13 is None else _Src(ws13)
    sb = None if ws2 is None else _Src(ws2)
    T, d = xs.shape
    C = (T * k) // E
    F = ex.F
    Fs = 0 if sa is None else sa.shape[0] // 2
    cfg = _cfg(wl, T, d, F, Fs)
    g, g32 = _out((T, E)), _out((T, E), F32)
    tokens, weights, prob = _out((E, C), np.int32), _out((E, C)), _out((T, E))
    ptr, rows = _out(T + 1, np.int32), _out(E * C, np.int32)
    out, f, P, st4 = _out((T, d)), _out(E), _out(E), _out(4)
    _L.orc_moe_forward_expert_choice(ctypes.byref(cfg), xs.ptr, xs.code, gs.ptr, gs.code,
                                     ex.p13, ex.p2,
                                     _same_code(*ex.flat, sa, sb), None if sa is None else sa.ptr,
                                     None if sb is None else sb.ptr, _p(g), _p(g32), _p(tokens),
                                     _p(weights), _p(prob), _p(ptr), _p(rows), _p(out), _p(f),
                                     _p(P), _p(st4))
    csr = expert_choice_csr(tokens, T)
    stats = {"f": f, "P": P, "l_balance": float(st4[0]), "l_balance_per_k": float(st4[1]),
             "z_loss": float(st4[2]), "counts": np.full(E, C, np.int64)}
    return {"g": g, "g32": g32, "tokens": tokens, "weights": weights, "prob": prob, "out": out,
            "csr": csr, "stats": stats}

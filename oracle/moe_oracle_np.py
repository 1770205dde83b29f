"""Independent numpy restatement of the CPU oracle.  TEST INFRASTRUCTURE ONLY.

The oracle the tests, the smoke check and the benchmark use is the plain C++ one
(moe_oracle.cpp through moe_oracle.py).  This module computes the same equations separately,
with numpy's matrix products, and serves only as a cross-check of it (tests that the two agree
on random layers).  The product path never imports, links or runs it, and it shares no code
with that path or with the C++ oracle.

Plain, slow, obviously correct: numpy in float64, one step per equation of the pages, no
blocking or fusion.  Where a step decides an integer (which experts a token selects, which
groups survive, which tokens an expert takes), the decision is taken on float32 values, the
precision of the kernels, so that both sides decide in the same precision; the float32 values
here are the correctly rounded images of the exact float64 quantities.

Pages cited (titles as published):
  [R]  "MoE 路由数学"  (jerryiiii.gitbook.io, llm-review, math_dictionary/moe-routing-math)
  [A]  "Mixture of Experts 架构：稀疏激活如何重塑大语言模型的效率与规模"  (x7peeps.com)
  [G]  "MoE混合专家模型深度解析：路由机制与负载均衡"  (guijiagi.com)
  [L17] "第 17 讲 · Systems for Mixture-of-Experts Models"  (semidirectx.com, cmu11-868 lecture17)
  [I]  "MoE 推理优化深入"  (jerryiiii.gitbook.io, notes/distributed/moe-inference-deep)

Readings taken where the pages are silent or disagree (each is listed with its reason in the
design notes of the repository):
  * capacity C = ceil(cf * k * T / E) ([L17] §2.4); cf <= 0 means no limit;
  * overflow pairs are dropped in token order and contribute zero; the surviving weights are
    not renormalised ([L17] §2.4);
  * f_i counts selections before capacity drops, normalised by T so that sum_i f_i = k
    ([R] §3.2 table, [A] load_balancing_loss code block);
  * for sigmoid scoring, P_i is the mean of s_i / sum_j s_j over tokens (unbiased scores);
    parity unpinned beyond self-consistency (no page gives a formula);
  * ties: lower expert index, lower group index, lower token index;
  * the k outputs of a token are in rank order (descending key);
  * expert-choice: C = T*k/E tokens per expert, selected by the raw logit column
    ([G] §2.2 ExpertChoiceRouter code block), weight = softmax probability p[t, e]
    (parity of the weights unpinned: the page returns raw logits);
  * expert FFN = SwiGLU (SiLU(x W1) * (x W3)) W2 without biases ([L17] §5.2);
  * router backward: the loss is alpha * L_balance + beta * z + <d_w, w> with f and the
    selection held fixed ([R] §3.4: f is not differentiable); the z-loss gradient uses the
    softmax of the logits in both scoring modes;
  * bias update: the load of an expert is its number of selections before capacity drops, the
    target is the mean load T*k/E, and a load equal to it leaves the bias unchanged ([A]
    update_bias code block; [L17] §3.4).
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64
F32 = np.float32


# ----------------------------------------------------------------------------------------------
# Router logits  ([R] §2.1 g = x W_gate; [L17] §2.1 router is a linear layer h W_g)
# ----------------------------------------------------------------------------------------------
def router_logits(x: np.ndarray, w_gate: np.ndarray):
    """g[t, e] = sum_c x[t, c] * W_gate[e, c].

    x [T, d] and w_gate [E, d] hold bf16 or fp32 values widened exactly to float64.  Returns
    (g, g32): g in float64 (products of bf16/fp32 values are exact in float64 and the sum is
    within a few float64 ulps of exact) and g32 = float32(g), on which decisions are taken.
    """
    g = np.asarray(x, F64) @ np.asarray(w_gate, F64).T
    return g, g.astype(F32)


# ----------------------------------------------------------------------------------------------
# Top-k selection with the tie rule ([R] §2.1 S = TopK(p, k); [A] moe_forward code block)
# ----------------------------------------------------------------------------------------------
def topk_desc(key: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, in descending key order.

    Equal keys rank by lower index (a stable sort of the negated key); -0.0 equals +0.0.
    """
    order = np.argsort(-np.asarray(key), axis=-1, kind="stable")
    return order[..., :k].astype(np.int32)


def softmax(g: np.ndarray) -> np.ndarray:
    """p = softmax(g) over the last axis ([R] §2.1), in float64."""
    g = np.asarray(g, F64)
    m = g.max(axis=-1, keepdims=True)
    e = np.exp(g - m)
    return e / e.sum(axis=-1, keepdims=True)


def softmax_topk_route(g32: np.ndarray, k: int, renormalize: bool = True,
                       route_scale: float = 1.0):
    """Softmax scoring, Top-k, renormalisation ([R] §2.1 equations for p, S and p~).

    S is selected on the float32 logits (softmax is monotone, so the k largest logits are the
    k largest probabilities).  Weights: w = p_S / sum_S p (renormalize) or w = p_S (Switch,
    [L17] §2.1), times route_scale.  Returns (idx [T,k] int32, w [T,k] f64, p [T,E] f64).
    """
    p = softmax(g32)
    idx = topk_desc(g32, k)
    pS = np.take_along_axis(p, idx.astype(np.int64), axis=-1)
    w = pS / pS.sum(axis=-1, keepdims=True) if renormalize else pS
    return idx, w * route_scale, p


def sigmoid(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, F64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def sigmoid_group_route(g32: np.ndarray, bias: np.ndarray, k: int, n_groups: int,
                        topk_groups: int, route_scale: float, renormalize: bool = True):
    """DeepSeek-V3 gate, in the order of the walk-through in [L17] §5.3:

      1. s = sigmoid(g)                      (affinity per expert, 0..1)
      2. s' = s + b                          (bias used for selection only)
      3. view s' as [T, n_groups, E/n_groups]
      4. group score = sum of the two largest s' in the group
      5. keep the topk_groups best groups (ties: lower group index)
      6. set s' of experts in the other groups to -inf
      7. S = top-k of s' (ties: lower expert index), in descending order
      8. w = s[S] (the unbiased scores)
      9. w /= sum(w)
     10. w *= route_scale

    The loss-free routing of [A] (loss_free_balancing_routing code block) is the special case
    n_groups = topk_groups = 1.  Steps 1-7 run in float32 (s32 = float32(sigmoid(g32)),
    s'32 = float32(s32 + b), group score = float32(top1 + top2)); steps 8-10 in float64 from
    s32.  Returns (idx [T,k] int32, w [T,k] f64, s [T,E] f64 = sigmoid(g32) unrounded).
    """
    T, E = g32.shape
    s = sigmoid(g32)
    s32 = s.astype(F32)
    sb = (s32 + np.asarray(bias, F32)[None, :]).astype(F32)              # float32 add
    if n_groups > 1 and topk_groups < n_groups:
        per = E // n_groups
        if per < 2:
            raise ValueError("a group score is the sum of the group's two largest scores: "
                             "a group needs at least two experts")
        grouped = sb.reshape(T, n_groups, per)
        top2 = -np.sort(-grouped, axis=-1, kind="stable")[..., :2]         # two largest, desc
        gscore = (top2[..., 0] + top2[..., 1]).astype(F32)                 # float32 add
        keep = topk_desc(gscore, topk_groups)                              # [T, topk_groups]
        mask = np.ones((T, n_groups), dtype=bool)
        np.put_along_axis(mask, keep.astype(np.int64), False, axis=-1)     # True = dropped group
        sb = np.where(np.repeat(mask, per, axis=1), F32(-np.inf), sb).astype(F32)
    idx = topk_desc(sb, k)
    wS = np.take_along_axis(s32.astype(F64), idx.astype(np.int64), axis=-1)
    if renormalize:
        wS = wS / wS.sum(axis=-1, keepdims=True)
    return idx, wS * route_scale, s


def groups_of(idx: np.ndarray, E: int, n_groups: int) -> np.ndarray:
    """Number of distinct expert groups each token's selection touches ([L17] §4.3)."""
    per = E // n_groups
    grp = idx // per
    return np.array([len(set(r.tolist())) for r in grp], dtype=np.int64)


# ----------------------------------------------------------------------------------------------
# Capacity and dispatch ([L17] §2.2 group by expert, §2.4 capacity and dropping)
# ----------------------------------------------------------------------------------------------
def capacity(cf: float, k: int, T: int, E: int):
    """C = ceil(cf * k * T / E) ([L17] §2.4); None when cf <= 0 (no limit).

    cf is taken as a float32 (the C-ABI carries it as one) and widened; the product
    ((cf*k)*T)/E is formed in float64 and rounded up.
    """
    cf = float(np.float32(cf))
    if cf <= 0:
        return None
    return int(math.ceil(cf * k * T / E))


def dispatch(idx: np.ndarray, E: int, C):
    """Group the (token, choice) pairs by expert, in token order, with the capacity limit.

      counts[e]  = #{(t, j) : idx[t, j] = e}          (before drops)
      pos[t, j]  = #{t' < t : e in S_t'}, e = idx[t, j] (one token picks an expert at most once)
      dropped    iff pos >= C (the first C tokens by token index are kept)
      kept[e]    = min(counts[e], C)
      offsets    = exclusive scan of kept, length E+1
      row_of     = offsets[e] + pos, or -1 when dropped
      perm[row]  = t * k + j for the kept pairs; -1 for rows >= offsets[E]
    """
    T, k = idx.shape
    onehot = np.zeros((T, E), dtype=np.int64)
    np.put_along_axis(onehot, idx.astype(np.int64), 1, axis=1)
    assert (onehot.sum(axis=1) == k).all(), "a token selected an expert twice"
    counts = onehot.sum(axis=0)
    before = np.cumsum(onehot, axis=0) - onehot          # earlier tokens choosing each expert
    pos = np.take_along_axis(before, idx.astype(np.int64), axis=1)
    cap = T * k if C is None else C
    kept = np.minimum(counts, cap)
    offsets = np.concatenate([[0], np.cumsum(kept)])
    e = idx.astype(np.int64)
    keep = pos < cap
    row_of = np.where(keep, offsets[e] + pos, -1)
    perm = np.full(T * k, -1, dtype=np.int64)
    pair = np.arange(T * k).reshape(T, k)
    perm[row_of[keep]] = pair[keep]
    return {
        "counts": counts.astype(np.int32),
        "kept": kept.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "pos": pos.astype(np.int32),
        "row_of": row_of.astype(np.int32),
        "perm": perm.astype(np.int32),
        "n_dropped": int((counts - kept).sum()),
        "capacity": cap,
    }


def expert_choice_route(g32: np.ndarray, k: int):
    """Expert-choice routing ([G] §2.2): each expert takes the C = T*k/E tokens with the largest
    logit in its column of the transposed logits (ties: lower token index).

    Returns (tokens [E, C] int32 in ascending token order, weights [E, C] f64 = p[t, e],
    p [T, E]).  The weight p[t, e] is a reading: the page returns the raw top logits.
    """
    T, E = g32.shape
    C = (T * k) // E
    p = softmax(g32)
    sel = topk_desc(g32.T, C)                      # [E, C] by descending logit
    tokens = np.sort(sel, axis=1).astype(np.int32)
    weights = np.take_along_axis(p.T, tokens.astype(np.int64), axis=1)
    return tokens, weights, p


# ----------------------------------------------------------------------------------------------
# Expert FFN, shared experts and combine ([L17] §5.2 SwiGLU, [R] §2.2 shared experts,
# [R] §2.1 Output = sum_S p~_i Expert_i(x), [L17] §2.2 step 4 index_add)
# ----------------------------------------------------------------------------------------------
def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a))."""
    a = np.asarray(a, F64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def swiglu_expert(x: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """Expert(x) = (SiLU(x W1) * (x W3)) W2 with w13 = [W1; W3] of shape [2F, d], w2 [d, F]."""
    F = w13.shape[0] // 2
    x = np.asarray(x, F64)
    a = x @ np.asarray(w13[:F], F64).T
    b = x @ np.asarray(w13[F:], F64).T
    h = silu(a) * b
    return h @ np.asarray(w2, F64).T


def expert_hidden(x, w13):
    """h = SiLU(x W1) * (x W3), the intermediate activation of one SwiGLU expert."""
    F = w13.shape[0] // 2
    x = np.asarray(x, F64)
    return silu(x @ np.asarray(w13[:F], F64).T) * (x @ np.asarray(w13[F:], F64).T)


def shared_out(x, ws13, ws2):
    """Sum of the always-on experts for every token ([R] §2.2).  The n_shared experts are
    passed concatenated as one expert of width n_shared * F_shared, which computes exactly the
    sum of the separate experts."""
    if ws13 is None:
        return np.zeros((x.shape[0], x.shape[1]), F64)
    return swiglu_expert(x, ws13, ws2)


def combine(T: int, d: int, idx, w, row_of, y_rows, shared=None):
    """out[t] = shared[t] + sum_{j : row_of[t,j] >= 0} w[t,j] * y_rows[row_of[t,j]].

    Dropped pairs contribute zero and the other weights are left as they are.
    """
    out = np.zeros((T, d), F64) if shared is None else np.array(shared, F64, copy=True)
    k = idx.shape[1]
    for j in range(k):
        r = row_of[:, j]
        ok = r >= 0
        out[ok] += w[ok, j:j + 1] * y_rows[r[ok]]
    return out


def expert_rows(x, idx, disp, w13, w2):
    """y_rows[row] = Expert_e(x[t]) for every kept pair (row = row_of[t, j], e = idx[t, j])."""
    perm = disp["perm"]
    offsets = disp["offsets"]
    nrows = int(offsets[-1])
    k = idx.shape[1]
    y = np.zeros((nrows, x.shape[1]), F64)
    for e in range(w13.shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        toks = perm[lo:hi] // k
        y[lo:hi] = swiglu_expert(x[toks], w13[e], w2[e])
    return y


# ----------------------------------------------------------------------------------------------
# Load-balance statistics ([R] §3.2, [A] load_balancing_loss and router_z_loss code blocks,
# [G] §3.1 and §3.2)
# ----------------------------------------------------------------------------------------------
def balance_loss(f: np.ndarray, P: np.ndarray) -> float:
    """L_balance = E * sum_i f_i * P_i ([R] §3.2 boxed equation)."""
    f = np.asarray(f, F64)
    P = np.asarray(P, F64)
    return float(len(f) * np.dot(f, P))


def aux_stats(g32: np.ndarray, idx: np.ndarray, E: int, score: str = "softmax"):
    """Statistics of a token-choice selection idx [T, k] (see aux_stats_from_counts)."""
    T = g32.shape[0]
    onehot = np.zeros((T, E), F64)
    np.put_along_axis(onehot, idx.astype(np.int64), 1.0, axis=1)
    return aux_stats_from_counts(g32, onehot.sum(axis=0), E, score)


def aux_stats_from_counts(g32: np.ndarray, counts: np.ndarray, E: int, score: str = "softmax"):
    """f_i = (1/T) #{t : i in S_t}, P_i = (1/T) sum_t prob[t, i], L = E sum f_i P_i,
    z = (1/T) sum_t (logsumexp_i g[t, i])^2.

    prob is the softmax of g (softmax scoring) or, for sigmoid scoring, s_i / sum_j s_j with
    s = sigmoid(g) (unbiased scores; a reading, see the module docstring).
    """
    T = g32.shape[0]
    counts = np.asarray(counts, F64)
    f = counts / T
    if score == "softmax":
        prob = softmax(g32)
    else:
        s = sigmoid(g32)
        prob = s / s.sum(axis=1, keepdims=True)
    P = prob.sum(axis=0) / T
    g = np.asarray(g32, F64)
    m = g.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(g - m).sum(axis=1, keepdims=True)))[:, 0]
    z = float(np.mean(lse ** 2))
    L = balance_loss(f, P)
    k = counts.sum() / T
    return {"f": f, "P": P, "l_balance": L, "l_balance_per_k": L / k if k else 0.0, "z_loss": z,
            "counts": counts.astype(np.int64)}


# ----------------------------------------------------------------------------------------------
# Router-side backward and the selection-bias update ([R] §3.4; [L17] §3.2 and §3.4;
# [A] load_balancing_loss, router_z_loss, loss_free_balancing_routing and update_bias code blocks)
# ----------------------------------------------------------------------------------------------
def router_backward(g32: np.ndarray, idx: np.ndarray, d_w, f, alpha: float, beta: float,
                    score: str = "softmax", renormalize: bool = True, route_scale: float = 1.0):
    """Gradient dL/dg [T, E] (float64) of the router-side loss

        L = alpha * E * sum_i f_i P_i  +  beta * z  +  sum_{t,j} d_w[t, j] * w[t, j]

    with respect to the logits g, the selection idx [T, k] and the frequencies f [E] held fixed:
    f_i is a count and Top-k a selection, so the balance term reaches g only through P_i
    ([R] §3.4; [L17] §3.2), and the sigmoid route's bias only enters the selection ([L17] §3.4).

      P_i = (1/T) sum_t prob[t, i], prob = softmax(g) or s / sum(s) with s = sigmoid(g)
      z   = (1/T) sum_t lse_t^2, lse_t = logsumexp(g_t)      (both scoring modes)
      w   = route_scale * v_S / sum_S v  (renormalize) or route_scale * v_S, v = p or s
      d_w = upstream gradient of the routing weights (None: that term is absent)

    Chain rule, step by step: the balance term gives dL/dprob[t, i] = alpha * E * f_i / T; the
    weights give dL/dv on the selected entries; softmax maps a gradient G on p to
    p * (G - <G, p>), the normalisation q = s / sum(s) maps c to (c - <c, q>) / sum(s), the
    sigmoid multiplies by s (1 - s); the z-loss adds beta * (2/T) * lse_t * p.
    """
    g = np.asarray(g32, F64)
    T, E = g.shape
    idx64 = np.asarray(idx).astype(np.int64)
    p = softmax(g)
    m = g.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(g - m).sum(axis=1))
    v = p if score == "softmax" else sigmoid(g)

    dv = np.zeros((T, E), F64)                          # dL/dv from the routing weights
    if d_w is not None:
        dW = np.asarray(d_w, F64)
        vS = np.take_along_axis(v, idx64, axis=1)
        if renormalize:
            sumS = vS.sum(axis=1, keepdims=True)
            wS = route_scale * vS / sumS
            dvS = (route_scale * dW - (dW * wS).sum(axis=1, keepdims=True)) / sumS
        else:
            dvS = route_scale * dW
        np.put_along_axis(dv, idx64, dvS, axis=1)        # a token's k experts are distinct

    c = np.zeros(E, F64) if f is None else alpha * E * np.asarray(f, F64) / T
    if score == "softmax":
        G = dv + c[None, :]                              # dL/dp
        dg = p * (G - (G * p).sum(axis=1, keepdims=True))
    else:
        s = v
        ssum = s.sum(axis=1, keepdims=True)
        q = s / ssum
        ds = dv + (c[None, :] - (c[None, :] * q).sum(axis=1, keepdims=True)) / ssum
        dg = ds * s * (1.0 - s)
    dg = dg + beta * (2.0 / T) * lse[:, None] * p
    return dg


def router_param_grads(x: np.ndarray, w_gate: np.ndarray, dg: np.ndarray):
    """With g = x W_gate^T: dL/dW_gate = dg^T x  [E, d] and dL/dx = dg W_gate  [T, d]
    (float64)."""
    dg = np.asarray(dg, F64)
    return dg.T @ np.asarray(x, F64), dg @ np.asarray(w_gate, F64)


def bias_update(bias: np.ndarray, counts: np.ndarray, T: int, k: int, gamma: float):
    """One step of the loss-free balancing bias rule ([L17] §3.4; [A] update_bias code block):
    an expert whose load is above the mean load T*k/E gets b -= gamma, one below gets
    b += gamma, one exactly at the mean keeps b.  The load is the number of (token, choice)
    selections before any capacity drop, compared exactly as integers (counts * E vs T * k).
    The bias is float32 state and the update is one float32 addition.
    """
    b = np.asarray(bias, F32).copy()
    counts = np.asarray(counts, np.int64)
    E = len(b)
    over = counts * E > T * k
    under = counts * E < T * k
    g32 = F32(gamma)
    b[over] = (b[over] - g32).astype(F32)
    b[under] = (b[under] + g32).astype(F32)
    return b


# ----------------------------------------------------------------------------------------------
# FP8 (E4M3) expert weights and activations for decode ("Systems for Mixture-of-Experts Models"
# §1.4: DeepSeek-V3 keeps its weights in FP8; "MoE 推理优化深入" §4.2: per-expert quantisation)
# ----------------------------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities;
    largest finite 448 = 1.75 * 2^8, smallest subnormal 2^-9), ties to the even mantissa, values
    beyond 448 saturated to +-448.  Input float32 values, output float64 values on the grid."""
    v = np.asarray(v, F32).astype(F64)
    a = np.abs(v)
    # spacing of the grid around a: 2^(e-3) in the binade [2^e, 2^(e+1)), e >= -6; 2^-9 below
    _, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    r = np.rint(a / quantum) * quantum                   # np.rint: ties to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def quantize_rows_fp8(V: np.ndarray):
    """Per-row E4M3 quantisation with the decisions in float32: amax = max |v| over the row,
    inv = float32(448 / amax), code = e4m3(float32(v * inv)), scale = float32(amax / 448);
    a row of zeros gets codes 0 and scale 0.  Returns (codes as float64 values [rows, cols],
    scales float64 [rows]); the row is represented by codes * scale."""
    V32 = np.asarray(V, F32)
    amax = np.abs(V32).max(axis=1).astype(F32)
    nz = amax > 0
    inv = np.zeros_like(amax)
    inv[nz] = (F32(E4M3_MAX) / amax[nz]).astype(F32)
    scaled = (V32 * inv[:, None]).astype(F32)
    codes = e4m3_round(scaled)
    scale = np.zeros_like(amax)
    scale[nz] = (amax[nz] / F32(E4M3_MAX)).astype(F32)
    return codes, scale.astype(F64)


def fp8_expert_weights(w13, w2, ws13=None, ws2=None):
    """Quantised expert weights: every weight row (output channel) of W13 [E, 2F, d],
    W2 [E, d, F] and of the shared expert gets its own scale.  Returns a dict of dequantised
    float64 arrays with the same shapes (codes * scale)."""
    out = {"w13": dequantized_fp8(w13), "w2": dequantized_fp8(w2), "ws13": None, "ws2": None}
    if ws13 is not None:
        out["ws13"] = dequantized_fp8(ws13)
        out["ws2"] = dequantized_fp8(ws2)
    return out


def moe_forward_fp8(wl, x, w_gate, bias, wq, tokens=None):
    """The layer with FP8 expert weights (dequantised, from fp8_expert_weights) and FP8
    activations: every row that enters an expert GEMM (the token's x for the gate/up
    projection, its h for the down projection) is quantised per row as in quantize_rows_fp8,
    the products are exact in float64.  Routing, weights and statistics are those of the bf16
    layer (the router runs in bf16).  h is formed in float64 and rounded to float32 before its
    quantisation decision (the precision of the kernels).  tokens: evaluate only these tokens'
    outputs (routing still over all T).  Returns (out rows [len(tokens) or T, d], route dict)."""
    r = route(wl, x, w_gate, bias)
    T = r["g32"].shape[0]
    E = r["g32"].shape[1]
    C = capacity(wl.capacity_factor, wl.k, T, E)
    disp = dispatch(r["idx"], E, C)
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    xq, xs = quantize_rows_fp8(np.asarray(x, F64)[toks])
    xd = xq * xs[:, None]                                  # dequantised token rows
    d = xd.shape[1]
    out = np.zeros((len(toks), d), F64)
    if wq["ws13"] is not None:
        out += fp8_ffn(xd, wq["ws13"], wq["ws2"])
    for e in range(E):
        sel_t, sel_j = np.nonzero((r["idx"][toks] == e) & (disp["row_of"][toks] >= 0))
        if len(sel_t) == 0:
            continue
        y = fp8_ffn(xd[sel_t], wq["w13"][e], wq["w2"][e])
        out[sel_t] += r["w"][toks][sel_t, sel_j][:, None] * y
    return out, r


def fp8_ffn(xd, W13, W2):
    """One SwiGLU expert on dequantised E4M3 token rows xd with dequantised weights W13 [2F, d]
    and W2 [d, F]: h = SiLU(x W1) * (x W3) in float64, rounded to float32, quantised per row,
    then y = h_q W2."""
    F = W13.shape[0] // 2
    gu = xd @ W13.T
    h = silu(gu[:, :F]) * gu[:, F:]
    hq, hs = quantize_rows_fp8(h.astype(F32))
    return (hq * hs[:, None]) @ W2.T


def dequantized_fp8(W):
    """codes * scale of the per-row quantisation of a weight tensor (last axis = row)."""
    W = np.asarray(W, F64)
    c, s = quantize_rows_fp8(W.reshape(-1, W.shape[-1]))
    return (c * s[:, None]).reshape(W.shape)


def moe_forward_fp8_sampled(x, idx, w, row_of, expert_weights, shared_weights=None, tokens=None):
    """moe_forward_fp8 for the sampled tokens only, from a given selection, with the bf16 expert
    weights fetched one expert at a time (expert_weights(e) -> (w13 [2F,d], w2 [d,F]) float64,
    shared_weights() -> (ws13, ws2) or None) and quantised here, so that full-size layers can
    be checked without quantising every expert."""
    tokens = np.asarray(tokens)
    xq, xs = quantize_rows_fp8(np.asarray(x[tokens], F64))
    xd = xq * xs[:, None]
    out = np.zeros_like(xd)
    if shared_weights is not None:
        sw = shared_weights()
        if sw is not None:
            out += fp8_ffn(xd, dequantized_fp8(sw[0]), dequantized_fp8(sw[1]))
    sel = idx[tokens]
    keep = row_of[tokens] >= 0
    for e in np.unique(sel[keep]):
        w13, w2 = expert_weights(int(e))
        rows, slots = np.nonzero((sel == e) & keep)
        y = fp8_ffn(xd[rows], dequantized_fp8(w13), dequantized_fp8(w2))
        out[rows] += w[tokens][rows, slots][:, None] * y
    return out


def expected_distinct_experts(E: int, k: int, B: int) -> float:
    """E * (1 - (1 - k/E)^B): experts touched by a batch of B tokens under uniform, independent
    routing ([L17] §1.4)."""
    return E * (1.0 - (1.0 - k / E) ** B)


# ----------------------------------------------------------------------------------------------
# The whole layer
# ----------------------------------------------------------------------------------------------
def route(wl, x, w_gate, bias):
    """Routing for a workload: returns dict with g, g32, idx, w, prob."""
    g, g32 = router_logits(x, w_gate)
    if wl.score == "softmax":
        idx, w, p = softmax_topk_route(g32, wl.k, wl.renormalize, wl.route_scale)
    else:
        idx, w, p = sigmoid_group_route(g32, bias, wl.k, wl.n_groups, wl.topk_groups,
                                        wl.route_scale, wl.renormalize)
    return {"g": g, "g32": g32, "idx": idx, "w": w, "prob": p}


def moe_forward(wl, x, w_gate, bias, w13, w2, ws13=None, ws2=None):
    """Token-choice MoE layer forward ([R] §2.1 and §2.2, [L17] §2.2 steps 1-4 and §5.2):
    route, dispatch with capacity, SwiGLU experts, shared experts, weighted combine, and the
    load-balance statistics."""
    T, d = x.shape
    r = route(wl, x, w_gate, bias)
    C = capacity(wl.capacity_factor, wl.k, T, wl.E)
    disp = dispatch(r["idx"], wl.E, C)
    y = expert_rows(x, r["idx"], disp, w13, w2)
    sh = shared_out(x, ws13, ws2) if ws13 is not None else None
    out = combine(T, d, r["idx"], r["w"], disp["row_of"], y, sh)
    stats = aux_stats(r["g32"], r["idx"], wl.E, wl.score)
    return {**r, "disp": disp, "y_rows": y, "shared": sh, "out": out, "stats": stats}


def moe_forward_tokens(wl, x, idx, w, row_of, w13, w2, ws13=None, ws2=None, tokens=None):
    """out[t] for a subset of tokens, computed one token at a time from that token's own
    selection; used to check full-size runs on sampled rows."""
    tokens = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    res = np.zeros((len(tokens), x.shape[1]), F64)
    for n, t in enumerate(tokens):
        xt = np.asarray(x[t:t + 1], F64)
        acc = shared_out(xt, ws13, ws2)[0] if ws13 is not None else np.zeros(x.shape[1], F64)
        for j in range(idx.shape[1]):
            if row_of[t, j] >= 0:
                e = int(idx[t, j])
                acc = acc + w[t, j] * swiglu_expert(xt, w13[e], w2[e])[0]
        res[n] = acc
    return res


def moe_forward_expert_choice(wl, x, w_gate, w13, w2, ws13=None, ws2=None):
    """Expert-choice variant ([G] §2.2): out[t] = shared[t] + sum_{e chose t} p[t,e] Expert_e(x_t)."""
    T, d = x.shape
    g, g32 = router_logits(x, w_gate)
    tokens, weights, p = expert_choice_route(g32, wl.k)
    out = shared_out(x, ws13, ws2) if ws13 is not None else np.zeros((T, d), F64)
    for e in range(wl.E):
        ye = swiglu_expert(x[tokens[e]], w13[e], w2[e])
        out[tokens[e]] += weights[e][:, None] * ye
    csr = expert_choice_csr(tokens, T)
    stats = aux_stats_from_counts(g32, csr["counts"], wl.E, "softmax")
    return {"g": g, "g32": g32, "tokens": tokens, "weights": weights, "prob": p, "out": out,
            "csr": csr, "stats": stats}


def expert_choice_csr(tokens: np.ndarray, T: int):
    """Per-token view of an expert-choice selection: for token t, the rows e*C + i of the
    experts e that chose it (tokens[e, i] = t), in ascending expert order.

    Returns ptr [T+1], rows [E*C], experts [E*C] and counts [E] (each expert holds C tokens)."""
    E, C = tokens.shape
    lists = [[] for _ in range(T)]
    for e in range(E):
        for i in range(C):
            lists[int(tokens[e, i])].append(e * C + i)
    ptr = np.zeros(T + 1, np.int64)
    ptr[1:] = np.cumsum([len(l) for l in lists])
    rows = np.array([r for l in lists for r in l], dtype=np.int64)
    return {"ptr": ptr.astype(np.int32), "rows": rows.astype(np.int32),
            "experts": (rows // max(C, 1)).astype(np.int32),
            "counts": np.full(E, C, dtype=np.int64)}


def moe_forward_sampled(x, idx, w, row_of, expert_weights, shared_weights=None, tokens=None):
    """out[t] for the sampled tokens only, from a given selection (idx, w, row_of):
    out[t] = Shared(x_t) + sum_{j : row_of[t,j] >= 0} w[t,j] Expert_{idx[t,j]}(x_t).

    expert_weights(e) -> (w13 [2F,d], w2 [d,F]) as float64 arrays, fetched once per expert, so
    that full-size layers can be checked without holding every expert in float64 at once;
    shared_weights() -> (ws13, ws2) or None.  Same arithmetic as moe_forward_tokens.
    """
    tokens = np.asarray(tokens)
    xs = np.asarray(x[tokens], F64)
    out = np.zeros_like(xs)
    if shared_weights is not None:
        sw = shared_weights()
        if sw is not None:
            out += swiglu_expert(xs, sw[0], sw[1])
    sel = idx[tokens]
    keep = row_of[tokens] >= 0
    for e in np.unique(sel[keep]):
        w13, w2 = expert_weights(int(e))
        rows, slots = np.nonzero((sel == e) & keep)
        out[rows] += w[tokens][rows, slots][:, None] * swiglu_expert(xs[rows], w13, w2)
    return out

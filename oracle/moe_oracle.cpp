// CPU oracle of the single-GPU MoE layer forward.  TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline and reference legs may load
// this library (through oracle/moe_oracle.py).  The product path (the CUDA library and its
// Python binding) never loads, links or runs it, and it shares no code with that path: no
// header, helper, table or constant generator in common.
//
// Plain, slow, obviously correct C++: plain loops in the order of the equations, double
// accumulation, std::thread over independent rows (tokens, experts or output columns) and
// nothing else -- no BLAS, no blocking of a sum, no fusion.  Every dot product runs in index
// order; where several are computed side by side for speed, each keeps its own accumulator
// and its own order.  Where a step decides an integer (which experts a token selects, which
// groups survive, which tokens an expert takes, which E4M3 code a value gets) the decision is
// taken on float32 values, the precision of the kernels, so that both sides decide in the same
// precision.  Inputs are read exactly: bf16 (stored as its 16 bits), float32 and float64
// values all widen exactly to double.
//
// Pages cited (titles as published):
//   [R]   "MoE 路由数学"  (jerryiiii.gitbook.io, llm-review, math_dictionary/moe-routing-math)
//   [A]   "Mixture of Experts 架构：稀疏激活如何重塑大语言模型的效率与规模"  (x7peeps.com)
//   [G]   "MoE混合专家模型深度解析：路由机制与负载均衡"  (guijiagi.com)
//   [L17] "第 17 讲 · Systems for Mixture-of-Experts Models"  (semidirectx.com, cmu11-868 lecture17)
//   [I]   "MoE 推理优化深入"  (jerryiiii.gitbook.io, notes/distributed/moe-inference-deep)
//
// Readings where the pages are silent or disagree:
//   * capacity C = ceil(cf * k * T / E) ([L17] §2.4); cf <= 0 means no limit;
//   * overflow pairs are dropped in token order and contribute zero; the surviving weights are
//     not renormalised ([L17] §2.4);
//   * f_i counts selections before capacity drops, normalised by T so that sum_i f_i = k
//     ([R] §3.2 table, [A] load_balancing_loss code block);
//   * for sigmoid scoring, P_i is the mean of s_i / sum_j s_j over tokens (unbiased scores):
//     parity unpinned beyond self-consistency, no page gives a formula;
//   * ties: lower expert index, lower group index, lower token index; -0.0 equals +0.0;
//   * the k outputs of a token are in rank order (descending key);
//   * expert choice: C = T*k/E tokens per expert, selected by the raw logit column ([G] §2.2
//     ExpertChoiceRouter code block), weight = softmax probability p[t, e] (parity of the
//     weights unpinned: the page returns raw logits);
//   * expert FFN = SwiGLU (SiLU(x W1) * (x W3)) W2 without biases ([L17] §5.2);
//   * router backward: the loss is alpha * L_balance + beta * z + <d_w, w> with f and the
//     selection held fixed ([R] §3.4); the z-loss gradient uses softmax(g) in both scoring modes;
//   * bias update: load = selections before capacity drops, target = mean load T*k/E, a load
//     equal to it leaves the bias unchanged ([A] update_bias code block; [L17] §3.4);
//   * FP8: E4M3 with one float32 scale per row (amax / 448), round to nearest even, saturating
//     ([L17] §1.4 FP8 weights; [I] §4.2 quantised experts; neither fixes a scheme).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------------------------
// Element access: a pointer plus its type; every value widens exactly to double.
// ---------------------------------------------------------------------------------------------
enum Dtype : int32_t { BF16 = 0, F32 = 1, F64 = 2 };

inline float bf16_bits_to_float(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

inline double elem(const void* p, int32_t dt, int64_t i) {
  switch (dt) {
    case BF16: return bf16_bits_to_float(static_cast<const uint16_t*>(p)[i]);
    case F32: return static_cast<const float*>(p)[i];
    default: return static_cast<const double*>(p)[i];
  }
}

// Row r (length n) of a row-major matrix, widened to double.
void row_to_double(const void* p, int32_t dt, int64_t r, int64_t n, double* out) {
  for (int64_t c = 0; c < n; ++c) out[c] = elem(p, dt, r * n + c);
}

// ---------------------------------------------------------------------------------------------
// Threads: fn(i) for i in [0, n), contiguous chunks, one std::thread per chunk.
// ---------------------------------------------------------------------------------------------
int g_threads = 0;

int thread_count() {
  if (g_threads > 0) return g_threads;
  const char* env = std::getenv("MOE_ORACLE_THREADS");
  int n = env ? std::atoi(env) : 0;
  if (n < 1) n = static_cast<int>(std::thread::hardware_concurrency());
  return n < 1 ? 1 : n;
}

void parallel_for(int64_t n, const std::function<void(int64_t)>& fn) {
  const int64_t nt = std::min<int64_t>(thread_count(), n);
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t chunk = (n + nt - 1) / nt;
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t lo = t * chunk, hi = std::min(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([lo, hi, &fn] {
      for (int64_t i = lo; i < hi; ++i) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

// y[j] = sum_c a[c] * W[row0 + j][c] for j in [0, m): each sum in index order c = 0..K-1, with
// its own accumulator (four rows are walked side by side).
void rows_dot(const double* a, const void* W, int32_t wdt, int64_t row0, int64_t m, int64_t K,
              double* y) {
  int64_t j = 0;
  for (; j + 4 <= m; j += 4) {
    double s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    const int64_t b0 = (row0 + j) * K, b1 = b0 + K, b2 = b1 + K, b3 = b2 + K;
    for (int64_t c = 0; c < K; ++c) {
      const double ac = a[c];
      s0 += ac * elem(W, wdt, b0 + c);
      s1 += ac * elem(W, wdt, b1 + c);
      s2 += ac * elem(W, wdt, b2 + c);
      s3 += ac * elem(W, wdt, b3 + c);
    }
    y[j] = s0;
    y[j + 1] = s1;
    y[j + 2] = s2;
    y[j + 3] = s3;
  }
  for (; j < m; ++j) {
    double s = 0;
    const int64_t b = (row0 + j) * K;
    for (int64_t c = 0; c < K; ++c) s += a[c] * elem(W, wdt, b + c);
    y[j] = s;
  }
}

// ---------------------------------------------------------------------------------------------
// Small pieces of the routing math
// ---------------------------------------------------------------------------------------------
// Indices of the k largest keys, in descending key order; equal keys rank by lower index
// (a stable sort of the keys, largest first).  -0.0 and +0.0 compare equal.
template <typename K>
void topk_row(const K* key, int64_t n, int64_t k, int32_t* out, int64_t stride = 1) {
  std::vector<int32_t> order(n);
  for (int64_t i = 0; i < n; ++i) order[i] = static_cast<int32_t>(i);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return key[a * stride] > key[b * stride];
  });
  for (int64_t j = 0; j < k; ++j) out[j] = order[j];
}

// p = softmax(g) over one row ([R] §2.1), in double.
void softmax_row(const double* g, int64_t n, double* p) {
  double m = -INFINITY;
  for (int64_t i = 0; i < n; ++i) m = std::max(m, g[i]);
  double s = 0;
  for (int64_t i = 0; i < n; ++i) {
    p[i] = std::exp(g[i] - m);
    s += p[i];
  }
  for (int64_t i = 0; i < n; ++i) p[i] /= s;
}

// logsumexp of one row of logits, in double.
double lse_row(const double* g, int64_t n) {
  double m = -INFINITY;
  for (int64_t i = 0; i < n; ++i) m = std::max(m, g[i]);
  double s = 0;
  for (int64_t i = 0; i < n; ++i) s += std::exp(g[i] - m);
  return m + std::log(s);
}

double sigmoid(double g) { return 1.0 / (1.0 + std::exp(-g)); }

// SiLU(a) = a * sigmoid(a) = a / (1 + e^-a)
double silu(double a) { return a / (1.0 + std::exp(-a)); }

}  // namespace

extern "C" {

void orc_set_threads(int32_t n) { g_threads = n; }
int32_t orc_threads() { return thread_count(); }

// ---------------------------------------------------------------------------------------------
// Router logits ([R] §2.1 g = x W_gate; [L17] §2.1 the router is a linear layer)
//   g[t, e] = sum_c x[t, c] * W_gate[e, c]  in double, index order; g32 = float32(g).
// Products of bf16 or float32 values are exact in double, so g is within a few double ulps of
// the exact value and g32 is its correctly rounded image (barring a double-rounding tie).
// ---------------------------------------------------------------------------------------------
void orc_router_logits(int64_t T, int64_t d, int64_t E, const void* x, int32_t xdt,
                       const void* w_gate, int32_t wdt, double* g, float* g32) {
  parallel_for(T, [&](int64_t t) {
    std::vector<double> xr(d), row(E);
    row_to_double(x, xdt, t, d, xr.data());
    rows_dot(xr.data(), w_gate, wdt, 0, E, d, row.data());
    for (int64_t e = 0; e < E; ++e) {
      if (g) g[t * E + e] = row[e];
      g32[t * E + e] = static_cast<float>(row[e]);
    }
  });
}

// Top-k of each row of keys [rows, n] (see topk_row); float32 keys arrive widened exactly.
void orc_topk_desc(int64_t rows, int64_t n, int64_t k, const double* key, int32_t* idx) {
  parallel_for(rows, [&](int64_t r) { topk_row(key + r * n, n, k, idx + r * k); });
}

void orc_softmax(int64_t rows, int64_t n, const double* g, double* p) {
  parallel_for(rows, [&](int64_t r) { softmax_row(g + r * n, n, p + r * n); });
}

// Softmax scoring, Top-k, renormalisation ([R] §2.1 equations for p, S and p~; [A] moe_forward
// code block).  S is selected on the float32 logits: softmax is monotone, so the k largest
// logits are the k largest probabilities.  w = p_S / sum_S p (renormalize) or p_S (Switch,
// [L17] §2.1), times route_scale.  g holds the float32 logits widened (the selection keys);
// p [T, E] may be NULL.
void orc_softmax_topk_route(int64_t T, int64_t E, int64_t k, const double* g,
                            int32_t renormalize, double route_scale, int32_t* idx, double* w,
                            double* p_out) {
  parallel_for(T, [&](int64_t t) {
    std::vector<double> p(E);
    softmax_row(g + t * E, E, p.data());
    int32_t* it = idx + t * k;
    topk_row(g + t * E, E, k, it);
    double sum = 0;
    for (int64_t j = 0; j < k; ++j) sum += p[it[j]];
    for (int64_t j = 0; j < k; ++j)
      w[t * k + j] = (renormalize ? p[it[j]] / sum : p[it[j]]) * route_scale;
    if (p_out) std::copy(p.begin(), p.end(), p_out + t * E);
  });
}

// DeepSeek-V3 gate, in the order of the walk-through in [L17] §5.3:
//   1. s = sigmoid(g)                  (affinity per expert, 0..1)
//   2. s' = s + b                      (bias used for selection only)
//   3. view s' as [n_groups, E / n_groups]
//   4. group score = sum of the two largest s' in the group
//   5. keep the topk_groups best groups (ties: lower group index)
//   6. set s' of experts in the other groups to -inf
//   7. S = top-k of s' (ties: lower expert index), in descending order
//   8. w = s[S] (the unbiased scores)
//   9. w /= sum(w)                     (renormalize)
//  10. w *= route_scale
// The loss-free routing of [A] (loss_free_balancing_routing code block) is the case
// n_groups = topk_groups = 1.  Steps 1-7 decide in float32: s32 = float32(sigmoid(g32)),
// s'32 = float32(s32 + b), group score = float32(top1 + top2); steps 8-10 run in double from
// s32.  g holds the logits in double (float32 logits widened); s_out [T, E] = sigmoid(g)
// unrounded (may be NULL).  Returns 0, or -1 when a group has
// fewer than two experts (its score, the sum of its two largest, is undefined).
int32_t orc_sigmoid_group_route(int64_t T, int64_t E, int64_t k, const double* g,
                                const float* bias, int64_t n_groups, int64_t topk_groups,
                                double route_scale, int32_t renormalize, int32_t* idx, double* w,
                                double* s_out) {
  const bool limit = n_groups > 1 && topk_groups < n_groups;
  const int64_t per = E / n_groups;
  if (limit && per < 2) return -1;
  parallel_for(T, [&](int64_t t) {
    std::vector<float> s32(E), sb(E);
    for (int64_t e = 0; e < E; ++e) {
      const double s = sigmoid(g[t * E + e]);
      if (s_out) s_out[t * E + e] = s;
      s32[e] = static_cast<float>(s);
      sb[e] = s32[e] + bias[e];                         // float32 addition
    }
    if (limit) {
      std::vector<float> gscore(n_groups);
      for (int64_t q = 0; q < n_groups; ++q) {
        float a = -INFINITY, b = -INFINITY;             // largest, second largest
        for (int64_t i = 0; i < per; ++i) {
          const float v = sb[q * per + i];
          if (v > a) {
            b = a;
            a = v;
          } else if (v > b) {
            b = v;
          }
        }
        gscore[q] = a + b;                              // float32 addition
      }
      std::vector<int32_t> keep(topk_groups);
      topk_row(gscore.data(), n_groups, topk_groups, keep.data());
      std::vector<char> kept(n_groups, 0);
      for (int64_t j = 0; j < topk_groups; ++j) kept[keep[j]] = 1;
      for (int64_t e = 0; e < E; ++e)
        if (!kept[e / per]) sb[e] = -INFINITY;
    }
    int32_t* it = idx + t * k;
    topk_row(sb.data(), E, k, it);
    double sum = 0;
    for (int64_t j = 0; j < k; ++j) sum += static_cast<double>(s32[it[j]]);
    for (int64_t j = 0; j < k; ++j) {
      const double v = static_cast<double>(s32[it[j]]);
      w[t * k + j] = (renormalize ? v / sum : v) * route_scale;
    }
  });
  return 0;
}

// s = sigmoid(g) = 1 / (1 + e^-g), elementwise, in double.
void orc_sigmoid(int64_t n, const double* g, double* s) {
  for (int64_t i = 0; i < n; ++i) s[i] = sigmoid(g[i]);
}

// counts[e] = #{(t, j) : idx[t, j] = e} over a selection idx [T, k].
void orc_count_selections(int64_t T, int64_t k, int64_t E, const int32_t* idx, double* counts) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0.0;
  for (int64_t i = 0; i < T * k; ++i) counts[idx[i]] += 1.0;
}

// Experts touched by a batch of B tokens under uniform, independent routing:
// E (1 - (1 - k/E)^B) ([L17] §1.4).
double orc_expected_distinct_experts(int64_t E, int64_t k, int64_t B) {
  return static_cast<double>(E) *
         (1.0 - std::pow(1.0 - static_cast<double>(k) / static_cast<double>(E),
                         static_cast<double>(B)));
}

// Number of distinct expert groups each token's selection touches ([L17] §4.3).
void orc_groups_of(int64_t T, int64_t k, const int32_t* idx, int64_t E, int64_t n_groups,
                   int64_t* out) {
  const int64_t per = E / n_groups;
  for (int64_t t = 0; t < T; ++t) {
    std::vector<char> seen(n_groups, 0);
    int64_t n = 0;
    for (int64_t j = 0; j < k; ++j) {
      const int64_t q = idx[t * k + j] / per;
      if (!seen[q]) {
        seen[q] = 1;
        ++n;
      }
    }
    out[t] = n;
  }
}

// ---------------------------------------------------------------------------------------------
// Capacity and dispatch ([L17] §2.2 group by expert, §2.4 capacity and dropping)
// ---------------------------------------------------------------------------------------------
// C = ceil(cf * k * T / E) ([L17] §2.4), cf taken as float32 and widened, the product
// ((cf * k) * T) / E formed in double; -1 when cf <= 0 (no limit).
int64_t orc_capacity(float cf, int64_t k, int64_t T, int64_t E) {
  const double c = static_cast<double>(cf);
  if (!(c > 0)) return -1;
  return static_cast<int64_t>(std::ceil(c * static_cast<double>(k) * static_cast<double>(T) /
                                        static_cast<double>(E)));
}

// Group the (token, choice) pairs by expert, in token order, with the capacity limit:
//   counts[e]  = #{(t, j) : idx[t, j] = e}          (before drops)
//   pos[t, j]  = #{t' < t : e in S_t'}, e = idx[t, j] (a token picks an expert at most once)
//   dropped    iff pos >= C (the first C tokens by token index are kept)
//   kept[e]    = min(counts[e], C)
//   offsets    = exclusive scan of kept, length E+1
//   row_of     = offsets[e] + pos, or -1 when dropped
//   perm[row]  = t * k + j for the kept pairs; -1 for rows >= offsets[E]
// C < 0: no limit.  Returns 0, or -1 when a token selects an expert twice or an index is out
// of range.
int32_t orc_dispatch(int64_t T, int64_t k, int64_t E, const int32_t* idx, int64_t C,
                     int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* pos,
                     int32_t* row_of, int32_t* perm, int64_t* n_dropped) {
  const int64_t cap = C < 0 ? T * k : C;
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  // token order: a running count per expert gives each pair the number of earlier tokens
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t j = 0; j < k; ++j) {
      const int32_t e = idx[t * k + j];
      if (e < 0 || e >= E) return -1;
      for (int64_t q = 0; q < j; ++q)
        if (idx[t * k + q] == e) return -1;
      pos[t * k + j] = counts[e];
      counts[e] += 1;
    }
  }
  offsets[0] = 0;
  int64_t dropped = 0;
  for (int64_t e = 0; e < E; ++e) {
    kept[e] = static_cast<int32_t>(std::min<int64_t>(counts[e], cap));
    offsets[e + 1] = offsets[e] + kept[e];
    dropped += counts[e] - kept[e];
  }
  for (int64_t r = 0; r < T * k; ++r) perm[r] = -1;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t j = 0; j < k; ++j) {
      const int32_t e = idx[t * k + j];
      const int32_t p = pos[t * k + j];
      if (p < cap) {
        const int32_t row = offsets[e] + p;
        row_of[t * k + j] = row;
        perm[row] = static_cast<int32_t>(t * k + j);
      } else {
        row_of[t * k + j] = -1;
      }
    }
  }
  *n_dropped = dropped;
  return 0;
}

// Expert-choice routing ([G] §2.2): each expert takes the C = T*k/E tokens with the largest
// logit in its column of the transposed logits (ties: lower token index).  tokens [E, C] in
// ascending token order, weights [E, C] = p[t, e] (softmax of the token's logits; a reading,
// the page returns the raw top logits), p [T, E] (may be NULL).
void orc_expert_choice_route(int64_t T, int64_t E, int64_t k, const double* g, int32_t* tokens,
                             double* weights, double* p_out) {
  const int64_t C = (T * k) / E;
  std::vector<double> p(T * E);
  parallel_for(T, [&](int64_t t) { softmax_row(g + t * E, E, p.data() + t * E); });
  parallel_for(E, [&](int64_t e) {
    int32_t* te = tokens + e * C;
    topk_row(g + e, T, C, te, E);                       // column e, stride E
    std::sort(te, te + C);
    for (int64_t i = 0; i < C; ++i) weights[e * C + i] = p[te[i] * E + e];
  });
  if (p_out) std::copy(p.begin(), p.end(), p_out);
}

// Per-token view of an expert-choice selection: for token t, the rows e*C + i of the experts e
// that chose it (tokens[e, i] = t), in ascending expert order.  ptr [T+1], rows [E*C],
// experts [E*C] (the expert of each listed row; may be NULL).
void orc_expert_choice_csr(int64_t E, int64_t C, int64_t T, const int32_t* tokens, int32_t* ptr,
                           int32_t* rows, int32_t* experts) {
  std::vector<int64_t> n(T, 0);
  for (int64_t r = 0; r < E * C; ++r) n[tokens[r]] += 1;
  ptr[0] = 0;
  for (int64_t t = 0; t < T; ++t) ptr[t + 1] = static_cast<int32_t>(ptr[t] + n[t]);
  std::vector<int64_t> fill(T, 0);
  for (int64_t e = 0; e < E; ++e)
    for (int64_t i = 0; i < C; ++i) {
      const int32_t t = tokens[e * C + i];
      rows[ptr[t] + fill[t]] = static_cast<int32_t>(e * C + i);
      if (experts) experts[ptr[t] + fill[t]] = static_cast<int32_t>(e);
      fill[t] += 1;
    }
}

// ---------------------------------------------------------------------------------------------
// Expert FFN ([L17] §5.2 SwiGLU), shared experts ([R] §2.2) and combine ([R] §2.1 Output =
// sum_S p~_i Expert_i(x); [L17] §2.2 step 4)
// ---------------------------------------------------------------------------------------------
void orc_silu(int64_t n, const double* a, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = silu(a[i]);
}

// h[r] = SiLU(x[r] W1^T) * (x[r] W3^T) for the rows r listed in `rows` (NULL: r = 0..n-1) of x
// [*, d]; w13 = [W1; W3] of shape [2F, d] (gate rows first).  h [n, F] double.
void orc_expert_hidden(int64_t n, const int32_t* rows, int64_t d, int64_t F, const void* x,
                       int32_t xdt, const void* w13, int32_t wdt, double* h) {
  parallel_for(n, [&](int64_t i) {
    std::vector<double> xr(d), a(F), b(F);
    row_to_double(x, xdt, rows ? rows[i] : i, d, xr.data());
    rows_dot(xr.data(), w13, wdt, 0, F, d, a.data());     // x W1^T
    rows_dot(xr.data(), w13, wdt, F, F, d, b.data());     // x W3^T
    for (int64_t f = 0; f < F; ++f) h[i * F + f] = silu(a[f]) * b[f];
  });
}

// y[i] = Expert(x[rows[i]]) = (SiLU(x W1^T) * (x W3^T)) W2^T, w2 [d, F].  y [n, d] double.
void orc_swiglu(int64_t n, const int32_t* rows, int64_t d, int64_t F, const void* x, int32_t xdt,
                const void* w13, int32_t w13dt, const void* w2, int32_t w2dt, double* y) {
  parallel_for(n, [&](int64_t i) {
    std::vector<double> xr(d), a(F), b(F), h(F);
    row_to_double(x, xdt, rows ? rows[i] : i, d, xr.data());
    rows_dot(xr.data(), w13, w13dt, 0, F, d, a.data());
    rows_dot(xr.data(), w13, w13dt, F, F, d, b.data());
    for (int64_t f = 0; f < F; ++f) h[f] = silu(a[f]) * b[f];
    rows_dot(h.data(), w2, w2dt, 0, d, F, y + i * d);     // h W2^T
  });
}

// out[t] = shared[t] + sum_{j : row_of[t,j] >= 0} w[t,j] * y_rows[row_of[t,j]], in the order
// j = 0..k-1.  Dropped pairs contribute zero and the other weights are left as they are.
// shared [T, d] may be NULL (zeros).
void orc_combine(int64_t T, int64_t d, int64_t k, const double* w, const int32_t* row_of,
                 const double* y_rows, const double* shared, double* out) {
  parallel_for(T, [&](int64_t t) {
    double* o = out + t * d;
    for (int64_t c = 0; c < d; ++c) o[c] = shared ? shared[t * d + c] : 0.0;
    for (int64_t j = 0; j < k; ++j) {
      const int32_t r = row_of[t * k + j];
      if (r < 0) continue;
      const double wt = w[t * k + j];
      for (int64_t c = 0; c < d; ++c) o[c] += wt * y_rows[static_cast<int64_t>(r) * d + c];
    }
  });
}

// ---------------------------------------------------------------------------------------------
// Load-balance statistics ([R] §3.2; [A] load_balancing_loss and router_z_loss code blocks;
// [G] §3.1 and §3.2)
// ---------------------------------------------------------------------------------------------
// L_balance = E * sum_i f_i P_i ([R] §3.2 boxed equation).
double orc_balance_loss(int64_t E, const double* f, const double* P) {
  double s = 0;
  for (int64_t i = 0; i < E; ++i) s += f[i] * P[i];
  return static_cast<double>(E) * s;
}

// f_i = counts_i / T, P_i = (1/T) sum_t prob[t, i], L = E sum f_i P_i,
// z = (1/T) sum_t (logsumexp_i g[t, i])^2; prob = softmax(g) (score 0) or, for sigmoid scoring
// (score 1), s_i / sum_j s_j with s = sigmoid(g) (unbiased scores; a reading).
// out4 = {L_balance, L_balance / k (k = sum counts / T), z, k}.
void orc_aux_stats_from_counts(int64_t T, int64_t E, const double* g, const double* counts,
                               int32_t score, double* f, double* P, double* out4) {
  std::vector<double> prob(T * E), lse(T);
  parallel_for(T, [&](int64_t t) {
    double* pr = prob.data() + t * E;
    if (score == 0) {
      softmax_row(g + t * E, E, pr);
    } else {
      double s = 0;
      for (int64_t e = 0; e < E; ++e) {
        pr[e] = sigmoid(g[t * E + e]);
        s += pr[e];
      }
      for (int64_t e = 0; e < E; ++e) pr[e] /= s;
    }
    lse[t] = lse_row(g + t * E, E);
  });
  double nsel = 0;
  for (int64_t e = 0; e < E; ++e) {
    f[e] = counts[e] / static_cast<double>(T);
    nsel += counts[e];
    double s = 0;
    for (int64_t t = 0; t < T; ++t) s += prob[t * E + e];
    P[e] = s / static_cast<double>(T);
  }
  double z = 0;
  for (int64_t t = 0; t < T; ++t) z += lse[t] * lse[t];
  z /= static_cast<double>(T);
  const double L = orc_balance_loss(E, f, P);
  const double k = nsel / static_cast<double>(T);
  out4[0] = L;
  out4[1] = k != 0 ? L / k : 0.0;
  out4[2] = z;
  out4[3] = k;
}

// ---------------------------------------------------------------------------------------------
// Router-side backward and the selection-bias update ([R] §3.4; [L17] §3.2 and §3.4;
// [A] load_balancing_loss, router_z_loss, loss_free_balancing_routing and update_bias code
// blocks)
// ---------------------------------------------------------------------------------------------
// dL/dg [T, E] (double) of L = alpha * E * sum_i f_i P_i + beta * z + sum_{t,j} d_w[t,j] w[t,j]
// with the selection idx and the frequencies f held fixed (f_i is a count and Top-k a
// selection, so the balance term reaches g only through P_i; the sigmoid route's bias only
// enters the selection):
//   P_i = (1/T) sum_t prob[t, i], prob = softmax(g) or q = s / sum(s) with s = sigmoid(g)
//   z   = (1/T) sum_t lse_t^2, lse_t = logsumexp(g_t)          (both scoring modes)
//   w   = route_scale * v_S / sum_S v (renormalize) or route_scale * v_S, v = p or s
// Chain rule, step by step: the balance term gives dL/dprob[t, i] = alpha E f_i / T; the
// weights give dL/dv on the selected entries; softmax maps a gradient G on p to
// p (G - <G, p>); the normalisation q = s / sum(s) maps c to (c - <c, q>) / sum(s); the
// sigmoid multiplies by s (1 - s); the z-loss adds beta (2/T) lse_t p.
// d_w [T, k] and f [E] may be NULL (that term is absent).
void orc_router_backward(int64_t T, int64_t E, int64_t k, const double* g, const int32_t* idx,
                         const double* d_w, const double* f, double alpha, double beta,
                         int32_t score, int32_t renormalize, double route_scale, double* dg) {
  parallel_for(T, [&](int64_t t) {
    std::vector<double> p(E), v(E), dv(E, 0.0);
    softmax_row(g + t * E, E, p.data());
    const double lse = lse_row(g + t * E, E);
    for (int64_t e = 0; e < E; ++e) v[e] = score == 0 ? p[e] : sigmoid(g[t * E + e]);
    if (d_w) {
      const int32_t* it = idx + t * k;
      const double* dW = d_w + t * k;
      if (renormalize) {
        double sumS = 0;
        for (int64_t j = 0; j < k; ++j) sumS += v[it[j]];
        double dot = 0;                                  // sum_j dW_j w_j
        for (int64_t j = 0; j < k; ++j) dot += dW[j] * (route_scale * v[it[j]] / sumS);
        for (int64_t j = 0; j < k; ++j) dv[it[j]] = (route_scale * dW[j] - dot) / sumS;
      } else {
        for (int64_t j = 0; j < k; ++j) dv[it[j]] = route_scale * dW[j];
      }
    }
    std::vector<double> c(E, 0.0);
    if (f)
      for (int64_t e = 0; e < E; ++e) c[e] = alpha * static_cast<double>(E) * f[e] / T;
    double* out = dg + t * E;
    if (score == 0) {
      double gp = 0;                                     // <G, p>, G = dv + c
      for (int64_t e = 0; e < E; ++e) gp += (dv[e] + c[e]) * p[e];
      for (int64_t e = 0; e < E; ++e) out[e] = p[e] * ((dv[e] + c[e]) - gp);
    } else {
      double ssum = 0;
      for (int64_t e = 0; e < E; ++e) ssum += v[e];
      double cq = 0;                                     // <c, q>
      for (int64_t e = 0; e < E; ++e) cq += c[e] * (v[e] / ssum);
      for (int64_t e = 0; e < E; ++e) {
        const double ds = dv[e] + (c[e] - cq) / ssum;
        out[e] = ds * v[e] * (1.0 - v[e]);
      }
    }
    for (int64_t e = 0; e < E; ++e) out[e] += beta * (2.0 / T) * lse * p[e];
  });
}

// With g = x W_gate^T: dL/dW_gate = dg^T x [E, d] and dL/dx = dg W_gate [T, d] (double; each
// sum in index order).
void orc_router_param_grads(int64_t T, int64_t d, int64_t E, const void* x, int32_t xdt,
                            const void* w_gate, int32_t wdt, const double* dg, double* dW,
                            double* dx) {
  parallel_for(E, [&](int64_t e) {
    for (int64_t c = 0; c < d; ++c) {
      double s = 0;
      for (int64_t t = 0; t < T; ++t) s += dg[t * E + e] * elem(x, xdt, t * d + c);
      dW[e * d + c] = s;
    }
  });
  parallel_for(T, [&](int64_t t) {
    for (int64_t c = 0; c < d; ++c) {
      double s = 0;
      for (int64_t e = 0; e < E; ++e) s += dg[t * E + e] * elem(w_gate, wdt, e * d + c);
      dx[t * d + c] = s;
    }
  });
}

// One step of the loss-free balancing bias rule ([L17] §3.4; [A] update_bias code block): an
// expert whose load is above the mean load T*k/E gets b -= gamma, one below gets b += gamma,
// one exactly at the mean keeps b.  The load is the number of (token, choice) selections
// before any capacity drop, compared exactly as integers (counts * E vs T * k).  The bias is
// float32 state and the update is one float32 addition.
void orc_bias_update(int64_t E, const float* bias, const int64_t* counts, int64_t T, int64_t k,
                     float gamma, float* out) {
  for (int64_t e = 0; e < E; ++e) {
    const int64_t load = counts[e] * E, target = T * k;
    if (load > target) out[e] = bias[e] - gamma;
    else if (load < target) out[e] = bias[e] + gamma;
    else out[e] = bias[e];
  }
}

// ---------------------------------------------------------------------------------------------
// FP8 (E4M3) expert weights and activations for decode ([L17] §1.4: DeepSeek-V3 keeps its
// weights in FP8; [I] §4.2: per-expert quantisation)
// ---------------------------------------------------------------------------------------------
// Nearest E4M3 value of a float32 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
// infinities; largest finite 448 = 1.75 * 2^8, smallest subnormal 2^-9), ties to the even
// mantissa, beyond 448 saturated to +-448.  The grid spacing in the binade [2^e, 2^(e+1)) is
// 2^(e-3) for e >= -6, and 2^-9 below.
double e4m3(float v32) {
  const double v = static_cast<double>(v32);
  const double a = std::fabs(v);
  int ex = 0;
  std::frexp(a > 0 ? a : 1.0, &ex);                    // a = m 2^ex, m in [0.5, 1)
  const int e = std::max(ex - 1, -6);
  const double quantum = std::ldexp(1.0, e - 3);
  double r = std::nearbyint(a / quantum) * quantum;    // default rounding: ties to even
  r = std::min(r, 448.0);
  return std::copysign(r, v);
}

void orc_e4m3_round(int64_t n, const float* v, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3(v[i]);
}

// Test switch: with it on, the row quantiser below is the identity (codes = the float32 values,
// scale 1), so that a test can check that the FP8 layer reduces to the bf16 layer and thereby
// that it quantises the right rows and applies their scales in the right places.
int g_fp8_identity = 0;
void orc_set_fp8_identity(int32_t on) { g_fp8_identity = on; }

// Per-row E4M3 quantisation with the decisions in float32: amax = max |v| over the row,
// inv = float32(448 / amax), code = e4m3(float32(v * inv)), scale = float32(amax / 448); a row
// of zeros gets codes 0 and scale 0.  The row is represented by codes * scale.
void orc_quantize_rows_fp8(int64_t rows, int64_t cols, const float* V, double* codes,
                           double* scales) {
  if (g_fp8_identity) {
    for (int64_t i = 0; i < rows * cols; ++i) codes[i] = V[i];
    for (int64_t r = 0; r < rows; ++r) scales[r] = 1.0;
    return;
  }
  parallel_for(rows, [&](int64_t r) {
    const float* v = V + r * cols;
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) amax = std::max(amax, std::fabs(v[c]));
    const float inv = amax > 0 ? 448.0f / amax : 0.0f;
    for (int64_t c = 0; c < cols; ++c) codes[r * cols + c] = e4m3(v[c] * inv);
    scales[r] = amax > 0 ? static_cast<double>(amax / 448.0f) : 0.0;
  });
}

// codes * scale of the per-row quantisation of a weight tensor given as float32 rows
// [rows, cols] (bf16 weights widen exactly to float32).
void orc_dequantized_fp8(int64_t rows, int64_t cols, const void* W, int32_t wdt, double* out) {
  parallel_for(rows, [&](int64_t r) {
    std::vector<float> v(cols);
    std::vector<double> c(cols);
    for (int64_t i = 0; i < cols; ++i) v[i] = static_cast<float>(elem(W, wdt, r * cols + i));
    double s = 0;
    orc_quantize_rows_fp8(1, cols, v.data(), c.data(), &s);
    for (int64_t i = 0; i < cols; ++i) out[r * cols + i] = c[i] * s;
  });
}

// One SwiGLU expert on dequantised E4M3 token rows xd [n, d] with dequantised weights
// W13 [2F, d] and W2 [d, F] (double): h = SiLU(x W1^T) * (x W3^T) in double, rounded to
// float32, quantised per row, then y = h_q W2^T.  y [n, d].
void orc_fp8_ffn(int64_t n, int64_t d, int64_t F, const double* xd, const double* W13,
                 const double* W2, double* y) {
  parallel_for(n, [&](int64_t i) {
    std::vector<double> a(F), b(F), hq(F);
    std::vector<float> h32(F);
    rows_dot(xd + i * d, W13, F64, 0, F, d, a.data());
    rows_dot(xd + i * d, W13, F64, F, F, d, b.data());
    for (int64_t f = 0; f < F; ++f) h32[f] = static_cast<float>(silu(a[f]) * b[f]);
    double hs = 0;
    orc_quantize_rows_fp8(1, F, h32.data(), hq.data(), &hs);
    for (int64_t f = 0; f < F; ++f) hq[f] *= hs;
    rows_dot(hq.data(), W2, F64, 0, d, F, y + i * d);
  });
}

// ---------------------------------------------------------------------------------------------
// The layer on given selections, evaluated token by token (sampled checks of full-size layers):
//   out[n] = Shared(x_t) + sum_{j : row_of[t, j] >= 0} w[t, j] Expert_{idx[t, j]}(x_t),
//   t = tokens[n]
// Expert weights come one pointer per expert (w13_e [2F, d], w2_e [d, F]); only the experts the
// listed tokens select are read.  ws13 / ws2 (n_shared experts concatenated, [2Fs, d] and
// [d, Fs]) may be NULL.  out [n_tok, d] double.
// ---------------------------------------------------------------------------------------------
void orc_forward_tokens(int64_t n_tok, const int32_t* tokens, int64_t d, int64_t k, int64_t F,
                        int64_t Fs, const void* x, int32_t xdt, const int32_t* idx,
                        const double* w, const int32_t* row_of, const void* const* w13,
                        const void* const* w2, int32_t wdt, const void* ws13, const void* ws2,
                        double* out) {
  // one task per (token, addend): addend 0 is the shared expert, 1..k the routed choices; each
  // task writes its own row of a scratch array, summed in order afterwards
  const int64_t per = k + 1;
  std::vector<double> part(n_tok * per * d, 0.0);
  std::vector<char> live(n_tok * per, 0);
  parallel_for(n_tok * per, [&](int64_t task) {
    const int64_t n = task / per, a = task % per;
    const int32_t t = tokens[n];
    double* y = part.data() + task * d;
    if (a == 0) {
      if (!ws13) return;
      orc_swiglu(1, &t, d, Fs, x, xdt, ws13, wdt, ws2, wdt, y);
      live[task] = 1;
      return;
    }
    const int64_t j = a - 1;
    if (row_of[static_cast<int64_t>(t) * k + j] < 0) return;
    const int32_t e = idx[static_cast<int64_t>(t) * k + j];
    orc_swiglu(1, &t, d, F, x, xdt, w13[e], wdt, w2[e], wdt, y);
    const double wt = w[static_cast<int64_t>(t) * k + j];
    for (int64_t c = 0; c < d; ++c) y[c] *= wt;
    live[task] = 1;
  });
  for (int64_t n = 0; n < n_tok; ++n) {
    double* o = out + n * d;
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t a = 0; a < per; ++a) {
      if (!live[n * per + a]) continue;
      const double* y = part.data() + (n * per + a) * d;
      for (int64_t c = 0; c < d; ++c) o[c] += y[c];
    }
  }
}

// The FP8 layer on given selections for the listed tokens ([L17] §1.4; [I] §4.2): every row
// that enters an expert GEMM (the token's x for gate/up, its h for down) is quantised per row
// as in orc_quantize_rows_fp8, the weights per row likewise (quantize_weights = 1: w13/w2/ws13/
// ws2 hold the bf16/float32 weights and each needed expert is quantised here; 0: they hold the
// dequantised values already, as double).  The products are exact in double.  Summation: the
// shared experts first, then the routed experts in ascending expert order.  out [n_tok, d].
void orc_forward_tokens_fp8(int64_t n_tok, const int32_t* tokens, int64_t d, int64_t k,
                            int64_t F, int64_t Fs, int64_t E, const void* x, int32_t xdt,
                            const int32_t* idx, const double* w, const int32_t* row_of,
                            const void* const* w13, const void* const* w2, int32_t wdt,
                            const void* ws13, const void* ws2, int32_t quantize_weights,
                            double* out) {
  std::vector<float> x32(n_tok * d);
  for (int64_t n = 0; n < n_tok; ++n)
    for (int64_t c = 0; c < d; ++c)
      x32[n * d + c] = static_cast<float>(elem(x, xdt, static_cast<int64_t>(tokens[n]) * d + c));
  std::vector<double> xd(n_tok * d), xs(n_tok);
  orc_quantize_rows_fp8(n_tok, d, x32.data(), xd.data(), xs.data());
  for (int64_t n = 0; n < n_tok; ++n)
    for (int64_t c = 0; c < d; ++c) xd[n * d + c] *= xs[n];
  for (int64_t i = 0; i < n_tok * d; ++i) out[i] = 0.0;
  // one expert's weights as dequantised double arrays
  auto weights_of = [&](const void* a13, const void* a2, int64_t FF, std::vector<double>& W13,
                        std::vector<double>& W2) {
    W13.assign(2 * FF * d, 0.0);
    W2.assign(d * FF, 0.0);
    if (quantize_weights) {
      orc_dequantized_fp8(2 * FF, d, a13, wdt, W13.data());
      orc_dequantized_fp8(d, FF, a2, wdt, W2.data());
    } else {
      for (int64_t i = 0; i < 2 * FF * d; ++i) W13[i] = elem(a13, wdt, i);
      for (int64_t i = 0; i < d * FF; ++i) W2[i] = elem(a2, wdt, i);
    }
  };
  std::vector<double> W13, W2;
  if (ws13) {
    weights_of(ws13, ws2, Fs, W13, W2);
    std::vector<double> y(n_tok * d);
    orc_fp8_ffn(n_tok, d, Fs, xd.data(), W13.data(), W2.data(), y.data());
    for (int64_t i = 0; i < n_tok * d; ++i) out[i] += y[i];
  }
  for (int64_t e = 0; e < E; ++e) {
    std::vector<int64_t> sel_n, sel_j;
    for (int64_t n = 0; n < n_tok; ++n)
      for (int64_t j = 0; j < k; ++j) {
        const int64_t tj = static_cast<int64_t>(tokens[n]) * k + j;
        if (idx[tj] == e && row_of[tj] >= 0) {
          sel_n.push_back(n);
          sel_j.push_back(j);
        }
      }
    if (sel_n.empty()) continue;
    weights_of(w13[e], w2[e], F, W13, W2);
    const int64_t m = static_cast<int64_t>(sel_n.size());
    std::vector<double> xe(m * d), y(m * d);
    for (int64_t i = 0; i < m; ++i)
      std::copy(xd.begin() + sel_n[i] * d, xd.begin() + (sel_n[i] + 1) * d, xe.begin() + i * d);
    orc_fp8_ffn(m, d, F, xe.data(), W13.data(), W2.data(), y.data());
    for (int64_t i = 0; i < m; ++i) {
      const double wt = w[static_cast<int64_t>(tokens[sel_n[i]]) * k + sel_j[i]];
      for (int64_t c = 0; c < d; ++c) out[sel_n[i] * d + c] += wt * y[i * d + c];
    }
  }
}

// ---------------------------------------------------------------------------------------------
// The whole layer
// ---------------------------------------------------------------------------------------------
struct OrcConfig {
  int64_t T, d, E, k, F, Fs;
  int32_t score;            // 0 softmax, 1 sigmoid + selection bias
  int32_t n_groups, topk_groups, renormalize;
  double route_scale;
  float capacity_factor;    // <= 0: no limit
};

// Token-choice routing of a layer: logits, then the softmax or the sigmoid/group gate.
// g32 [T, E], idx [T, k], w [T, k]; prob [T, E] (softmax p, or sigmoid s) may be NULL.
int32_t orc_route(const OrcConfig* c, const void* x, int32_t xdt, const void* w_gate,
                  int32_t gdt, const float* bias, double* g, float* g32, int32_t* idx, double* w,
                  double* prob) {
  orc_router_logits(c->T, c->d, c->E, x, xdt, w_gate, gdt, g, g32);
  std::vector<double> gw(c->T * c->E);                 // the float32 logits, widened
  for (int64_t i = 0; i < c->T * c->E; ++i) gw[i] = g32[i];
  if (c->score == 0) {
    orc_softmax_topk_route(c->T, c->E, c->k, gw.data(), c->renormalize, c->route_scale, idx, w,
                           prob);
    return 0;
  }
  std::vector<float> zero;
  if (!bias) zero.assign(c->E, 0.0f);
  return orc_sigmoid_group_route(c->T, c->E, c->k, gw.data(), bias ? bias : zero.data(),
                                 c->n_groups, c->topk_groups, c->route_scale, c->renormalize,
                                 idx, w, prob);
}

// Token-choice MoE layer forward ([R] §2.1 and §2.2; [L17] §2.2 steps 1-4 and §5.2): route,
// dispatch with capacity, SwiGLU experts on the dispatched rows, shared experts, weighted
// combine, and the load-balance statistics.  Expert weights one pointer per expert.
// Outputs (caller-owned): g32 [T,E]; idx, w [T,k]; counts, kept [E]; offsets [E+1]; pos,
// row_of [T,k]; perm [T*k]; n_dropped; y_rows [T*k, d] (rows past offsets[E] untouched);
// shared [T, d] (NULL when Fs == 0); out [T, d]; f, P [E]; stats4 as in
// orc_aux_stats_from_counts.  Returns 0, or a negative code from routing or dispatch.
int32_t orc_moe_forward(const OrcConfig* c, const void* x, int32_t xdt, const void* w_gate,
                        int32_t gdt, const float* bias, const void* const* w13,
                        const void* const* w2, int32_t wdt, const void* ws13, const void* ws2,
                        double* g, float* g32, int32_t* idx, double* w, double* prob,
                        int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* pos,
                        int32_t* row_of, int32_t* perm, int64_t* n_dropped, double* y_rows,
                        double* shared, double* out, double* f, double* P, double* stats4) {
  const int64_t T = c->T, d = c->d, E = c->E, k = c->k;
  int32_t st = orc_route(c, x, xdt, w_gate, gdt, bias, g, g32, idx, w, prob);
  if (st) return st;
  const int64_t C = orc_capacity(c->capacity_factor, k, T, E);
  st = orc_dispatch(T, k, E, idx, C, counts, kept, offsets, pos, row_of, perm, n_dropped);
  if (st) return st;
  // y_rows[row] = Expert_e(x[t]) for every kept pair (row = offsets[e] + pos, t = perm / k)
  const int64_t nrows = offsets[E];
  std::vector<int32_t> row_expert(nrows);
  for (int64_t e = 0; e < E; ++e)
    for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) row_expert[r] = static_cast<int32_t>(e);
  parallel_for(nrows, [&](int64_t r) {
    const int32_t t = static_cast<int32_t>(perm[r] / k);
    const int32_t e = row_expert[r];
    orc_swiglu(1, &t, d, c->F, x, xdt, w13[e], wdt, w2[e], wdt, y_rows + r * d);
  });
  if (c->Fs > 0) orc_swiglu(T, nullptr, d, c->Fs, x, xdt, ws13, wdt, ws2, wdt, shared);
  orc_combine(T, d, k, w, row_of, y_rows, c->Fs > 0 ? shared : nullptr, out);
  std::vector<double> cnt(E), gw(T * E);
  for (int64_t e = 0; e < E; ++e) cnt[e] = counts[e];
  for (int64_t i = 0; i < T * E; ++i) gw[i] = g32[i];
  orc_aux_stats_from_counts(T, E, gw.data(), cnt.data(), c->score, f, P, stats4);
  return 0;
}

// Expert-choice variant ([G] §2.2): out[t] = shared[t] + sum_{e chose t} p[t,e] Expert_e(x_t),
// the sum over the choosing experts in ascending expert order.  tokens, weights [E, C] with
// C = T*k/E; ptr [T+1], rows [E*C] (orc_expert_choice_csr); out [T, d]; f, P [E] and stats4
// from the counts C per expert.
void orc_moe_forward_expert_choice(const OrcConfig* c, const void* x, int32_t xdt,
                                   const void* w_gate, int32_t gdt, const void* const* w13,
                                   const void* const* w2, int32_t wdt, const void* ws13,
                                   const void* ws2, double* g, float* g32, int32_t* tokens,
                                   double* weights, double* prob, int32_t* ptr, int32_t* rows,
                                   double* out, double* f, double* P, double* stats4) {
  const int64_t T = c->T, d = c->d, E = c->E, k = c->k;
  const int64_t C = (T * k) / E;
  orc_router_logits(T, d, E, x, xdt, w_gate, gdt, g, g32);
  std::vector<double> gw(T * E);                       // the float32 logits, widened
  for (int64_t i = 0; i < T * E; ++i) gw[i] = g32[i];
  orc_expert_choice_route(T, E, k, gw.data(), tokens, weights, prob);
  orc_expert_choice_csr(E, C, T, tokens, ptr, rows, nullptr);
  std::vector<double> y(E * C * d);
  parallel_for(E * C, [&](int64_t r) {
    const int64_t e = r / C;
    orc_swiglu(1, tokens + r, d, c->F, x, xdt, w13[e], wdt, w2[e], wdt, y.data() + r * d);
  });
  if (c->Fs > 0) orc_swiglu(T, nullptr, d, c->Fs, x, xdt, ws13, wdt, ws2, wdt, out);
  else
    for (int64_t i = 0; i < T * d; ++i) out[i] = 0.0;
  parallel_for(T, [&](int64_t t) {
    for (int32_t q = ptr[t]; q < ptr[t + 1]; ++q) {
      const int64_t r = rows[q];
      const double wt = weights[r];
      for (int64_t cc = 0; cc < d; ++cc) out[t * d + cc] += wt * y[r * d + cc];
    }
  });
  std::vector<double> cnt(E, static_cast<double>(C));
  orc_aux_stats_from_counts(T, E, gw.data(), cnt.data(), 0, f, P, stats4);
}

}  // extern "C"

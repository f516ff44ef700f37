// Plain fp64 CPU oracle of the sparse Mixture-of-Experts FFN layer's
// forward pass and its backward, in single-threaded C++.
//
// TEST INFRASTRUCTURE ONLY.  This is a checker: the tests, the smoke check
// and the benchmark's CPU-baseline leg may call it; the CUDA library never
// does, and it shares no code with the CUDA path.  It restates the same
// definitions as moe_oracle.py, in plain loops written in the order the
// pages state the method, and the tests hold the two oracles to each other
// and to the pages' worked examples.
//
// Inputs are the stored bits the GPU reads: fp32 or bf16 elements, decoded
// exactly to fp64 on every read (bf16 is the upper half of an fp32 word),
// so both sides start from identical values.  Every sum runs in index
// order in fp64; there is no blocking, threading or reordering.
//
// Sources (page title -- section):
//   [P1] "'More parameters is better' is not the story: the expert group
//        quietly activated inside a large model" -- 3.1 Router, 3.3 Gate,
//        4.2 model definition.
//   [P2] "MoE mixture-of-experts architecture: principles and engineering
//        practice" -- 4.2 building an MoE model.
//   [P3] "MoE architecture revealed: why total parameters != active
//        parameters" -- 2.3 router design, 3.3 TinyMoE.
//   [P5] "Training a 200B LLM from scratch 5/25: how does MoE compute with
//        part of its parameters?" -- "Who decides which experts to call?",
//        "Shared experts".
//
// Readings (the same as the numpy oracle's): selection on the logits with
// ties to the lower expert index; weights = the softmax of the selected
// logits; capacity C = max(min_capacity, ceil(cf*T*k/E)) with the ceiling
// of the exact rational value of the caller's fp32 cf, no limit when
// cf <= 0; overflow in slot-major priority (every token's first choice in
// token order, then every second choice); a dropped slot adds nothing; GeLU
// is the exact erf form; SwiGLU is W2 (silu(W1 v) * (W3 v)); the shared
// expert is added with weight 1; usage statistic lambda * std_{n-1}(f) /
// (mean(f) + 1e-8) on pre-capacity counts f = counts / T; a token with a
// non-finite logit is routed to no expert.  The routing variants -- raw
// probabilities, token-major priority, a LayerNorm in front, rerouting --
// and the other balance forms are here too (mo_config.route, .balance).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// stored inputs
// ---------------------------------------------------------------------------
enum { MO_F32 = 0, MO_BF16 = 1 };

// Element i of a stored tensor, exactly, as fp64.
inline double rd(const void* p, int dtype, long long i) {
  if (dtype == MO_BF16) {
    const uint32_t u = static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
  }
  return static_cast<const float*>(p)[i];
}

inline bool all_finite(const double* v, int n) {
  for (int i = 0; i < n; ++i)
    if (!std::isfinite(v[i])) return false;
  return true;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// router ([P1] 3.1, 3.3, 4.2; [P3] 2.3)
// ---------------------------------------------------------------------------

// l[t,e] = sum_i x[t,i] Wr[e,i] (+ bias[e]) (+ noise[t,e]).  x [T,d] and Wr
// [E,d] in `dtype`; bias [E] and noise [T,E] fp32, either may be null.
// [P1] 3.1: the logits are h W_r; [P3] 2.3: Gumbel noise is added to the
// router's scores before the top-k.
void mo_router_logits(int T, int d, int E, int dtype, const void* x, const void* Wr, const float* bias,
                      const float* noise, double* l) {
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int i = 0; i < d; ++i)
        s += rd(x, dtype, static_cast<long long>(t) * d + i) * rd(Wr, dtype, static_cast<long long>(e) * d + i);
      if (bias) s += bias[e];
      if (noise) s += noise[static_cast<long long>(t) * E + e];
      l[static_cast<long long>(t) * E + e] = s;
    }
  }
}

// Row-wise layer norm of the stored x [T,d] into fp64 rows n [T,d]:
// (x - mean) / sqrt(var + 1e-5), var the biased (1/d) variance -- [P2] 5.2's
// LayerNorm in front of the router, at its initial identity scale and zero
// shift.
void mo_layer_norm(int T, int d, int dtype, const void* x, double* n) {
  for (int t = 0; t < T; ++t) {
    double mu = 0.0;
    for (int i = 0; i < d; ++i) mu += rd(x, dtype, static_cast<long long>(t) * d + i);
    mu /= d;
    double var = 0.0;
    for (int i = 0; i < d; ++i) {
      const double c = rd(x, dtype, static_cast<long long>(t) * d + i) - mu;
      var += c * c;
    }
    var /= d;
    const double r = 1.0 / std::sqrt(var + 1e-5);
    for (int i = 0; i < d; ++i)
      n[static_cast<long long>(t) * d + i] = (rd(x, dtype, static_cast<long long>(t) * d + i) - mu) * r;
  }
}

// The gradient with respect to x of <g, layer_norm(x)>, added to dx [T,d]:
// with n the normalised row and r = 1 / sqrt(var + 1e-5), the chain rule of
// the row normalisation gives r (g - mean(g) - n mean(g n)).
void mo_layer_norm_backward(int T, int d, int dtype, const void* x, const double* g, double* dx) {
  std::vector<double> n(static_cast<size_t>(d));
  for (int t = 0; t < T; ++t) {
    double mu = 0.0;
    for (int i = 0; i < d; ++i) mu += rd(x, dtype, static_cast<long long>(t) * d + i);
    mu /= d;
    double var = 0.0;
    for (int i = 0; i < d; ++i) {
      const double c = rd(x, dtype, static_cast<long long>(t) * d + i) - mu;
      var += c * c;
    }
    var /= d;
    const double r = 1.0 / std::sqrt(var + 1e-5);
    const double* gt = g + static_cast<long long>(t) * d;
    double gm = 0.0, gn = 0.0;
    for (int i = 0; i < d; ++i) {
      n[i] = (rd(x, dtype, static_cast<long long>(t) * d + i) - mu) * r;
      gm += gt[i];
      gn += gt[i] * n[i];
    }
    gm /= d;
    gn /= d;
    for (int i = 0; i < d; ++i) dx[static_cast<long long>(t) * d + i] += r * (gt[i] - gm - n[i] * gn);
  }
}

// Router logits from fp64 rows xr [T,d] (the layer-normed x): l[t,e] = sum_i
// xr[t,i] Wr[e,i] (+ bias[e]) (+ noise[t,e]), Wr stored in `dtype`.
void mo_router_logits_rows(int T, int d, int E, int dtype, const double* xr, const void* Wr, const float* bias,
                           const float* noise, double* l) {
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int i = 0; i < d; ++i)
        s += xr[static_cast<long long>(t) * d + i] * rd(Wr, dtype, static_cast<long long>(e) * d + i);
      if (bias) s += bias[e];
      if (noise) s += noise[static_cast<long long>(t) * E + e];
      l[static_cast<long long>(t) * E + e] = s;
    }
  }
}

// Top-k experts per token by (logit descending, index ascending) -- softmax
// is monotone, so this is [P1] 4.2's top-k of the probabilities -- and their
// weights w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0), the softmax of the
// selected logits ([P1] 3.3: p_i / (p_i + p_j); [P3] 3.3).  A token with a
// non-finite logit gets idx = -1 and w = 0 in every slot.  Returns the
// number of such tokens.
int mo_top_k_probs(int T, int E, int k, const double* l, int raw, int* idx, double* w);

int mo_top_k(int T, int E, int k, const double* l, int* idx, double* w) {
  return mo_top_k_probs(T, E, k, l, 0, idx, w);
}

// mo_top_k with raw != 0: the weights are the selected entries of the
// softmax over all E experts, not renormalised ([P2] 3.2: output = p1 e1 +
// p2 e2; [P4] 5.1 uses the top-k probabilities as they are).
int mo_top_k_probs(int T, int E, int k, const double* l, int raw, int* idx, double* w) {
  int nonfinite = 0;
  std::vector<char> taken(E);
  for (int t = 0; t < T; ++t) {
    const double* lt = l + static_cast<long long>(t) * E;
    int* it = idx + static_cast<long long>(t) * k;
    double* wt = w + static_cast<long long>(t) * k;
    if (!all_finite(lt, E)) {
      ++nonfinite;
      for (int j = 0; j < k; ++j) {
        it[j] = -1;
        wt[j] = 0.0;
      }
      continue;
    }
    // k rounds: the largest logit not yet taken; the first index wins a tie
    std::fill(taken.begin(), taken.end(), 0);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || lt[e] > lt[best])) best = e;
      taken[best] = 1;
      it[j] = best;
    }
    double z = 0.0;
    if (raw)
      for (int e = 0; e < E; ++e) z += std::exp(lt[e] - lt[it[0]]);
    else
      for (int j = 0; j < k; ++j) z += std::exp(lt[it[j]] - lt[it[0]]);
    for (int j = 0; j < k; ++j) wt[j] = std::exp(lt[it[j]] - lt[it[0]]) / z;
  }
  return nonfinite;
}

// Mean over the tokens with finite logits of H_t = -sum_e p_te ln p_te,
// p_t = the softmax over all E experts ([P3]'s monitoring of the router
// entropy).  NaN when no token has finite logits.
double mo_router_entropy(int T, int E, const double* l) {
  double sum = 0.0;
  long long n = 0;
  std::vector<double> p(E);
  for (int t = 0; t < T; ++t) {
    const double* lt = l + static_cast<long long>(t) * E;
    if (!all_finite(lt, E)) continue;
    double m = lt[0];
    for (int e = 1; e < E; ++e) m = lt[e] > m ? lt[e] : m;
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += (p[e] = std::exp(lt[e] - m));
    double h = 0.0;
    for (int e = 0; e < E; ++e) {
      const double pe = p[e] / z;
      if (pe > 0.0) h -= pe * std::log(pe);
    }
    sum += h;
    ++n;
  }
  return n ? sum / static_cast<double>(n) : std::nan("");
}

// ---------------------------------------------------------------------------
// capacity and dispatch ([P3] 2.3; [P1] 4.2 step 2)
// ---------------------------------------------------------------------------

// C = max(min_capacity, ceil(cf * T * k / E)), or T when cf <= 0 (no
// limit).  [P3] 2.3: batch 1024, top-2, 16 experts -> 1024 * 2 / 16 = 128.
// The ceiling is taken of the exact rational value of the fp32 cf the
// caller passed: cf = m * 2^p with an integer m, so ceil(m T k 2^p / E) is
// an integer division (128-bit numerator), never a rounded product.  A
// capacity above 2^31 - 1 is returned as 2^31 - 1.
int mo_capacity(int T, int k, int E, float capacity_factor, int min_capacity) {
  if (!(capacity_factor > 0.0f)) return T;
  int p = 0;
  const float frac = std::frexp(capacity_factor, &p);           // cf = frac * 2^p, frac in [0.5, 1)
  const long long m = static_cast<long long>(std::ldexp(frac, 24));  // cf = m * 2^(p - 24), exactly
  p -= 24;
  // m < 2^24, T k < 2^35, E < 2^31: the numerator is below 2^59, so a
  // value with p <= -59 lies in (0, 1) and one with p >= 40 is above 2^31
  long long cap;
  if (p <= -59) {
    cap = 1;
  } else if (p >= 40) {
    cap = 0x7fffffffLL;
  } else {
    unsigned __int128 num = static_cast<unsigned __int128>(m) * static_cast<unsigned long long>(T) *
                            static_cast<unsigned long long>(k);
    unsigned __int128 den = static_cast<unsigned __int128>(E);
    if (p >= 0) num <<= p;
    else den <<= -p;
    const unsigned __int128 c = (num + den - 1) / den;
    cap = c > 0x7fffffff ? 0x7fffffffLL : static_cast<long long>(c);
  }
  return static_cast<int>(cap > min_capacity ? cap : min_capacity);
}

// counts[e] = the (t, j) slots routed to expert e, before capacity.
void mo_usage_counts(int T, int k, int E, const int* idx, long long* counts) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long long s = 0; s < static_cast<long long>(T) * k; ++s)
    if (idx[s] >= 0) ++counts[idx[s]];
}

// Capacity in slot-major priority: for j = 0..k-1, for t = 0..T-1, the slot
// (t, j) takes the next free place of its expert if one of C is left, else
// it is dropped (rank -1).  fill[e] = the slots kept by expert e.
void mo_assign_capacity(int T, int k, int E, int C, const int* idx, int* rank, long long* fill) {
  for (int e = 0; e < E; ++e) fill[e] = 0;
  for (int j = 0; j < k; ++j) {
    for (int t = 0; t < T; ++t) {
      const long long s = static_cast<long long>(t) * k + j;
      const int e = idx[s];
      if (e >= 0 && fill[e] < C) rank[s] = static_cast<int>(fill[e]++);
      else rank[s] = -1;
    }
  }
}

// The same queue in token-major priority: token 0's choices in order, then
// token 1's, and so on.
void mo_assign_capacity_token_major(int T, int k, int E, int C, const int* idx, int* rank, long long* fill) {
  for (int e = 0; e < E; ++e) fill[e] = 0;
  for (long long s = 0; s < static_cast<long long>(T) * k; ++s) {
    const int e = idx[s];
    if (e >= 0 && fill[e] < C) rank[s] = static_cast<int>(fill[e]++);
    else rank[s] = -1;
  }
}

// Each token's experts ranked k .. 2k-1 by (logit descending, index
// ascending): its next-best experts, which slots that overflow can be
// rerouted to ([P3] 2.3).  -1 where fewer than 2k experts exist or the
// token has a non-finite logit.  backup [T,k].
void mo_backup_experts(int T, int E, int k, const double* l, int* backup) {
  const int nb = std::max(0, std::min(k, E - k));
  std::vector<char> taken(E);
  for (int t = 0; t < T; ++t) {
    const double* lt = l + static_cast<long long>(t) * E;
    int* bt = backup + static_cast<long long>(t) * k;
    for (int j = 0; j < k; ++j) bt[j] = -1;
    if (!all_finite(lt, E)) continue;
    std::fill(taken.begin(), taken.end(), 0);
    for (int r = 0; r < k + nb; ++r) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || lt[e] > lt[best])) best = e;
      taken[best] = 1;
      if (r >= k) bt[r - k] = best;
    }
  }
}

// The second capacity pass ([P3] 2.3: tokens beyond capacity are dropped or
// routed to the next-best expert).  The r-th slot of token t that the first
// pass dropped (r counted in choice order) tries backup[t,r] once; slots
// are visited in the first pass's priority order.  It is kept if that
// expert has room left after the first pass and the slots rerouted to it
// before, taking the next place after the expert's first-pass rows.
// served [T,k]: the expert serving each slot (-1 none); rank2 [T,k]: place
// among the expert's rerouted rows (-1 if not rerouted); fill2 [E]: rerouted
// rows per expert.
void mo_reroute_overflow(int T, int k, int E, int C, const int* idx, const int* backup, const int* rank,
                         const long long* fill, int token_major, int* served, int* rank2, long long* fill2) {
  const long long S = static_cast<long long>(T) * k;
  std::vector<int> nth(S, -1);
  for (int t = 0; t < T; ++t) {
    int r = 0;
    for (int j = 0; j < k; ++j) {
      const long long s = static_cast<long long>(t) * k + j;
      if (idx[s] >= 0 && rank[s] < 0) nth[s] = r++;
    }
  }
  for (long long s = 0; s < S; ++s) {
    served[s] = rank[s] >= 0 ? idx[s] : -1;
    rank2[s] = -1;
  }
  for (int e = 0; e < E; ++e) fill2[e] = 0;
  for (long long q = 0; q < S; ++q) {
    // q-th slot in priority order: token-major (t, j) = (q / k, q % k), or
    // slot-major (t, j) = (q % T, q / T)
    const long long s = token_major ? q : (q % T) * k + q / T;
    if (nth[s] < 0) continue;
    const int b = backup[(s / k) * k + nth[s]];
    if (b < 0) continue;
    if (fill[b] + fill2[b] < C) {
      rank2[s] = static_cast<int>(fill2[b]++);
      served[s] = b;
    }
  }
}

// offsets = the exclusive scan of fill (expert e's rows are [offsets[e],
// offsets[e+1]) of the expert-contiguous matrix); pos[t,j] = offsets[e] +
// rank for a kept slot, else -1.
void mo_dispatch_positions(int T, int k, int E, const int* idx, const int* rank, const long long* fill,
                           long long* offsets, long long* pos) {
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + fill[e];
  for (long long s = 0; s < static_cast<long long>(T) * k; ++s)
    pos[s] = rank[s] >= 0 ? offsets[idx[s]] + rank[s] : -1;
}

// ---------------------------------------------------------------------------
// experts and combine ([P2] 4.2; [P3] 3.3; [P5])
// ---------------------------------------------------------------------------

// One expert FFN on n rows v [n,d] (stored in `dtype`, row stride d) ->
// out [n,d] fp64.  act 0, GeLU: W2 gelu(W1 v + b1) + b2, gelu(z) = z (1 +
// erf(z / sqrt 2)) / 2 ([P2] 4.2, [P3] 3.3: Linear, GELU, Linear).  act 1,
// SwiGLU: W2 (silu(W1 v) * (W3 v)), silu(z) = z / (1 + e^-z).  W1, W3 [h,d],
// W2 [d,h] and the biases b1 [h], b2 [d] (null: none) in `dtype`.  Each
// weight row is read once for all n rows; every output element is its own
// sum in index order.
void mo_expert_ffn(int n, int d, int h, int act, int dtype, const void* v, const void* W1, const void* W3,
                   const void* b1, const void* W2, const void* b2, double* out) {
  std::vector<double> vr(static_cast<size_t>(n) * d), hid(static_cast<size_t>(n) * h), wrow(d), grow(d), orow(h);
  for (long long i = 0; i < static_cast<long long>(n) * d; ++i) vr[i] = rd(v, dtype, i);
  for (int u = 0; u < h; ++u) {
    for (int i = 0; i < d; ++i) wrow[i] = rd(W1, dtype, static_cast<long long>(u) * d + i);
    if (act == 1)
      for (int i = 0; i < d; ++i) grow[i] = rd(W3, dtype, static_cast<long long>(u) * d + i);
    for (int r = 0; r < n; ++r) {
      const double* vrow = vr.data() + static_cast<long long>(r) * d;
      double z = 0.0;
      for (int i = 0; i < d; ++i) z += wrow[i] * vrow[i];
      if (act == 0) {
        if (b1) z += rd(b1, dtype, u);
        hid[static_cast<long long>(r) * h + u] = z * 0.5 * (1.0 + std::erf(z / std::sqrt(2.0)));
      } else {
        double g = 0.0;
        for (int i = 0; i < d; ++i) g += grow[i] * vrow[i];
        hid[static_cast<long long>(r) * h + u] = z / (1.0 + std::exp(-z)) * g;
      }
    }
  }
  for (int col = 0; col < d; ++col) {
    for (int u = 0; u < h; ++u) orow[u] = rd(W2, dtype, static_cast<long long>(col) * h + u);
    const double bias = (act == 0 && b2) ? rd(b2, dtype, col) : 0.0;
    for (int r = 0; r < n; ++r) {
      const double* hr = hid.data() + static_cast<long long>(r) * h;
      double o = 0.0;
      for (int u = 0; u < h; ++u) o += orow[u] * hr[u];
      out[static_cast<long long>(r) * d + col] = o + bias;
    }
  }
}

// y[t] = sum over the kept slots j (ascending) of w[t,j] * out[t,j,:], plus
// shared[t] when given.  [P5] "Who decides which experts to call?": the two
// chosen experts' outputs mixed in the routing proportions, 0.75 E1(x) +
// 0.25 E3(x); "Shared experts": the always-on expert's output is added.
// out [T,k,d], w [T,k], kept [T,k] (nonzero = kept), shared [T,d] or null.
void mo_combine(int T, int k, int d, const double* out, const double* w, const int* kept, const double* shared,
                double* y) {
  for (int t = 0; t < T; ++t) {
    double* yt = y + static_cast<long long>(t) * d;
    for (int c = 0; c < d; ++c) yt[c] = 0.0;
    for (int j = 0; j < k; ++j) {
      const long long s = static_cast<long long>(t) * k + j;
      if (!kept[s]) continue;
      for (int c = 0; c < d; ++c) yt[c] += w[s] * out[s * d + c];
    }
    if (shared)
      for (int c = 0; c < d; ++c) yt[c] += shared[static_cast<long long>(t) * d + c];
  }
}

// lambda * std_{n-1}(f) / (mean(f) + 1e-8) on f = counts / T ([P1] 3.1:
// L_balance = lambda * std(usage) / mean(usage); [P1] 4.2 averages the
// one-hot selection over the tokens, adds 1e-8 to the mean and uses the n-1
// standard deviation).  0 for a single expert.
double mo_balance_stat(int E, int T, const long long* counts, double lam) {
  if (E < 2) return 0.0;
  double mean = 0.0;
  for (int e = 0; e < E; ++e) mean += static_cast<double>(counts[e]) / T;
  mean /= E;
  double ss = 0.0;
  for (int e = 0; e < E; ++e) {
    const double f = static_cast<double>(counts[e]) / T - mean;
    ss += f * f;
  }
  return lam * std::sqrt(ss / (E - 1)) / (mean + 1e-8);
}

// The load statistic in the form `variant` gives, on the pre-capacity
// usage f = counts / T: 0, CV (mo_balance_stat); 1, lambda (std_{n-1}(f) +
// gamma max(f)) ([P2] 3.2's auxiliary loss on the experts' usage
// frequency); 2, lambda sum_e f_e P_e with P = I / T, I[e] the sum of the
// routing weights of the slots routed to e ([P3] 2.3's product of the
// usage fraction and the mean routing weight).  idx, w [T,k].
double mo_balance_stat_form(int E, int T, int k, const long long* counts, const int* idx, const double* w,
                            double lam, int variant, double gamma) {
  if (variant == 0) return mo_balance_stat(E, T, counts, lam);
  std::vector<double> f(static_cast<size_t>(E));
  for (int e = 0; e < E; ++e) f[e] = static_cast<double>(counts[e]) / T;
  if (variant == 1) {
    double mean = 0.0, mx = f[0];
    for (int e = 0; e < E; ++e) {
      mean += f[e];
      mx = std::max(mx, f[e]);
    }
    mean /= E;
    double ss = 0.0;
    for (int e = 0; e < E; ++e) ss += (f[e] - mean) * (f[e] - mean);
    const double sd = E > 1 ? std::sqrt(ss / (E - 1)) : 0.0;
    return lam * (sd + gamma * mx);
  }
  std::vector<double> imp(static_cast<size_t>(E), 0.0);
  for (long long s = 0; s < static_cast<long long>(T) * k; ++s)
    if (idx[s] >= 0) imp[idx[s]] += w[s];
  double v = 0.0;
  for (int e = 0; e < E; ++e) v += f[e] * (imp[e] / T);
  return lam * v;
}

// ---------------------------------------------------------------------------
// the layer
// ---------------------------------------------------------------------------

struct mo_config {
  int T, d, h, E, k;
  int act;    // 0 GeLU, 1 SwiGLU
  int dtype;  // storage of x and the weights: 0 fp32, 1 bf16
  int min_capacity;
  int has_shared;
  float capacity_factor;  // <= 0: no limit
  double lam;
  int balance;   // the balance form: 0 CV, 1 std + max, 2 switch (the forward's statistic, the backward's term)
  double gamma;  // its max weight (std + max)
  int route;     // MO_RAW_PROBS | MO_TOKEN_MAJOR | MO_LAYERNORM | MO_REROUTE
};

enum { MO_RAW_PROBS = 1, MO_TOKEN_MAJOR = 2, MO_LAYERNORM = 4, MO_REROUTE = 8 };



// Stored inputs (pointers in the config's dtype unless noted; null where
// absent).  W1/W3 [E,h,d], W2 [E,d,h], b1 [E,h], b2 [E,d]; the shared
// expert's Ws1/Ws3 [h,d], Ws2 [d,h], bs1 [h], bs2 [d]; bias [E] and noise
// [T,E] fp32.
struct mo_inputs {
  const void *x, *Wr, *W1, *W3, *b1, *W2, *b2, *Ws1, *Ws3, *bs1, *Ws2, *bs2;
  const float *bias, *noise;
};

// Outputs: y [T,d], idx/pos [T,k], w [T,k], counts/kept [E], offsets
// [E+1]; stats[0..8] = routed, kept and dropped slots, capacity, drop rate,
// balance statistic, tokens with a non-finite logit, mean router entropy,
// slots the rerouting pass kept.
struct mo_outputs {
  double* y;
  int* idx;
  double* w;
  long long *counts, *kept, *offsets, *pos;
  double* stats;
};

// The routing of a layer, shared by the forward and the backward: logits
// (from the layer-normed x with MO_LAYERNORM), top-k and weights, usage
// counts, capacity, ranks in the configured priority, with MO_REROUTE the
// second pass that offers the dropped slots their backups, and positions:
// each expert's first-pass rows, then its rerouted rows.  served [T,k] is
// the expert that serves each slot (-1 none); kept [E] counts both passes;
// *rerouted the slots the second pass kept.
static int route_layer(const mo_config* c, const mo_inputs* in, double* l, int* idx, double* w, long long* counts,
                       long long* kept, long long* offsets, long long* pos, int* served, int* C_out,
                       long long* rerouted) {
  const int T = c->T, d = c->d, E = c->E, k = c->k, dt = c->dtype;
  const long long S = static_cast<long long>(T) * k;
  if (c->route & MO_LAYERNORM) {
    std::vector<double> n(static_cast<size_t>(T) * d);
    mo_layer_norm(T, d, dt, in->x, n.data());
    mo_router_logits_rows(T, d, E, dt, n.data(), in->Wr, in->bias, in->noise, l);
  } else {
    mo_router_logits(T, d, E, dt, in->x, in->Wr, in->bias, in->noise, l);
  }
  const int nonfinite = mo_top_k_probs(T, E, k, l, (c->route & MO_RAW_PROBS) != 0, idx, w);
  mo_usage_counts(T, k, E, idx, counts);
  const int C = mo_capacity(T, k, E, c->capacity_factor, c->min_capacity);
  std::vector<int> rank(S);
  const bool tm = (c->route & MO_TOKEN_MAJOR) != 0;
  if (tm) mo_assign_capacity_token_major(T, k, E, C, idx, rank.data(), kept);
  else mo_assign_capacity(T, k, E, C, idx, rank.data(), kept);
  *rerouted = 0;
  if (c->route & MO_REROUTE) {
    std::vector<int> backup(S), rank2(S);
    std::vector<long long> fill2(E);
    mo_backup_experts(T, E, k, l, backup.data());
    mo_reroute_overflow(T, k, E, C, idx, backup.data(), rank.data(), kept, tm, served, rank2.data(), fill2.data());
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + kept[e] + fill2[e];
    for (long long s = 0; s < S; ++s) {
      if (rank[s] >= 0) pos[s] = offsets[idx[s]] + rank[s];
      else if (rank2[s] >= 0) pos[s] = offsets[served[s]] + kept[served[s]] + rank2[s];
      else pos[s] = -1;
    }
    for (int e = 0; e < E; ++e) {
      kept[e] += fill2[e];
      *rerouted += fill2[e];
    }
  } else {
    mo_dispatch_positions(T, k, E, idx, rank.data(), kept, offsets, pos);
    for (long long s = 0; s < S; ++s) served[s] = rank[s] >= 0 ? idx[s] : -1;
  }
  *C_out = C;
  return nonfinite;
}

// The whole forward pass, steps in the pages' order: logits, top-k and
// weights, usage counts, capacity, dispatch positions, each kept slot
// through its expert, the shared expert, the combine, the statistics.
// Returns 0, or -1 on an invalid configuration.
int mo_layer_forward(const mo_config* c, const mo_inputs* in, mo_outputs* out) {
  const int T = c->T, d = c->d, h = c->h, E = c->E, k = c->k, dt = c->dtype;
  if (T < 1 || d < 1 || h < 1 || E < 1 || k < 1 || k > E || (c->act != 0 && c->act != 1) ||
      (dt != MO_F32 && dt != MO_BF16) || c->balance < 0 || c->balance > 2 || (c->route & ~15))
    return -1;
  const long long S = static_cast<long long>(T) * k;
  const int es = dt == MO_BF16 ? 2 : 4;
  std::vector<double> l(static_cast<size_t>(T) * E);
  std::vector<int> served(S);
  int C = 0;
  long long rerouted = 0;
  const int nonfinite = route_layer(c, in, l.data(), out->idx, out->w, out->counts, out->kept, out->offsets,
                                    out->pos, served.data(), &C, &rerouted);

  // dispatch ([P1] 4.2 step 2: the tokens bound for the same expert grouped
  // together): the stored row of x[t] copied to row pos[t,j] of Xp; then
  // each expert once over its rows; slot (t,j)'s output is Yp[pos[t,j]]
  const long long rows = out->offsets[E];
  std::vector<char> Xp(static_cast<size_t>(rows) * d * es);
  for (long long s = 0; s < S; ++s)
    if (out->pos[s] >= 0)
      std::memcpy(Xp.data() + out->pos[s] * d * es, static_cast<const char*>(in->x) + (s / k) * d * es,
                  static_cast<size_t>(d) * es);
  std::vector<double> Yp(static_cast<size_t>(rows) * d);
  const auto at = [&](const void* base, long long elems) -> const void* {
    return base ? static_cast<const char*>(base) + elems * es : nullptr;
  };
  for (int e = 0; e < E; ++e) {
    const long long r0 = out->offsets[e], n = out->offsets[e + 1] - r0;
    if (n == 0) continue;
    mo_expert_ffn(static_cast<int>(n), d, h, c->act, dt, Xp.data() + r0 * d * es,
                  at(in->W1, static_cast<long long>(e) * h * d), at(in->W3, static_cast<long long>(e) * h * d),
                  at(in->b1, static_cast<long long>(e) * h), at(in->W2, static_cast<long long>(e) * d * h),
                  at(in->b2, static_cast<long long>(e) * d), Yp.data() + r0 * d);
  }
  std::vector<double> yslot(static_cast<size_t>(S) * d, 0.0);
  std::vector<int> keep(S);
  for (long long s = 0; s < S; ++s) {
    keep[s] = out->pos[s] >= 0;
    if (keep[s]) std::memcpy(&yslot[s * d], &Yp[out->pos[s] * d], sizeof(double) * d);
  }
  std::vector<double> shared;
  if (c->has_shared) {
    shared.resize(static_cast<size_t>(T) * d);
    mo_expert_ffn(T, d, h, c->act, dt, in->x, in->Ws1, in->Ws3, in->bs1, in->Ws2, in->bs2, shared.data());
  }
  mo_combine(T, k, d, yslot.data(), out->w, keep.data(), c->has_shared ? shared.data() : nullptr, out->y);

  long long routed = 0, kept = 0;
  for (int e = 0; e < E; ++e) {
    routed += out->counts[e];
    kept += out->kept[e];
  }
  out->stats[0] = static_cast<double>(routed);
  out->stats[1] = static_cast<double>(kept);
  out->stats[2] = static_cast<double>(S - kept);
  out->stats[3] = C;
  out->stats[4] = static_cast<double>(S - kept) / static_cast<double>(S);
  out->stats[5] = mo_balance_stat_form(E, T, k, out->counts, out->idx, out->w, c->lam, c->balance, c->gamma);
  out->stats[6] = nonfinite;
  out->stats[7] = mo_router_entropy(T, E, l.data());
  out->stats[8] = static_cast<double>(rerouted);
  return 0;
}

// ---------------------------------------------------------------------------
// backward (the training step): gradients of L = <dY, y> + B(I/T)
// ---------------------------------------------------------------------------

// Chain rule through one expert for n rows v [n,d] (stored in `dtype`) with
// upstream gradient g_out [n,d] (fp64): dv [n,d] and the forward output out
// [n,d] are written; the weight gradients are ADDED to dW1/dW3 [h,d], dW2
// [d,h], db1 [h], db2 [d] (null where the activation has none), so that a
// caller may sum several calls.  SwiGLU, hid = silu(a) b with a = W1 v and
// b = W3 v: dhid = W2^T g, da = dhid b silu'(a) with silu'(a) = s (1 + a (1 -
// s)), s = sigmoid(a), db = dhid silu(a).  GeLU, hid = gelu(z) with z = W1 v
// + b1: dz = dhid gelu'(z), gelu'(z) = Phi(z) + z phi(z).  Then dW2 += g
// hid^T, dW1 += da v^T (dz v^T), dW3 += db v^T, db1 += sum dz, db2 += sum g,
// dv = W1^T da + W3^T db (W1^T dz).  Sums in index order.
void mo_expert_ffn_backward(int n, int d, int h, int act, int dtype, const void* v, const double* g_out,
                            const void* W1, const void* W3, const void* b1, const void* W2, const void* b2,
                            double* dv, double* out, double* dW1, double* dW3, double* dW2, double* db1,
                            double* db2) {
  const long long nd = static_cast<long long>(n) * d, nh = static_cast<long long>(n) * h;
  std::vector<double> vr(nd), pre(nh), up(nh), hid(nh), dhid(nh, 0.0), w(static_cast<size_t>(d));
  for (long long i = 0; i < nd; ++i) vr[i] = rd(v, dtype, i);
  // forward: the pre-activations and hidden values of every row
  for (int u = 0; u < h; ++u) {
    for (int i = 0; i < d; ++i) w[i] = rd(W1, dtype, static_cast<long long>(u) * d + i);
    std::vector<double> w3(act == 1 ? d : 0);
    if (act == 1)
      for (int i = 0; i < d; ++i) w3[i] = rd(W3, dtype, static_cast<long long>(u) * d + i);
    for (int r = 0; r < n; ++r) {
      const double* vrow = vr.data() + static_cast<long long>(r) * d;
      double z = 0.0;
      for (int i = 0; i < d; ++i) z += w[i] * vrow[i];
      const long long o = static_cast<long long>(r) * h + u;
      if (act == 0) {
        if (b1) z += rd(b1, dtype, u);
        pre[o] = z;
        hid[o] = z * 0.5 * (1.0 + std::erf(z / std::sqrt(2.0)));
      } else {
        double g = 0.0;
        for (int i = 0; i < d; ++i) g += w3[i] * vrow[i];
        pre[o] = z;
        up[o] = g;
        hid[o] = z / (1.0 + std::exp(-z)) * g;
      }
    }
  }
  // the output, dW2 (db2) and the hidden gradient, one output column at a time
  for (int c = 0; c < d; ++c) {
    std::vector<double> w2(h);
    for (int u = 0; u < h; ++u) w2[u] = rd(W2, dtype, static_cast<long long>(c) * h + u);
    const double bias = (act == 0 && b2) ? rd(b2, dtype, c) : 0.0;
    for (int r = 0; r < n; ++r) {
      const double* hr = hid.data() + static_cast<long long>(r) * h;
      double o = 0.0;
      for (int u = 0; u < h; ++u) o += w2[u] * hr[u];
      out[static_cast<long long>(r) * d + c] = o + bias;
      const double g = g_out[static_cast<long long>(r) * d + c];
      double* dh = dhid.data() + static_cast<long long>(r) * h;
      for (int u = 0; u < h; ++u) {
        dW2[static_cast<long long>(c) * h + u] += g * hr[u];
        dh[u] += g * w2[u];
      }
      if (act == 0 && db2) db2[c] += g;
    }
  }
  // the pre-activation gradients, then dW1, dW3 (db1) and dv
  std::vector<double> da(nh), db(act == 1 ? nh : 0);
  for (long long o = 0; o < nh; ++o) {
    const double z = pre[o];
    if (act == 0) {
      const double pdf = std::exp(-0.5 * z * z) / std::sqrt(2.0 * std::acos(-1.0));
      da[o] = dhid[o] * (0.5 * (1.0 + std::erf(z / std::sqrt(2.0))) + z * pdf);
    } else {
      const double s = 1.0 / (1.0 + std::exp(-z));
      da[o] = dhid[o] * up[o] * s * (1.0 + z * (1.0 - s));
      db[o] = dhid[o] * z * s;
    }
  }
  for (long long i = 0; i < nd; ++i) dv[i] = 0.0;
  for (int u = 0; u < h; ++u) {
    for (int i = 0; i < d; ++i) w[i] = rd(W1, dtype, static_cast<long long>(u) * d + i);
    std::vector<double> w3(act == 1 ? d : 0);
    if (act == 1)
      for (int i = 0; i < d; ++i) w3[i] = rd(W3, dtype, static_cast<long long>(u) * d + i);
    for (int r = 0; r < n; ++r) {
      const long long o = static_cast<long long>(r) * h + u;
      const double* vrow = vr.data() + static_cast<long long>(r) * d;
      double* dvr = dv + static_cast<long long>(r) * d;
      for (int i = 0; i < d; ++i) {
        dW1[static_cast<long long>(u) * d + i] += da[o] * vrow[i];
        dvr[i] += da[o] * w[i];
      }
      if (act == 1) {
        for (int i = 0; i < d; ++i) {
          dW3[static_cast<long long>(u) * d + i] += db[o] * vrow[i];
          dvr[i] += db[o] * w3[i];
        }
      } else if (db1) {
        db1[u] += da[o];
      }
    }
  }
}

// The differentiable balance term on g = I/T, I[e] the sum of the routing
// weights of the slots routed to e before capacity (the importance of [P4]
// 2.2), in the form `variant` gives.  Returns B and writes dB/dw for every
// slot into dw [T,k] (0 for an unrouted slot); dg_e/dw = 1/T.
//   0, CV ([P1] 3.1 / 4.2): B = lambda std_{n-1}(g) / (mean(g) + 1e-8);
//      with dev = g - mean, dB/dg_e = lambda (dev_e / ((E-1) std) /
//      (mean + 1e-8) - std / (mean + 1e-8)^2 / E), the first term 0 when
//      std = 0.
//   1, std + max ([P2] 3.2): B = lambda (std_{n-1}(g) + gamma max(g));
//      dB/dg_e = lambda (dev_e / ((E-1) std) + gamma [e is the first
//      largest]).
//   2, switch ([P3] 2.3): B = lambda sum_e f_e g_e with f = counts / T the
//      usage fraction, a constant; dB/dg_e = lambda f_e.
double mo_balance_term_grad(int T, int k, int E, const int* idx, const double* w, double lam, int variant,
                            double gamma, double* dw) {
  std::vector<double> g(static_cast<size_t>(E), 0.0), f(static_cast<size_t>(E), 0.0), dB(static_cast<size_t>(E), 0.0);
  const long long S = static_cast<long long>(T) * k;
  for (long long s = 0; s < S; ++s)
    if (idx[s] >= 0) {
      g[idx[s]] += w[s];
      f[idx[s]] += 1.0;
    }
  for (int e = 0; e < E; ++e) {
    g[e] /= T;
    f[e] /= T;
  }
  double mean = 0.0, sd = 0.0;
  for (int e = 0; e < E; ++e) mean += g[e];
  mean /= E;
  if (E > 1) {
    double ss = 0.0;
    for (int e = 0; e < E; ++e) ss += (g[e] - mean) * (g[e] - mean);
    sd = std::sqrt(ss / (E - 1));
  }
  double val = 0.0;
  if (variant == 0) {
    if (E > 1) {
      const double m = mean + 1e-8;
      val = lam * sd / m;
      for (int e = 0; e < E; ++e)
        dB[e] = lam * ((sd > 0.0 ? (g[e] - mean) / ((E - 1) * sd) : 0.0) / m - sd / (m * m) / E);
    }
  } else if (variant == 1) {
    int top = 0;
    for (int e = 1; e < E; ++e)
      if (g[e] > g[top]) top = e;
    val = lam * (sd + gamma * g[top]);
    for (int e = 0; e < E; ++e) dB[e] = lam * (E > 1 && sd > 0.0 ? (g[e] - mean) / ((E - 1) * sd) : 0.0);
    dB[top] += lam * gamma;
  } else {
    for (int e = 0; e < E; ++e) {
      val += f[e] * g[e];
      dB[e] = lam * f[e];
    }
    val *= lam;
  }
  for (long long s = 0; s < S; ++s) dw[s] = idx[s] >= 0 ? dB[idx[s]] / T : 0.0;
  return val;
}

// Gradients of one layer, fp64.  dY [T,d] is stored in the config's dtype.
// Every pointer is caller-owned and fully written (zeroed first): dX [T,d],
// dWr [E,d], dW1/dW3 [E,h,d], dW2 [E,d,h], db1 [E,h], db2 [E,d] (GeLU), the
// shared expert's dWs1/dWs3 [h,d], dWs2 [d,h], dbs1 [h], dbs2 [d]; the
// logit gradient dl [T,E], y [T,d]; loss = <dY, y> + B and B.  Pointers for
// parts the configuration does not have may be null.
struct mo_grads {
  double *dX, *dWr, *dW1, *dW3, *dW2, *db1, *db2, *dWs1, *dWs3, *dWs2, *dbs1, *dbs2, *dl, *y;
  double loss, balance;
};

// The training step's backward with the routing of c->route (raw
// probabilities, token-major priority, a LayerNorm in front, rerouting)
// and the balance term of c->balance (mo_balance_term_grad):
//   per slot, G[t,j] = [kept] <dY[t], FFN_e(x[t])> + dB/dw[t,j];
//   dl[t, idx_j] = w_j (G_j - sum_j' w_j' G_j') (the softmax over the
//   selected logits), other logits 0;
//   dWr = dl^T x; dX = dl Wr + the experts' input gradients (a routed row's
//   upstream gradient is w_j dY[t]) + the shared expert's (upstream dY).
// Returns 0, or -1 on an invalid configuration.
int mo_layer_backward(const mo_config* c, const mo_inputs* in, const void* dY, mo_grads* g) {
  const int T = c->T, d = c->d, h = c->h, E = c->E, k = c->k, dt = c->dtype;
  if (T < 1 || d < 1 || h < 1 || E < 1 || k < 1 || k > E || (c->act != 0 && c->act != 1) ||
      (dt != MO_F32 && dt != MO_BF16) || c->balance < 0 || c->balance > 2 || (c->route & ~15))
    return -1;
  const long long S = static_cast<long long>(T) * k, Td = static_cast<long long>(T) * d;
  const int es = dt == MO_BF16 ? 2 : 4;
  // the forward's routing
  std::vector<double> l(static_cast<size_t>(T) * E), w(S);
  std::vector<int> idx(S), served(S);
  std::vector<long long> counts(E), kept(E), offsets(E + 1), pos(S);
  int C = 0;
  long long rerouted = 0;
  route_layer(c, in, l.data(), idx.data(), w.data(), counts.data(), kept.data(), offsets.data(), pos.data(),
              served.data(), &C, &rerouted);

  std::vector<double> dy(Td);
  for (long long i = 0; i < Td; ++i) dy[i] = rd(dY, dt, i);
  const auto zero = [](double* p, long long n) {
    if (p)
      for (long long i = 0; i < n; ++i) p[i] = 0.0;
  };
  const long long hd = static_cast<long long>(h) * d;
  zero(g->dX, Td);
  zero(g->dWr, static_cast<long long>(E) * d);
  zero(g->dW1, E * hd);
  zero(g->dW3, c->act == 1 ? E * hd : 0);
  zero(g->dW2, E * hd);
  zero(g->db1, c->act == 0 ? static_cast<long long>(E) * h : 0);
  zero(g->db2, c->act == 0 ? static_cast<long long>(E) * d : 0);
  zero(g->y, Td);
  zero(g->dl, static_cast<long long>(T) * E);
  std::vector<double> G(S, 0.0);
  const auto at = [&](const void* base, long long elems) -> const void* {
    return base ? static_cast<const char*>(base) + elems * es : nullptr;
  };
  // each expert over the slots it serves, in slot order (token, then
  // choice); a rerouted slot's output still carries its weight w_j, so its
  // logit gradient stays on idx_j
  for (int e = 0; e < E; ++e) {
    std::vector<long long> slots;
    for (long long s = 0; s < S; ++s)
      if (served[s] == e) slots.push_back(s);
    const int n = static_cast<int>(slots.size());
    if (n == 0) continue;
    std::vector<char> v(static_cast<size_t>(n) * d * es);
    std::vector<double> go(static_cast<size_t>(n) * d), dv(static_cast<size_t>(n) * d), out(static_cast<size_t>(n) * d);
    for (int r = 0; r < n; ++r) {
      const long long t = slots[r] / k;
      std::memcpy(v.data() + static_cast<long long>(r) * d * es, static_cast<const char*>(in->x) + t * d * es,
                  static_cast<size_t>(d) * es);
      for (int i = 0; i < d; ++i) go[static_cast<long long>(r) * d + i] = w[slots[r]] * dy[t * d + i];
    }
    mo_expert_ffn_backward(n, d, h, c->act, dt, v.data(), go.data(), at(in->W1, e * hd), at(in->W3, e * hd),
                           at(in->b1, static_cast<long long>(e) * h), at(in->W2, e * hd),
                           at(in->b2, static_cast<long long>(e) * d), dv.data(), out.data(), g->dW1 + e * hd,
                           c->act == 1 ? g->dW3 + e * hd : nullptr, g->dW2 + e * hd,
                           c->act == 0 && g->db1 ? g->db1 + static_cast<long long>(e) * h : nullptr,
                           c->act == 0 && g->db2 ? g->db2 + static_cast<long long>(e) * d : nullptr);
    for (int r = 0; r < n; ++r) {
      const long long s = slots[r], t = s / k;
      double dot = 0.0;
      for (int i = 0; i < d; ++i) {
        const double o = out[static_cast<long long>(r) * d + i];
        dot += dy[t * d + i] * o;
        g->y[t * d + i] += w[s] * o;
        g->dX[t * d + i] += dv[static_cast<long long>(r) * d + i];
      }
      G[s] += dot;
    }
  }
  if (c->has_shared) {
    const long long sh = static_cast<long long>(h) * d;
    zero(g->dWs1, sh);
    zero(g->dWs3, c->act == 1 ? sh : 0);
    zero(g->dWs2, sh);
    zero(g->dbs1, c->act == 0 ? h : 0);
    zero(g->dbs2, c->act == 0 ? d : 0);
    std::vector<double> dv(Td), out(Td);
    mo_expert_ffn_backward(T, d, h, c->act, dt, in->x, dy.data(), in->Ws1, in->Ws3, in->bs1, in->Ws2, in->bs2,
                           dv.data(), out.data(), g->dWs1, c->act == 1 ? g->dWs3 : nullptr, g->dWs2,
                           c->act == 0 ? g->dbs1 : nullptr, c->act == 0 ? g->dbs2 : nullptr);
    for (long long i = 0; i < Td; ++i) {
      g->dX[i] += dv[i];
      g->y[i] += out[i];
    }
  }
  std::vector<double> dB(S);
  const double B = mo_balance_term_grad(T, k, E, idx.data(), w.data(), c->lam, c->balance, c->gamma, dB.data());
  for (long long s = 0; s < S; ++s) G[s] += dB[s];
  // the logit gradient: the softmax over the selected logits, dl[t, idx_j]
  // = w_j (G_j - sum_j' w_j' G_j'); with raw probabilities (w_j = p_{idx_j}
  // of the softmax over all E) every logit e gets p_e ([e selected] G_e -
  // sum_j w_j G_j)
  const bool raw = (c->route & MO_RAW_PROBS) != 0;
  std::vector<double> p(static_cast<size_t>(E));
  for (int t = 0; t < T; ++t) {
    const long long s0 = static_cast<long long>(t) * k;
    if (idx[s0] < 0) continue;
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += w[s0 + j] * G[s0 + j];
    double* dlt = g->dl + static_cast<long long>(t) * E;
    if (raw) {
      const double* lt = l.data() + static_cast<long long>(t) * E;
      double z = 0.0;
      for (int e = 0; e < E; ++e) z += std::exp(lt[e] - lt[idx[s0]]);
      for (int e = 0; e < E; ++e) {
        p[e] = std::exp(lt[e] - lt[idx[s0]]) / z;
        dlt[e] = -p[e] * sum;
      }
      for (int j = 0; j < k; ++j) dlt[idx[s0 + j]] += p[idx[s0 + j]] * G[s0 + j];
    } else {
      for (int j = 0; j < k; ++j) dlt[idx[s0 + j]] += w[s0 + j] * (G[s0 + j] - sum);
    }
  }
  // dWr = dl^T xr and the router's part of dX, xr = x or (MO_LAYERNORM) its
  // layer-normed rows, whose backward the router's input gradient dl Wr
  // then goes through
  const bool ln = (c->route & MO_LAYERNORM) != 0;
  std::vector<double> xr(ln ? Td : 0), gr(ln ? Td : 0, 0.0);
  if (ln) mo_layer_norm(T, d, dt, in->x, xr.data());
  for (int e = 0; e < E; ++e) {
    for (int t = 0; t < T; ++t) {
      const double q = g->dl[static_cast<long long>(t) * E + e];
      if (q == 0.0) continue;
      double* dxr = ln ? gr.data() + static_cast<long long>(t) * d : g->dX + static_cast<long long>(t) * d;
      for (int i = 0; i < d; ++i) {
        const long long o = static_cast<long long>(t) * d + i;
        g->dWr[static_cast<long long>(e) * d + i] += q * (ln ? xr[o] : rd(in->x, dt, o));
        dxr[i] += q * rd(in->Wr, dt, static_cast<long long>(e) * d + i);
      }
    }
  }
  if (ln) mo_layer_norm_backward(T, d, dt, in->x, gr.data(), g->dX);
  double ly = 0.0;
  for (long long i = 0; i < Td; ++i) ly += dy[i] * g->y[i];
  g->balance = B;
  g->loss = ly + B;
  return 0;
}

}  // extern "C"

// C ABI of the sparse-MoE layer (declared and documented in include/moe.h).
// Argument checks, workspace carving and the launch sequence; every step of
// the computation runs in this library's kernels.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

moe_status validate(const moe_config* cfg) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (cfg->T < 1 || cfg->d < 1 || cfg->h < 1 || cfg->E < 1 || cfg->E > 1024) return MOE_ERR_INVALID_ARG;
  if (cfg->k < 1 || cfg->k > 8 || cfg->k > cfg->E) return MOE_ERR_INVALID_ARG;
  if (cfg->act != MOE_ACT_GELU && cfg->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype != MOE_F32 && cfg->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (cfg->min_capacity < 0 || !(cfg->capacity_factor == cfg->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(cfg->T) * cfg->k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  if (cfg->dtype == MOE_BF16 && ((cfg->d % 8) || (cfg->h % 8))) return MOE_ERR_UNSUPPORTED;
  if (cfg->route_flags & ~(MOE_ROUTE_RAW_PROBS | MOE_ROUTE_TOKEN_MAJOR | MOE_ROUTE_LAYERNORM | MOE_ROUTE_REROUTE))
    return MOE_ERR_INVALID_ARG;
  if ((cfg->route_flags & MOE_ROUTE_REROUTE) && cfg->k > 4) return MOE_ERR_UNSUPPORTED;
  if (cfg->balance < MOE_BALANCE_CV || cfg->balance > MOE_BALANCE_SWITCH) return MOE_ERR_INVALID_ARG;
  if (!(cfg->balance_gamma == cfg->balance_gamma) || isinf(cfg->balance_gamma)) return MOE_ERR_INVALID_ARG;
  if ((cfg->gemm_flags & ~(MOE_GEMM_CTA_PAIRS | MOE_GEMM_SINGLE_CTA)) ||
      ((cfg->gemm_flags & MOE_GEMM_CTA_PAIRS) && (cfg->gemm_flags & MOE_GEMM_SINGLE_CTA)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int capacity_of(const moe_config* cfg) {
  const float cf = cfg->capacity_factor;
  if (cf <= 0.f) return cfg->T;
  // ceil(cf*T*k/E) of the exact value: cf = m * 2^e with m a 24-bit
  // integer, so the quotient is a ratio of integers and the ceiling is
  // taken in 128-bit integer arithmetic, free of rounding.
  long long c;
  if (static_cast<double>(cf) * cfg->T * cfg->k / cfg->E >= 2147483647.0) {
    c = 2147483647LL;
  } else {
    int e2 = 0;
    const float fr = frexpf(cf, &e2);  // cf = fr * 2^e2, fr in [0.5, 1)
    const long long m = static_cast<long long>(ldexpf(fr, 24));
    const int e = e2 - 24;              // cf = m * 2^e exactly
    if (e < -100) {
      c = 1;  // 0 < cf*T*k/E < 2^30 * 2^24 * 2^-100 < 1
    } else {
      __int128 num = static_cast<__int128>(m) * cfg->T * cfg->k;
      __int128 den = cfg->E;
      if (e >= 0) num <<= e;
      else den <<= -e;
      c = static_cast<long long>((num + den - 1) / den);
    }
  }
  if (c < cfg->min_capacity) c = cfg->min_capacity;
  return static_cast<int>(c);
}

size_t esize(const moe_config* cfg) { return cfg->dtype == MOE_BF16 ? 2 : 4; }

// Workspace carving.  training 0/1 (forward): [header | dispatch scratch |
// (inference) intermediates | shared hidden].  training 2 (backward):
// [header | dYg | slot weights | weighted hidden rows (hi, lo) | dAB | dXp |
// dot | dl | importance | coef | router partials | shared dAB | LayerNorm
// terms | dense logit gradient].
struct WsLayout {
  size_t dispatch_off, route_off, ent, backup;
  size_t idx, w, counts, kept, offsets, pos, Xp, H, Yp, Sx, Hs;
  size_t dYg, wp, Hw, Hw_lo, dAB, dXp, dot, dl, imp, coef, rpart, dABs, lnc, dld;
  size_t total;
};

WsLayout layout(const moe_config* cfg, int training) {
  WsLayout L{};
  size_t o = kWsHeader;
  const size_t T = cfg->T, k = cfg->k, E = cfg->E, d = cfg->d, h = cfg->h, es = esize(cfg);
  const size_t hz = cfg->act == MOE_ACT_SWIGLU ? 2 * h : h;  // width of the pre-activation rows
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes, 256);
    return at;
  };
  if (training == 2) {
    L.dYg = take(T * k * d * es);
    L.wp = take(T * k * 4);
    L.Hw = take(T * k * h * es);
    L.Hw_lo = take(T * k * h * es);
    L.dAB = take(T * k * hz * es);
    L.dXp = take(T * k * d * 4);
    L.dot = take(T * k * 4);
    L.dl = take(T * k * 4);
    L.imp = take(E * 8);
    L.coef = take(E * 4);
    L.rpart = take(router_wgrad_partial_bytes(*cfg));
    L.dABs = cfg->has_shared ? take(T * hz * es) : 0;
    L.lnc = (cfg->route_flags & MOE_ROUTE_LAYERNORM) ? take(3 * T * 4) : 0;
    L.dld = (cfg->route_flags & MOE_ROUTE_RAW_PROBS) ? take(T * E * 4) : 0;
    L.total = o;
    return L;
  }
  L.dispatch_off = take(dispatch_ep_scratch_bytes(*cfg));  // also serves moe_dispatch_ep
  L.route_off = take(route_scratch_bytes(*cfg));
  L.ent = take(T * 4);
  L.imp = cfg->balance == MOE_BALANCE_SWITCH ? take(E * 8) : 0;
  L.backup = (cfg->route_flags & MOE_ROUTE_REROUTE) ? take(T * k * 4) : 0;
  if (!training) {
    L.idx = take(T * k * 4);
    L.w = take(T * k * 4);
    L.counts = take(E * 4);
    L.kept = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.pos = take(T * k * 4);
    L.Xp = take(T * k * d * es);
    L.H = take(T * k * h * es);
    L.Yp = take(T * k * d * es);
    L.Sx = cfg->has_shared ? take(T * d * es) : 0;
  }
  L.Hs = cfg->has_shared ? take(T * h * es) : 0;
  L.total = o;
  return L;
}

inline void* at(void* ws, size_t off) { return static_cast<uint8_t*>(ws) + off; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Shared expert riding along in the routed launches (bf16): its input rows,
// weights and outputs.
struct SharedFfn {
  const void* x;  // [T, d]
  const moe_weights* w;
  void* Hs;       // [T, h]
  void* Sx;       // [T, d]
  void* Zs;       // pre-activations, nullable
};

// Expert GEMM launches under this many FLOPs take CTA pair tiles by
// default: the small prefill's (9.5e10 and 4.7e10) gained 4%, the large
// prefill's (7.7e12 and 3.9e12) lost 10% (the four-expert profiling slice of
// the large prefill, 4.8e11 and 2.4e11, keeps the large prefill's tiles).
constexpr double kPairAutoFlops = 2e11;

moe_status run_ffn(const moe_config* cfg, const void* Xp, long long a_rows, const int* offsets, int G, int rows,
                   const void* W1, const void* W3, const void* b1, const void* W2, const void* b2, void* H,
                   void* Yp, void* Z, int* err, cudaStream_t st, const SharedFfn* sh = nullptr) {
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  GemmParams g1{};
  g1.offsets = offsets;
  g1.G = G;
  g1.rows = rows;
  g1.N = cfg->h;
  g1.K = cfg->d;
  g1.mode = swiglu ? kModeSwiGLU : kModeGeLU;
  g1.out = H;
  g1.zsave = Z;
  g1.ldz = swiglu ? 2LL * cfg->h : cfg->h;
  g1.bias = swiglu ? nullptr : b1;
  g1.err = err;
  g1.sched = err ? err + 1 : nullptr;
  // CTA pair tiles as gemm_flags asks, else for a launch short enough to
  // gain from them (see MOE_GEMM_CTA_PAIRS); each launch's FLOPs are counted
  // over every row it may run (the T k routed bound and the shared expert)
  const double launch_rows = static_cast<double>(a_rows) + (sh ? static_cast<double>(cfg->T) : 0.0);
  const double flops1 = 2.0 * launch_rows * cfg->d * (swiglu ? 2.0 * cfg->h : cfg->h);
  const double flops2 = 2.0 * launch_rows * cfg->d * cfg->h;
  auto pairs_for = [&](double flops) {
    if (cfg->gemm_flags & MOE_GEMM_CTA_PAIRS) return 1;
    if (cfg->gemm_flags & MOE_GEMM_SINGLE_CTA) return 0;
    return flops < kPairAutoFlops ? 1 : 0;
  };
  g1.cta_pairs = pairs_for(flops1);
  GemmParams g2 = g1;
  g2.cta_pairs = pairs_for(flops2);
  g2.N = cfg->d;
  g2.K = cfg->h;
  g2.mode = kModePlain;
  g2.out = Yp;
  g2.zsave = nullptr;
  g2.bias = swiglu ? nullptr : b2;
  moe_status s;
  if (cfg->dtype == MOE_BF16) {
    GemmExtra x1{}, x2{};
    if (sh) {
      // the shared expert is one more group of T rows in each launch
      g1.xrows = g2.xrows = cfg->T;
      g1.xout = sh->Hs;
      g1.xzsave = sh->Zs;
      g1.xbias = swiglu ? nullptr : sh->w->bs1;
      g2.xout = sh->Sx;
      g2.xbias = swiglu ? nullptr : sh->w->bs2;
      x1.A = sh->x;
      x1.B0 = sh->w->Ws1;
      x1.B1 = swiglu ? sh->w->Ws3 : nullptr;
      x2.A = sh->Hs;
      x2.B0 = sh->w->Ws2;
    }
    s = launch_grouped_gemm_tc(g1, kKindFwd, Xp, a_rows, W1, swiglu ? W3 : nullptr,
                               static_cast<long long>(G) * cfg->h, st, sh ? &x1 : nullptr);
    if (s != MOE_OK) return s;
    s = launch_grouped_gemm_tc(g2, kKindFwd, H, a_rows, W2, nullptr, static_cast<long long>(G) * cfg->d, st,
                               sh ? &x2 : nullptr);
  } else {
    if (Z || sh) return MOE_ERR_UNSUPPORTED;
    s = launch_grouped_gemm_f32(g1, Xp, a_rows, W1, swiglu ? W3 : nullptr, st);
    if (s != MOE_OK) return s;
    s = launch_grouped_gemm_f32(g2, H, a_rows, W2, nullptr, st);
  }
  return s;
}

// Backward of one expert group set (routed: G experts over offsets; shared:
// G = 1 over `rows` rows).  dYg [a_rows, d] holds the upstream gradient
// rows in expert order as stored, and wp [a_rows] each row's routing weight
// (nullable: 1), so the expert's upstream gradient is wp[r] * dYg[r].  Z:
// the saved fp32 pre-activations; Xin: the forward input rows.  The Dgrad
// epilogue leaves wp[r] * act(z[r]) in Hw + Hw_lo (scratch [a_rows, h] each:
// its bf16 rounding and the bf16 residual), and the W2 gradient contracts
// dYg with both, so that gradient carries no rounding of its operands
// beyond 2^-16.  Writes dAB (scratch), dXin (fp32, [a_rows, d]),
// dW1/dW3/dW2 (fp32) and, for GeLU, db1/db2.
moe_status run_ffn_bwd(const moe_config* cfg, long long a_rows, const int* offsets, int G, int rows,
                       const void* dYg, const float* wp, const float* Z, void* Hw, void* Hw_lo, const void* Xin,
                       const void* W1, const void* W3, const void* W2, void* dAB, float* dXin, float* dW1,
                       float* dW3, float* dW2, float* db1, float* db2, int* err, cudaStream_t st) {
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  const int h = cfg->h, d = cfg->d;
  const long long hz = swiglu ? 2LL * h : h;
  // dH = wp * (dYg . W2_g) -> activation backward -> dAB = [dA | dB] (or dZ)
  GemmParams a{};
  a.offsets = offsets;
  a.G = G;
  a.rows = rows;
  a.N = h;
  a.K = d;
  a.mode = swiglu ? kModeSwiGLUBwd : kModeGeLUBwd;
  a.out = dAB;
  a.ldo = hz;
  a.zin = Z;
  a.ldz = hz;
  a.row_scale = wp;
  a.hout = Hw;
  a.hout_lo = Hw_lo;
  a.err = err;
  a.sched = err ? err + 1 : nullptr;
  moe_status s = launch_grouped_gemm_tc(a, kKindDgrad, dYg, a_rows, W2, nullptr, static_cast<long long>(G) * d, st);
  if (s != MOE_OK) return s;
  // dXin = dA . W1_g + dB . W3_g  (fp32)
  GemmParams b{};
  b.offsets = offsets;
  b.G = G;
  b.rows = rows;
  b.N = d;
  b.K = static_cast<int>(hz);
  b.k_split = swiglu ? h : 0;
  b.mode = kModePlain;
  b.out_f32 = 1;
  b.out = dXin;
  b.err = err;
  b.sched = err ? err + 1 : nullptr;
  s = launch_grouped_gemm_tc(b, kKindDgrad, dAB, a_rows, W1, swiglu ? W3 : nullptr, static_cast<long long>(G) * h,
                             st);
  if (s != MOE_OK) return s;
  // dW2_g = dYg_g^T . (Hw + Hw_lo)_g, Hw + Hw_lo = wp * act(Z)
  GemmParams c{};
  c.offsets = offsets;
  c.G = G;
  c.rows = rows;
  c.M = d;
  c.N = h;
  c.mode = kModePlain;
  c.out_f32 = 1;
  c.out = dW2;
  c.b_lo = 1;
  c.err = err;
  c.sched = err ? err + 1 : nullptr;
  s = launch_grouped_gemm_tc(c, kKindWgrad, dYg, a_rows, Hw, Hw_lo, a_rows, st);
  if (s != MOE_OK) return s;
  // [dW1; dW3]_g = [dA | dB]_g^T . Xin_g
  GemmParams w{};
  w.offsets = offsets;
  w.G = G;
  w.rows = rows;
  w.M = static_cast<int>(hz);
  w.N = d;
  w.m_split = swiglu ? h : 0;
  w.mode = kModePlain;
  w.out_f32 = 1;
  w.out = dW1;
  w.out2 = swiglu ? dW3 : nullptr;
  w.err = err;
  w.sched = err ? err + 1 : nullptr;
  s = launch_grouped_gemm_tc(w, kKindWgrad, dAB, a_rows, Xin, nullptr, a_rows, st);
  if (s != MOE_OK) return s;
  if (!swiglu) {
    if (db1) {
      s = launch_group_colsum(dAB, hz, offsets, G, rows, h, nullptr, db1, st);
      if (s != MOE_OK) return s;
    }
    if (db2) {
      s = launch_group_colsum(dYg, d, offsets, G, rows, d, wp, db2, st);
      if (s != MOE_OK) return s;
    }
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_capacity(const moe_config* cfg, int* C_out) {
  const moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!C_out) return MOE_ERR_INVALID_ARG;
  *C_out = capacity_of(cfg);
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config* cfg, int training, size_t* bytes) {
  const moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  if (training < 0 || training > 2) return MOE_ERR_INVALID_ARG;
  *bytes = layout(cfg, training).total;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* Wr, const float* expert_bias,
                     const float* noise, int* idx, float* w, int* counts, float* entropy, void* ws,
                     moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!x || !Wr || !idx || !w || !counts) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wr) || (ws && !aligned16(ws))) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = layout(cfg, 1);
  void* scratch = ws && route_scratch_bytes(*cfg) ? at(ws, L.route_off) : nullptr;
  int* backup = ws && (cfg->route_flags & MOE_ROUTE_REROUTE) ? static_cast<int*>(at(ws, L.backup)) : nullptr;
  int* err = ws ? static_cast<int*>(ws) : nullptr;
  return launch_route(*cfg, x, Wr, expert_bias, noise, idx, w, counts, entropy, scratch, backup, nullptr, err, st);
}

moe_status moe_dispatch(const moe_config* cfg, const int* idx, const void* x, int* kept, int* offsets, int* pos,
                        void* Xp, moe_stats* stats, void* ws, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!idx || !x || !kept || !offsets || !pos || !Xp || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Xp) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(cfg, 1);
  const int* backup = (cfg->route_flags & MOE_ROUTE_REROUTE) ? static_cast<const int*>(at(ws, L.backup)) : nullptr;
  return launch_dispatch(*cfg, capacity_of(cfg), idx, x, kept, offsets, pos, Xp, stats, at(ws, L.dispatch_off),
                         backup,
                         reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_dispatch_static(const moe_config* cfg, const int* idx, const void* x, int* kept, int* offsets,
                               int* pos, void* Xp, moe_stats* stats, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!idx || !x || !kept || !offsets || !pos || !Xp) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Xp)) return MOE_ERR_INVALID_ARG;
  if (cfg->route_flags & MOE_ROUTE_REROUTE) return MOE_ERR_UNSUPPORTED;  // the backups live in a workspace
  void* scratch = nullptr;
  s = static_dispatch_scratch(dispatch_scratch_bytes(*cfg), &scratch);
  if (s != MOE_OK) return s;
  return launch_dispatch(*cfg, capacity_of(cfg), idx, x, kept, offsets, pos, Xp, stats, scratch, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_slot_counts(const moe_config* cfg, const int* idx, int* counts, moe_stream_t stream) {
  const moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!idx || !counts) return MOE_ERR_INVALID_ARG;
  return launch_slot_counts(*cfg, idx, counts, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_dispatch_ep(const moe_config* cfg, const int* idx, const void* x, const int* rank_adjust,
                           const int* send_adjust, int capacity, int* pos, void* Xsend, void* ws,
                           moe_stream_t stream) {
  const moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!idx || !x || !rank_adjust || !send_adjust || !pos || !ws || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (cfg->route_flags & (MOE_ROUTE_TOKEN_MAJOR | MOE_ROUTE_REROUTE)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(ws) || (Xsend && !aligned16(Xsend))) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(cfg, 1);
  return launch_dispatch_ep(*cfg, idx, x, rank_adjust, send_adjust, capacity, pos, Xsend, at(ws, L.dispatch_off),
                            reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_permute_rows(const void* src, const int* map, long long n, long long row_bytes, int scatter,
                            void* dst, moe_stream_t stream) {
  if (n < 0 || (n > 0 && (!src || !map || !dst))) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!aligned16(src) || !aligned16(dst))) return MOE_ERR_INVALID_ARG;
  return launch_permute_rows(src, map, n, row_bytes, scatter, dst, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* Xp, const int* offsets, const void* W1,
                          const void* W3, const void* b1, const void* W2, const void* b2, void* H, void* Yp,
                          void* ws, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  if (!Xp || !offsets || !W1 || !W2 || !H || !Yp || !ws || (swiglu && !W3)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Xp) || !aligned16(W1) || !aligned16(W2) || !aligned16(H) || !aligned16(Yp) ||
      (swiglu && !aligned16(W3)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  if (launch_zero(err, kWsZeroBytes, nullptr, 0, st) != MOE_OK) return MOE_ERR_CUDA;
  const long long a_rows = static_cast<long long>(cfg->T) * cfg->k;
  return run_ffn(cfg, Xp, a_rows, offsets, cfg->E, 0, W1, W3, b1, W2, b2, H, Yp, nullptr, err, st);
}

moe_status moe_expert_ffn_shared(const moe_config* cfg, const void* Xp, const int* offsets, const moe_weights* wts,
                                 void* H, void* Yp, const void* x, void* Hs, void* Sx, void* ws, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  if (!Xp || !offsets || !wts || !H || !Yp || !x || !Hs || !Sx || !ws) return MOE_ERR_INVALID_ARG;
  if (!wts->W1 || !wts->W2 || (swiglu && !wts->W3) || !wts->Ws1 || !wts->Ws2 || (swiglu && !wts->Ws3))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {Xp, H, Yp, x, Hs, Sx, wts->W1, wts->W2, wts->Ws1, wts->Ws2};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  if (launch_zero(err, kWsZeroBytes, nullptr, 0, st) != MOE_OK) return MOE_ERR_CUDA;
  const long long a_rows = static_cast<long long>(cfg->T) * cfg->k;
  SharedFfn sh{x, wts, Hs, Sx, nullptr};
  return run_ffn(cfg, Xp, a_rows, offsets, cfg->E, 0, wts->W1, wts->W3, wts->b1, wts->W2, wts->b2, H, Yp, nullptr,
                 err, st, &sh);
}

moe_status moe_combine(const moe_config* cfg, const void* Yp, const int* pos, const float* w, const void* Sx,
                       void* y, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!Yp || !pos || !w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Yp) || !aligned16(y) || (Sx && !aligned16(Sx))) return MOE_ERR_INVALID_ARG;
  return launch_combine(*cfg, Yp, pos, w, Sx, y, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_layer_fwd(const moe_config* cfg, const moe_weights* wts, const void* x, const float* noise, void* y,
                         moe_saved* saved, moe_stats* stats, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!wts || !x || !y || !ws || !wts->Wr || !wts->W1 || !wts->W2) return MOE_ERR_INVALID_ARG;
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  if (swiglu && !wts->W3) return MOE_ERR_INVALID_ARG;
  if (cfg->has_shared && (!wts->Ws1 || !wts->Ws2 || (swiglu && !wts->Ws3))) return MOE_ERR_INVALID_ARG;
  const int training = saved != nullptr;
  const WsLayout L = layout(cfg, training);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws) || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;

  moe_saved S;
  if (training) {
    S = *saved;
    if (!S.idx || !S.w || !S.counts || !S.kept || !S.offsets || !S.pos || !S.Xp || !S.H || !S.Yp ||
        (cfg->has_shared && !S.Sx))
      return MOE_ERR_INVALID_ARG;
  } else {
    S.idx = static_cast<int*>(at(ws, L.idx));
    S.w = static_cast<float*>(at(ws, L.w));
    S.counts = static_cast<int*>(at(ws, L.counts));
    S.kept = static_cast<int*>(at(ws, L.kept));
    S.offsets = static_cast<int*>(at(ws, L.offsets));
    S.pos = static_cast<int*>(at(ws, L.pos));
    S.Xp = at(ws, L.Xp);
    S.H = at(ws, L.H);
    S.Yp = at(ws, L.Yp);
    S.Sx = cfg->has_shared ? at(ws, L.Sx) : nullptr;
    S.Z = nullptr;
    S.Hs = nullptr;
    S.Zs = nullptr;
    S.logits = nullptr;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);  // zeroed by the router's first launch

  float* ent = stats ? static_cast<float*>(at(ws, L.ent)) : nullptr;
  int* backup = (cfg->route_flags & MOE_ROUTE_REROUTE) ? static_cast<int*>(at(ws, L.backup)) : nullptr;
  float* out_logits = training && cfg->dtype == MOE_BF16 ? S.logits : nullptr;
  s = launch_route(*cfg, x, wts->Wr, wts->expert_bias, noise, S.idx, S.w, S.counts, ent,
                   route_scratch_bytes(*cfg) ? at(ws, L.route_off) : nullptr, backup, out_logits, err, st);
  if (s != MOE_OK) return s;
  s = launch_dispatch(*cfg, capacity_of(cfg), S.idx, x, S.kept, S.offsets, S.pos, S.Xp, stats,
                      at(ws, L.dispatch_off), backup, st, ent);
  if (s != MOE_OK) return s;
  if (stats) {
    if (cfg->balance == MOE_BALANCE_SWITCH) {
      s = launch_balance_stat_switch(*cfg, S.idx, S.w, S.counts, static_cast<unsigned long long*>(at(ws, L.imp)),
                                     stats, st);
      if (s != MOE_OK) return s;
    }
  }
  const long long a_rows = static_cast<long long>(cfg->T) * cfg->k;
  if (cfg->has_shared && cfg->dtype == MOE_BF16) {
    // bf16: the shared expert runs inside the routed launches
    SharedFfn sh{x, wts, training && S.Hs ? S.Hs : at(ws, L.Hs), S.Sx, training ? S.Zs : nullptr};
    s = run_ffn(cfg, S.Xp, a_rows, S.offsets, cfg->E, 0, wts->W1, wts->W3, wts->b1, wts->W2, wts->b2, S.H, S.Yp,
                training ? S.Z : nullptr, err, st, &sh);
    if (s != MOE_OK) return s;
  } else {
    s = run_ffn(cfg, S.Xp, a_rows, S.offsets, cfg->E, 0, wts->W1, wts->W3, wts->b1, wts->W2, wts->b2, S.H, S.Yp,
                training ? S.Z : nullptr, err, st);
    if (s != MOE_OK) return s;
    if (cfg->has_shared) {
      void* Hs = training && S.Hs ? S.Hs : at(ws, L.Hs);
      s = run_ffn(cfg, x, cfg->T, nullptr, 1, cfg->T, wts->Ws1, wts->Ws3, wts->bs1, wts->Ws2, wts->bs2, Hs, S.Sx,
                  training ? S.Zs : nullptr, err, st);
      if (s != MOE_OK) return s;
    }
  }
  return launch_combine(*cfg, S.Yp, S.pos, S.w, cfg->has_shared ? S.Sx : nullptr, y, st);
}

moe_status moe_layer_bwd(const moe_config* cfg, const moe_weights* wts, const void* x, const moe_saved* saved,
                         const void* dY, const moe_grads* grads, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!wts || !x || !saved || !dY || !grads || !ws) return MOE_ERR_INVALID_ARG;
  const bool swiglu = cfg->act == MOE_ACT_SWIGLU;
  if (cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if ((cfg->d % 64) || (cfg->h % 64)) return MOE_ERR_UNSUPPORTED;
  const bool raw = (cfg->route_flags & MOE_ROUTE_RAW_PROBS) != 0;
  if (raw && (cfg->route_flags & MOE_ROUTE_LAYERNORM)) return MOE_ERR_UNSUPPORTED;
  if (!wts->Wr || !wts->W1 || !wts->W2 || (swiglu && !wts->W3)) return MOE_ERR_INVALID_ARG;
  if (cfg->has_shared && (!wts->Ws1 || !wts->Ws2 || (swiglu && !wts->Ws3))) return MOE_ERR_INVALID_ARG;
  const moe_saved& S = *saved;
  if (!S.idx || !S.w || !S.offsets || !S.pos || !S.Xp || !S.Yp || !S.Z) return MOE_ERR_INVALID_ARG;
  if (raw && !S.logits) return MOE_ERR_INVALID_ARG;
  if (cfg->has_shared && !S.Zs) return MOE_ERR_INVALID_ARG;
  const moe_grads& g = *grads;
  if (!g.dX || !g.dWr || !g.dW1 || !g.dW2 || (swiglu && !g.dW3)) return MOE_ERR_INVALID_ARG;
  if (cfg->has_shared && (!g.dWs1 || !g.dWs2 || (swiglu && !g.dWs3))) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(cfg, 2);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws) || !aligned16(x) || !aligned16(dY) || !aligned16(g.dX)) return MOE_ERR_INVALID_ARG;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  s = launch_zero(err, kWsZeroBytes, at(ws, L.imp), sizeof(unsigned long long) * cfg->E, st);
  if (s != MOE_OK) return s;
  void* dYg = at(ws, L.dYg);
  float* wp = static_cast<float*>(at(ws, L.wp));
  void* dAB = at(ws, L.dAB);
  float* dXp = static_cast<float*>(at(ws, L.dXp));
  float* dot = static_cast<float*>(at(ws, L.dot));
  float* dl = static_cast<float*>(at(ws, L.dl));
  const long long a_rows = static_cast<long long>(cfg->T) * cfg->k;

  // routing-weight gradients and the router
  s = launch_bwd_gather(*cfg, dY, S.Yp, S.pos, S.w, dYg, wp, dot, st);
  if (s != MOE_OK) return s;
  float* lnc = (cfg->route_flags & MOE_ROUTE_LAYERNORM) ? static_cast<float*>(at(ws, L.lnc)) : nullptr;
  if (cfg->balance == MOE_BALANCE_SWITCH && !S.counts) return MOE_ERR_INVALID_ARG;
  s = launch_router_bwd(*cfg, x, wts->Wr, S.idx, S.w, S.counts, dot,
                        static_cast<unsigned long long*>(at(ws, L.imp)), static_cast<float*>(at(ws, L.coef)), dl,
                        lnc, st);
  if (s != MOE_OK) return s;
  if (raw) {
    // every logit has a gradient: dl becomes the dense [T, E] matrix
    float* dld = static_cast<float*>(at(ws, L.dld));
    s = launch_router_bwd_raw(*cfg, S.logits, S.idx, S.w, dot, static_cast<float*>(at(ws, L.coef)), dld, st);
    if (s != MOE_OK) return s;
    dl = dld;
  }
  s = launch_router_wgrad(*cfg, x, S.idx, dl, lnc, static_cast<float*>(at(ws, L.rpart)), g.dWr, st);
  if (s != MOE_OK) return s;
  // routed experts
  s = run_ffn_bwd(cfg, a_rows, S.offsets, cfg->E, 0, dYg, wp, S.Z, at(ws, L.Hw), at(ws, L.Hw_lo), S.Xp, wts->W1,
                  wts->W3, wts->W2, dAB, dXp, g.dW1, g.dW3, g.dW2, g.db1, g.db2, err, st);
  if (s != MOE_OK) return s;
  // shared expert: its input gradient lands in dX directly (its weighted
  // hidden rows reuse the routed experts' scratch, T <= T*k rows, after the
  // routed launches on the same stream)
  if (cfg->has_shared) {
    s = run_ffn_bwd(cfg, cfg->T, nullptr, 1, cfg->T, dY, nullptr, S.Zs, at(ws, L.Hw), at(ws, L.Hw_lo), x, wts->Ws1,
                    wts->Ws3, wts->Ws2, at(ws, L.dABs), g.dX, g.dWs1, g.dWs3, g.dWs2, g.dbs1, g.dbs2, err, st);
    if (s != MOE_OK) return s;
  }
  return launch_bwd_dx(*cfg, dXp, S.pos, S.idx, dl, wts->Wr, x, lnc, cfg->has_shared ? 1 : 0, g.dX, st);
}

moe_status moe_check_error(const void* ws, int* code_out, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (code_out) *code_out = code;
  return code ? MOE_ERR_TIMEOUT : MOE_OK;
}

moe_status moe_selftest_wait_timeout(void* ws, moe_stream_t stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  return launch_selftest_wait(static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream));
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or type";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
  }
  return "unknown status";
}

}  // extern "C"

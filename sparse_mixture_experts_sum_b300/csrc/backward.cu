// Backward of the MoE layer outside the expert GEMMs: the gather of the
// upstream gradient into expert order, the routing-weight and router
// gradients (with the load-balance term), the router weight gradient, the
// GeLU bias gradients, and the assembly of dX.
//
// Loss: L = <dY, y> + B(I / T), I[e] = the sum of the routing weights of
// the slots routed to e -- the importance of [P4] "GPT-4 has 1.8 trillion
// parameters..." 2.2 -- and B the balance term: lambda * CV in the std/mean
// form of [P1] "'More parameters is better' is not the story..." 3.1 (std
// with n-1, +1e-8 on the mean), or lambda * (std + gamma * max) ([P2] 3.2),
// or lambda * sum_e (counts_e / T) g_e ([P3] 2.3).  Gradients flow back to
// the router and to the experts that served the slots ([P1] 3.3).  Per slot
// (t, j) routed to e:
//   dot[t,j] = <dY[t], Yp[pos[t,j]]>          (kept slots; 0 when dropped)
//   G[t,j]   = dot[t,j] + dB/dw[t,j]
//   dl[t,j]  = w[t,j] (G[t,j] - sum_j' w[t,j'] G[t,j'])   (softmax over the
//              selected logits, [P1] 3.3; the other logits get no gradient)
//   dWr[e]  += dl[t,j] x[t];   dX[t] += dl[t,j] Wr[e]
// With raw softmax weights (w_j = p_{idx_j} over all E) every logit gets
// p_e ([e selected] G_e - sum_j w_j G_j), and dWr, dX take that dense
// [T, E] gradient.
// Every reduction runs in a fixed order or in integers, so the results are
// the same bits on every run.
//
// LayerNorm before the router ([P2] "MoE mixture-of-experts architecture:
// principles and engineering practice" 5.2):
// the router saw n_t = r_t (x_t - mu_t).  Then dWr[e] += dl[t,j] n_t, and
// with g_t = sum_j dl[t,j] Wr[e_j] the input gradient is the normalisation's
// backward r_t (g - mean(g) - n_t mean(g n_t)).  Writing dl' = r_t dl,
// S_e = sum_i Wr[e,i], D_j = Wr[e_j] . (x_t - mu_t):
//   dX[t] += sum_j dl'_j Wr[e_j] - A_t - B_t (x_t - mu_t),
//   A_t = sum_j dl'_j S_{e_j} / d,  B_t = r_t^2 sum_j dl'_j D_j / d,
//   dWr[e] += dl'[t,j] (x_t - mu_t).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr double kImpScale = 4294967296.0;  // routing weights accumulate as 2^-32 fixed point
constexpr int MAXK_BWD = 8;                  // largest k

// One warp per token: dot[t,j] = <dY[t], Yp[pos]>, dYg[pos] = dY[t] (the
// stored bits: the routing weight is applied in fp32 by the expert GEMMs'
// epilogue, not folded into a rounded copy), wp[pos] = w[t,j].  KM = k
// rounded up to 2, 4 or 8 sizes the per-slot register arrays.
template <int KM>
__global__ void bwd_gather_kernel(const uint4* __restrict__ dY, const uint4* __restrict__ Yp,
                                  const int* __restrict__ pos, const float* __restrict__ w, int T, int k,
                                  int vec_per_row, uint4* __restrict__ dYg, float* __restrict__ wp,
                                  float* __restrict__ dot) {
  pdl_entry();
  const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int p[KM];
  float wt[KM], acc[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    p[j] = j < k ? pos[static_cast<size_t>(t) * k + j] : -1;
    wt[j] = j < k ? w[static_cast<size_t>(t) * k + j] : 0.f;
    acc[j] = 0.f;
  }
  for (int v = lane; v < vec_per_row; v += 32) {
    const uint4 q = dY[static_cast<size_t>(t) * vec_per_row + v];
    const uint32_t g[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (p[j] < 0) continue;
      const uint4 yq = Yp[static_cast<size_t>(p[j]) * vec_per_row + v];
      const uint32_t y[4] = {yq.x, yq.y, yq.z, yq.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[j] = fmaf(bf16lo(g[i]), bf16lo(y[i]), acc[j]);
        acc[j] = fmaf(bf16hi(g[i]), bf16hi(y[i]), acc[j]);
      }
      dYg[static_cast<size_t>(p[j]) * vec_per_row + v] = q;
    }
  }
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    float s = acc[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0 && j < k) {
      dot[static_cast<size_t>(t) * k + j] = p[j] >= 0 ? s : 0.f;
      if (p[j] >= 0) wp[p[j]] = wt[j];
    }
  }
}

// I[e] = sum of w over the slots routed to e, in 2^-32 fixed point (integer
// sums are exact, so the order of the atomics does not show).
__global__ void importance_kernel(const int* __restrict__ idx, const float* __restrict__ w, long long nslots, int E,
                                  unsigned long long* __restrict__ imp) {
  pdl_entry();
  extern __shared__ unsigned long long simp[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) simp[e] = 0ull;
  __syncthreads();
  for (long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; s < nslots;
       s += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = idx[s];
    if (e >= 0 && e < E) {
      const unsigned long long q = static_cast<unsigned long long>(static_cast<double>(w[s]) * kImpScale + 0.5);
      atomicAdd(&simp[e], q);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (simp[e]) atomicAdd(&imp[e], simp[e]);
}

// coef[e] = dB/dI[e] of the balance term B on g = I/T (fp64, fixed-order
// reductions; one block of 1024 threads, thread e owns expert e):
//   CV:      lambda * (dstd_e / (m + 1e-8) - std / (m + 1e-8)^2 / E) / T
//   STD_MAX: lambda * (dstd_e + gamma [e = lowest-index argmax of I]) / T
//   SWITCH:  lambda * (counts[e] / T) / T
// with m the mean of g and dstd_e = (g_e - m) / ((E - 1) std).
__global__ void __launch_bounds__(1024) balance_coef_kernel(const unsigned long long* __restrict__ imp,
                                                            const int* __restrict__ counts, int E, int T, float lam,
                                                            int variant, float gamma, float* __restrict__ coef) {
  pdl_entry();
  __shared__ double red[32];
  __shared__ unsigned long long rmax[32];
  __shared__ int rarg[32];
  __shared__ double mean_s, std_s;
  __shared__ int amax_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const double scale = 1.0 / (kImpScale * static_cast<double>(T));
  const unsigned long long my = tid < E ? imp[tid] : 0ull;
  const double fe = static_cast<double>(my) * scale;
  double v = fe;
  unsigned long long mx = my;
  int arg = tid < E ? tid : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v += __shfl_xor_sync(0xffffffffu, v, o);
    const unsigned long long omx = __shfl_xor_sync(0xffffffffu, mx, o);
    const int oarg = __shfl_xor_sync(0xffffffffu, arg, o);
    if (omx > mx || (omx == mx && oarg < arg)) {
      mx = omx;
      arg = oarg;
    }
  }
  if (lane == 0) {
    red[warp] = v;
    rmax[warp] = mx;
    rarg[warp] = arg;
  }
  __syncthreads();
  if (tid == 0) {
    double m = 0.0;
    unsigned long long bm = 0ull;
    int ba = 0x7fffffff;
    for (int w2 = 0; w2 < nwarps; ++w2) {
      m += red[w2];
      if (rmax[w2] > bm || (rmax[w2] == bm && rarg[w2] < ba)) {
        bm = rmax[w2];
        ba = rarg[w2];
      }
    }
    mean_s = m / E;
    amax_s = ba;
  }
  __syncthreads();
  const double m = mean_s;
  double dv2 = tid < E ? (fe - m) * (fe - m) : 0.0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dv2 += __shfl_xor_sync(0xffffffffu, dv2, o);
  __syncthreads();
  if (lane == 0) red[warp] = dv2;
  __syncthreads();
  if (tid == 0) {
    double var = 0.0;
    for (int w2 = 0; w2 < nwarps; ++w2) var += red[w2];
    std_s = E > 1 ? sqrt(var / (E - 1)) : 0.0;
  }
  __syncthreads();
  if (tid < E) {
    const double sd = std_s, den = m + 1e-8;
    const double dstd = (E > 1 && sd > 0.0) ? (fe - m) / ((E - 1) * sd) : 0.0;
    double g = 0.0;
    if (variant == MOE_BALANCE_STD_MAX) {
      g = static_cast<double>(lam) * (dstd + (tid == amax_s ? static_cast<double>(gamma) : 0.0));
    } else if (variant == MOE_BALANCE_SWITCH) {
      g = static_cast<double>(lam) * static_cast<double>(counts[tid]) / T;
    } else if (E > 1 && sd > 0.0) {
      g = static_cast<double>(lam) * (dstd / den - sd / (den * den) / E);
    }
    coef[tid] = static_cast<float>(g / T);
  }
}

// stats->balance_stat = lambda * sum_e (counts[e] / T) (I[e] / T), fp64, warps
// in order (one block of 1024 threads).
__global__ void __launch_bounds__(1024) balance_switch_stat_kernel(const unsigned long long* __restrict__ imp,
                                                                   const int* __restrict__ counts, int E, int T,
                                                                   float lam, moe_stats* __restrict__ stats) {
  pdl_entry();
  __shared__ double red[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const double invT = 1.0 / static_cast<double>(T);
  double v = tid < E ? static_cast<double>(counts[tid]) * invT * (static_cast<double>(imp[tid]) / kImpScale * invT)
                     : 0.0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w2 = 0; w2 < (blockDim.x >> 5); ++w2) s += red[w2];
    stats->balance_stat = static_cast<double>(lam) * s;
  }
}

// One thread per token: dl[t,j] = w_j (G_j - sum_j' w_j' G_j').
__global__ void router_bwd_kernel(const int* __restrict__ idx, const float* __restrict__ w,
                                  const float* __restrict__ dot, const float* __restrict__ coef, int T, int k, int E,
                                  float* __restrict__ dl) {
  pdl_entry();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float G[8], wt[8];
  float s = 0.f;
  const bool routed = idx[static_cast<size_t>(t) * k] >= 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    G[j] = 0.f;
    wt[j] = 0.f;
    if (j < k && routed) {
      const int e = idx[static_cast<size_t>(t) * k + j];
      wt[j] = w[static_cast<size_t>(t) * k + j];
      G[j] = dot[static_cast<size_t>(t) * k + j] + (e >= 0 && e < E ? coef[e] : 0.f);
      s = fmaf(wt[j], G[j], s);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < k) dl[static_cast<size_t>(t) * k + j] = routed ? wt[j] * (G[j] - s) : 0.f;
}

// LayerNorm before the router, one warp per token (after router_bwd_kernel):
// mu_t, r_t from two passes over x_t (the second also takes D_j and S_j
// against the k chosen router rows), then dl[t,:] *= r_t and
// lnc = {mu[T], A[T], B[T]}.
__global__ void ln_router_bwd_kernel(const bf16* __restrict__ x, const bf16* __restrict__ Wr,
                                     const int* __restrict__ idx, int T, int d, int k, int E, float* __restrict__ dl,
                                     float* __restrict__ lnc) {
  pdl_entry();
  const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const uint4* xv = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  const int nv = d >> 3;
  float s = 0.f;
  for (int i = lane; i < nv; i += 32) {
    const uint4 q = xv[i];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) s += bf16lo(u[c]) + bf16hi(u[c]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mu = s / static_cast<float>(d);
  int e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    e[j] = j < k ? idx[static_cast<size_t>(t) * k + j] : -1;
    if (e[j] >= E) e[j] = -1;
  }
  float q2 = 0.f, D[8], Sj[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) D[j] = Sj[j] = 0.f;
  for (int i = lane; i < nv; i += 32) {
    const uint4 q = xv[i];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
    float xc[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      xc[2 * c] = bf16lo(u[c]) - mu;
      xc[2 * c + 1] = bf16hi(u[c]) - mu;
      q2 = fmaf(xc[2 * c], xc[2 * c], fmaf(xc[2 * c + 1], xc[2 * c + 1], q2));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (e[j] < 0) continue;
      const uint4 wq = reinterpret_cast<const uint4*>(Wr + static_cast<size_t>(e[j]) * d)[i];
      const uint32_t wu[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float w0 = bf16lo(wu[c]), w1 = bf16hi(wu[c]);
        D[j] = fmaf(w0, xc[2 * c], fmaf(w1, xc[2 * c + 1], D[j]));
        Sj[j] += w0 + w1;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    q2 += __shfl_xor_sync(0xffffffffu, q2, o);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      D[j] += __shfl_xor_sync(0xffffffffu, D[j], o);
      Sj[j] += __shfl_xor_sync(0xffffffffu, Sj[j], o);
    }
  }
  if (lane != 0) return;
  const float inv_d = 1.0f / static_cast<float>(d);
  const float r = 1.0f / sqrtf(q2 * inv_d + 1e-5f);
  float A = 0.f, B = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      const float g = r * dl[static_cast<size_t>(t) * k + j];
      dl[static_cast<size_t>(t) * k + j] = g;
      if (e[j] >= 0) {
        A = fmaf(g, Sj[j], A);
        B = fmaf(g, D[j], B);
      }
    }
  }
  lnc[t] = mu;
  lnc[static_cast<size_t>(T) + t] = A * inv_d;
  lnc[2 * static_cast<size_t>(T) + t] = B * r * r * inv_d;
}

// Raw softmax weights (w_j = p_{idx_j}, p the softmax over all E experts):
// every logit gets a gradient, dlD[t,e] = p_e ([e selected] G_e - s), with
// G_j = dot[t,j] + coef[idx_j] and s = sum_j w_j G_j.  One warp per token;
// p from the forward's saved logits (one warp max, then exp(l - m) / Z).
template <int NV>
__global__ void router_bwd_raw_kernel(const float* __restrict__ logits, const int* __restrict__ idx,
                                      const float* __restrict__ w, const float* __restrict__ dot,
                                      const float* __restrict__ coef, int T, int k, int E, float* __restrict__ dlD) {
  pdl_entry();
  const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float* out = dlD + static_cast<size_t>(t) * E;
  if (idx[static_cast<size_t>(t) * k] < 0) {  // routed nowhere: no gradient
    for (int e = lane; e < E; e += 32) out[e] = 0.f;
    return;
  }
  int ej = -1;
  float gj = 0.f, sp = 0.f;
  if (lane < k) {
    ej = idx[static_cast<size_t>(t) * k + lane];
    gj = dot[static_cast<size_t>(t) * k + lane] + (ej >= 0 && ej < E ? coef[ej] : 0.f);
    sp = w[static_cast<size_t>(t) * k + lane] * gj;
  }
  // s = sum_j w_j G_j in slot order (every lane forms the same sum)
  float s = 0.f;
  int es[MAXK_BWD];
  float gs[MAXK_BWD];
#pragma unroll
  for (int j = 0; j < MAXK_BWD; ++j) {
    es[j] = __shfl_sync(0xffffffffu, ej, j);
    gs[j] = __shfl_sync(0xffffffffu, gj, j);
    const float pj = __shfl_sync(0xffffffffu, sp, j);
    if (j < k) s += pj;
  }
  float v[NV];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? logits[static_cast<size_t>(t) * E + e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (lane + 32 * i < E) z += expf(v[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float inv = 1.0f / z;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      float g = -s;
#pragma unroll
      for (int j = 0; j < MAXK_BWD; ++j)
        if (j < k && es[j] == e) g += gs[j];
      out[e] = expf(v[i] - m) * inv * g;
    }
  }
}

constexpr int RW_TOK = 512;   // tokens per block of the router weight gradient
constexpr int RW_EXP = 16;    // experts per block
constexpr int RW_WARPS = 4;
constexpr int RW_COLS = 256;  // columns per block: 8 per lane, one 16-byte load per token row

// partial[chunk][e][c] = sum over the chunk's tokens (each warp takes every
// RW_WARPS-th token, ascending) of sum_j [idx=e] dl[t,j] (x[t][c] - mu[t])
// (mu nullable: 0); DENSE: of dlD[t][e] x[t][c] for every expert e.  A block
// covers 256 columns (a lane owns 8 consecutive ones: one 16-byte load of a
// bf16 row) and 16 experts; every warp accumulates privately in shared
// memory, laid out acc[warp][e][q][lane] (column lane*8+q) so that a warp's
// updates hit 32 distinct banks; the warps are summed in a fixed order.
template <typename Tx, bool DENSE>
__global__ void __launch_bounds__(RW_WARPS * 32)
router_wgrad_partial_kernel(const Tx* __restrict__ x, const int* __restrict__ idx, const float* __restrict__ dl,
                            int T, int d, int k, int E, const float* __restrict__ mu,
                            float* __restrict__ partial) {
  pdl_entry();
  extern __shared__ float acc_s[];  // [RW_WARPS][RW_EXP][8][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* acc = acc_s + warp * (RW_EXP * 8 * 32);
  const int c0 = blockIdx.y * RW_COLS + lane * 8;
  const int e0 = blockIdx.z * RW_EXP;
  const int t0 = blockIdx.x * RW_TOK;
  for (int i = lane; i < RW_EXP * 8 * 32; i += 32) acc[i] = 0.f;
  __syncwarp();
  const int t1 = min(T, t0 + RW_TOK);
  constexpr int U = 4;  // token rows in flight per warp
  for (int tb = t0 + warp; tb < t1; tb += U * RW_WARPS) {
    float xv[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tb + u * RW_WARPS;
      if constexpr (sizeof(Tx) == 2) {
        uint4 q4 = make_uint4(0, 0, 0, 0);
        if (t < t1 && c0 + 8 <= d) q4 = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + c0);
        const uint32_t wv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xv[u][2 * i] = bf16lo(wv[i]);
          xv[u][2 * i + 1] = bf16hi(wv[i]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          xv[u][q] = (t < t1 && c0 + q < d) ? x[static_cast<size_t>(t) * d + c0 + q] : 0.f;
      }
      if (mu && t < t1) {
        const float m = mu[t];
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[u][q] -= m;
      }
    }
    if constexpr (DENSE) {
      // dl is [T, E]: lane e < RW_EXP fetches the chunk's expert e of each token
      float gu[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = tb + u * RW_WARPS;
        gu[u] = (t < t1 && lane < RW_EXP && e0 + lane < E) ? dl[static_cast<size_t>(t) * E + e0 + lane] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int e = 0; e < RW_EXP; ++e) {
          const float g = __shfl_sync(0xffffffffu, gu[u], e);
          if (e0 + e < E) {
            float* a = acc + e * 256 + lane;
#pragma unroll
            for (int q = 0; q < 8; ++q) a[q * 32] = fmaf(g, xv[u][q], a[q * 32]);
          }
        }
      }
    } else {
      // the slots' experts and logit gradients, loaded with the rows (lane j
      // of the warp fetches slot j of each token and shares it)
      int eu[U];
      float gu[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = tb + u * RW_WARPS;
        eu[u] = -1;
        gu[u] = 0.f;
        if (t < t1 && lane < k) {
          eu[u] = idx[static_cast<size_t>(t) * k + lane] - e0;
          gu[u] = dl[static_cast<size_t>(t) * k + lane];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        for (int j = 0; j < k; ++j) {
          const int e = __shfl_sync(0xffffffffu, eu[u], j);
          const float g = __shfl_sync(0xffffffffu, gu[u], j);
          if (e >= 0 && e < RW_EXP && e0 + e < E) {
            float* a = acc + e * 256 + lane;
#pragma unroll
            for (int q = 0; q < 8; ++q) a[q * 32] = fmaf(g, xv[u][q], a[q * 32]);
          }
        }
      }
    }
  }
  __syncthreads();
  const int ne = min(RW_EXP, E - e0);
  for (int i = threadIdx.x; i < ne * RW_COLS; i += blockDim.x) {
    const int e = i / RW_COLS, c = i - e * RW_COLS;
    const int cc = blockIdx.y * RW_COLS + c;
    const int off = e * 256 + (c & 7) * 32 + (c >> 3);
    float s = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < RW_WARPS; ++w2) s += acc_s[w2 * (RW_EXP * 8 * 32) + off];
    if (cc < d) partial[(static_cast<size_t>(blockIdx.x) * E + e0 + e) * d + cc] = s;
  }
}

// dWr[e][c] = sum over chunks (ascending) of partial[chunk][e][c].
__global__ void router_wgrad_reduce_kernel(const float* __restrict__ partial, int nchunks, long long Ed,
                                           float* __restrict__ dWr) {
  pdl_entry();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= Ed) return;
  float s = 0.f;
  for (int b = 0; b < nchunks; ++b) s += partial[static_cast<size_t>(b) * Ed + i];
  dWr[i] = s;
}

// One warp per token: dX[t] (+)= sum_{kept j} dXp[pos] + sum_j dl[t,j] Wr[idx_j] (fp32, j ascending)
// (- A_t - B_t (x[t] - mu_t) with LayerNorm before the router: LN, lnc).
// DENSE (raw softmax weights): dl is [T, E] and the router term is
// sum_e dl[t,e] Wr[e], e ascending.  KM = k rounded up to 2, 4 or 8 sizes
// the per-slot register arrays.
template <typename Tw, int KM, bool LN, bool DENSE>
__global__ void bwd_dx_kernel(const float* __restrict__ dXp, const int* __restrict__ pos, const int* __restrict__ idx,
                              const float* __restrict__ dl, const Tw* __restrict__ Wr, int T, int k, int d, int E,
                              const Tw* __restrict__ x, const float* __restrict__ lnc, int accumulate,
                              float* __restrict__ dX) {
  pdl_entry();
  const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int p[KM], e[KM];
  float g[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    p[j] = j < k ? pos[static_cast<size_t>(t) * k + j] : -1;
    e[j] = (!DENSE && j < k) ? idx[static_cast<size_t>(t) * k + j] : -1;
    g[j] = (!DENSE && j < k) ? dl[static_cast<size_t>(t) * k + j] : 0.f;
  }
  float* out = dX + static_cast<size_t>(t) * d;
  float lmu = 0.f, lA = 0.f, lB = 0.f;
  if (LN) {
    lmu = lnc[t];
    lA = lnc[static_cast<size_t>(T) + t];
    lB = lnc[2 * static_cast<size_t>(T) + t];
  }
#pragma unroll 4
  for (int c = lane * 4; c < d; c += 128) {
    float4 a = accumulate ? *reinterpret_cast<const float4*>(out + c) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (p[j] >= 0) {
        const float4 v = *reinterpret_cast<const float4*>(dXp + static_cast<size_t>(p[j]) * d + c);
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
      }
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (e[j] >= 0 && e[j] < E) {
        const Tw* wr = Wr + static_cast<size_t>(e[j]) * d + c;
        float w0, w1, w2, w3;
        if constexpr (sizeof(Tw) == 2) {
          w0 = __bfloat162float(wr[0]);
          w1 = __bfloat162float(wr[1]);
          w2 = __bfloat162float(wr[2]);
          w3 = __bfloat162float(wr[3]);
        } else {
          w0 = wr[0];
          w1 = wr[1];
          w2 = wr[2];
          w3 = wr[3];
        }
        a.x = fmaf(g[j], w0, a.x);
        a.y = fmaf(g[j], w1, a.y);
        a.z = fmaf(g[j], w2, a.z);
        a.w = fmaf(g[j], w3, a.w);
      }
    }
    if (DENSE) {
      const float* gl = dl + static_cast<size_t>(t) * E;
      for (int ee = 0; ee < E; ++ee) {
        const float gg = gl[ee];
        const Tw* wr = Wr + static_cast<size_t>(ee) * d + c;
        float w0, w1, w2, w3;
        if constexpr (sizeof(Tw) == 2) {
          w0 = __bfloat162float(wr[0]);
          w1 = __bfloat162float(wr[1]);
          w2 = __bfloat162float(wr[2]);
          w3 = __bfloat162float(wr[3]);
        } else {
          w0 = wr[0];
          w1 = wr[1];
          w2 = wr[2];
          w3 = wr[3];
        }
        a.x = fmaf(gg, w0, a.x);
        a.y = fmaf(gg, w1, a.y);
        a.z = fmaf(gg, w2, a.z);
        a.w = fmaf(gg, w3, a.w);
      }
    }
    if (LN) {
      const Tw* xr = x + static_cast<size_t>(t) * d + c;
      float x0, x1, x2, x3;
      if constexpr (sizeof(Tw) == 2) {
        x0 = __bfloat162float(xr[0]);
        x1 = __bfloat162float(xr[1]);
        x2 = __bfloat162float(xr[2]);
        x3 = __bfloat162float(xr[3]);
      } else {
        x0 = xr[0];
        x1 = xr[1];
        x2 = xr[2];
        x3 = xr[3];
      }
      a.x -= fmaf(lB, x0 - lmu, lA);
      a.y -= fmaf(lB, x1 - lmu, lA);
      a.z -= fmaf(lB, x2 - lmu, lA);
      a.w -= fmaf(lB, x3 - lmu, lA);
    }
    *reinterpret_cast<float4*>(out + c) = a;
  }
}

// out[g][n] = sum of scale[r] src[r][n] over the rows r of group g
// (ascending; scale nullable: 1).
__global__ void group_colsum_kernel(const bf16* __restrict__ src, long long ld, const int* __restrict__ offsets,
                                    int rows, int N, const float* __restrict__ scale, float* __restrict__ out) {
  pdl_entry();
  const int g = blockIdx.y;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int r0 = offsets ? offsets[g] : 0;
  const int r1 = offsets ? offsets[g + 1] : rows;
  float s = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float v = __bfloat162float(src[static_cast<size_t>(r) * ld + n]);
    s = scale ? fmaf(scale[r], v, s) : s + v;
  }
  out[static_cast<size_t>(g) * N + n] = s;
}

inline unsigned warp_grid(int T) { return static_cast<unsigned>((static_cast<long long>(T) * 32 + 255) / 256); }

}  // namespace

size_t router_wgrad_partial_bytes(const moe_config& cfg) {
  const size_t nchunks = (static_cast<size_t>(cfg.T) + RW_TOK - 1) / RW_TOK;
  return nchunks * cfg.E * cfg.d * sizeof(float);
}

moe_status launch_bwd_gather(const moe_config& cfg, const void* dY, const void* Yp, const int* pos, const float* w,
                             void* dYg, float* wp, float* dot, cudaStream_t st) {
  const uint4* dy = static_cast<const uint4*>(dY);
  const uint4* yp = static_cast<const uint4*>(Yp);
  uint4* dyg = static_cast<uint4*>(dYg);
  const int nv = cfg.d / 8;
  if (cfg.k <= 2)
    launch_pdl(bwd_gather_kernel<2>, dim3(warp_grid(cfg.T)), dim3(256), 0, st, dy, yp, pos, w, cfg.T, cfg.k, nv, dyg,
               wp, dot);
  else if (cfg.k <= 4)
    launch_pdl(bwd_gather_kernel<4>, dim3(warp_grid(cfg.T)), dim3(256), 0, st, dy, yp, pos, w, cfg.T, cfg.k, nv, dyg,
               wp, dot);
  else
    launch_pdl(bwd_gather_kernel<8>, dim3(warp_grid(cfg.T)), dim3(256), 0, st, dy, yp, pos, w, cfg.T, cfg.k, nv, dyg,
               wp, dot);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_router_bwd(const moe_config& cfg, const void* x, const void* Wr, const int* idx, const float* w,
                             const int* counts, const float* dot, unsigned long long* imp, float* coef, float* dl,
                             float* lnc, cudaStream_t st) {
  const long long nslots = static_cast<long long>(cfg.T) * cfg.k;
  long long blocks = (nslots + 255) / 256;
  if (blocks > 1184) blocks = 1184;
  launch_pdl(importance_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), sizeof(unsigned long long) * cfg.E, st,
             idx, w, nslots, cfg.E, imp);
  launch_pdl(balance_coef_kernel, dim3(1), dim3(1024), 0, st, imp, counts, cfg.E, cfg.T, cfg.lambda_balance,
             cfg.balance, cfg.balance_gamma, coef);
  launch_pdl(router_bwd_kernel, dim3((cfg.T + 255) / 256), dim3(256), 0, st, idx, w, dot, coef, cfg.T, cfg.k, cfg.E,
             dl);
  if (lnc) {
    if (cfg.dtype != MOE_BF16 || (cfg.d % 8)) return MOE_ERR_UNSUPPORTED;
    launch_pdl(ln_router_bwd_kernel, dim3(warp_grid(cfg.T)), dim3(256), 0, st, static_cast<const bf16*>(x),
               static_cast<const bf16*>(Wr), idx, cfg.T, cfg.d, cfg.k, cfg.E, dl, lnc);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_router_bwd_raw(const moe_config& cfg, const float* logits, const int* idx, const float* w,
                                 const float* dot, const float* coef, float* dlD, cudaStream_t st) {
  const int nv = (cfg.E + 31) / 32;
  const unsigned grid = warp_grid(cfg.T);
#define MOE_RAWBWD(NVv)                                                                                          \
  launch_pdl(router_bwd_raw_kernel<NVv>, dim3(grid), dim3(256), 0, st, logits, idx, w, dot, coef, cfg.T, cfg.k, \
             cfg.E, dlD)
  if (nv <= 1) MOE_RAWBWD(1);
  else if (nv <= 2) MOE_RAWBWD(2);
  else if (nv <= 4) MOE_RAWBWD(4);
  else if (nv <= 8) MOE_RAWBWD(8);
  else if (nv <= 16) MOE_RAWBWD(16);
  else MOE_RAWBWD(32);
#undef MOE_RAWBWD
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_balance_stat_switch(const moe_config& cfg, const int* idx, const float* w, const int* counts,
                                      unsigned long long* imp, moe_stats* stats, cudaStream_t st) {
  moe_status s = launch_zero(imp, sizeof(unsigned long long) * cfg.E, nullptr, 0, st);
  if (s != MOE_OK) return s;
  const long long nslots = static_cast<long long>(cfg.T) * cfg.k;
  long long blocks = (nslots + 255) / 256;
  if (blocks > 1184) blocks = 1184;
  launch_pdl(importance_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), sizeof(unsigned long long) * cfg.E, st,
             idx, w, nslots, cfg.E, imp);
  launch_pdl(balance_switch_stat_kernel, dim3(1), dim3(1024), 0, st, imp, counts, cfg.E, cfg.T, cfg.lambda_balance,
             stats);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_router_wgrad(const moe_config& cfg, const void* x, const int* idx, const float* dl,
                               const float* lnc, float* partial, float* dWr, cudaStream_t st) {
  const int nchunks = (cfg.T + RW_TOK - 1) / RW_TOK;
  dim3 grid(nchunks, (cfg.d + RW_COLS - 1) / RW_COLS, (cfg.E + RW_EXP - 1) / RW_EXP);
  const size_t smem = sizeof(float) * RW_WARPS * RW_EXP * 8 * 32;
  static DeviceOnce attr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const moe_status sa = attr.run(dev, [&] {
    const int b = static_cast<int>(smem);
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    return cudaFuncSetAttribute(router_wgrad_partial_kernel<bf16, false>, a, b) == cudaSuccess &&
                   cudaFuncSetAttribute(router_wgrad_partial_kernel<bf16, true>, a, b) == cudaSuccess &&
                   cudaFuncSetAttribute(router_wgrad_partial_kernel<float, false>, a, b) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  });
  if (sa != MOE_OK) return sa;
  // raw softmax weights: dl is the dense [T, E] logit gradient
  const bool dense = (cfg.route_flags & MOE_ROUTE_RAW_PROBS) != 0;
  if (cfg.dtype == MOE_BF16 && dense)
    launch_pdl(router_wgrad_partial_kernel<bf16, true>, dim3(grid), dim3(RW_WARPS * 32), smem, st,
               static_cast<const bf16*>(x), idx, dl, cfg.T, cfg.d, cfg.k, cfg.E, lnc, partial);
  else if (cfg.dtype == MOE_BF16)
    launch_pdl(router_wgrad_partial_kernel<bf16, false>, dim3(grid), dim3(RW_WARPS * 32), smem, st,
               static_cast<const bf16*>(x), idx, dl, cfg.T, cfg.d, cfg.k, cfg.E, lnc, partial);
  else if (!dense)
    launch_pdl(router_wgrad_partial_kernel<float, false>, dim3(grid), dim3(RW_WARPS * 32), smem, st,
               static_cast<const float*>(x), idx, dl, cfg.T, cfg.d, cfg.k, cfg.E, lnc, partial);
  else
    return MOE_ERR_UNSUPPORTED;
  const long long Ed = static_cast<long long>(cfg.E) * cfg.d;
  launch_pdl(router_wgrad_reduce_kernel, dim3(static_cast<unsigned>((Ed + 255) / 256)), dim3(256), 0, st, partial,
             nchunks, Ed, dWr);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <typename Tw, int KM>
void launch_bwd_dx_t(const moe_config& cfg, const float* dXp, const int* pos, const int* idx, const float* dl,
                     const void* Wr, const void* x, const float* lnc, int accumulate, float* dX, cudaStream_t st) {
  const Tw* w = static_cast<const Tw*>(Wr);
  const Tw* xx = static_cast<const Tw*>(x);
  const bool dense = (cfg.route_flags & MOE_ROUTE_RAW_PROBS) != 0;
  if (dense)
    launch_pdl(bwd_dx_kernel<Tw, KM, false, true>, dim3(warp_grid(cfg.T)), dim3(256), 0, st, dXp, pos, idx, dl, w,
               cfg.T, cfg.k, cfg.d, cfg.E, xx, lnc, accumulate, dX);
  else if (lnc)
    launch_pdl(bwd_dx_kernel<Tw, KM, true, false>, dim3(warp_grid(cfg.T)), dim3(256), 0, st, dXp, pos, idx, dl, w,
               cfg.T, cfg.k, cfg.d, cfg.E, xx, lnc, accumulate, dX);
  else
    launch_pdl(bwd_dx_kernel<Tw, KM, false, false>, dim3(warp_grid(cfg.T)), dim3(256), 0, st, dXp, pos, idx, dl, w,
               cfg.T, cfg.k, cfg.d, cfg.E, xx, lnc, accumulate, dX);
}

template <typename Tw>
void launch_bwd_dx_k(const moe_config& cfg, const float* dXp, const int* pos, const int* idx, const float* dl,
                     const void* Wr, const void* x, const float* lnc, int accumulate, float* dX, cudaStream_t st) {
  if (cfg.k <= 2)
    launch_bwd_dx_t<Tw, 2>(cfg, dXp, pos, idx, dl, Wr, x, lnc, accumulate, dX, st);
  else if (cfg.k <= 4)
    launch_bwd_dx_t<Tw, 4>(cfg, dXp, pos, idx, dl, Wr, x, lnc, accumulate, dX, st);
  else
    launch_bwd_dx_t<Tw, 8>(cfg, dXp, pos, idx, dl, Wr, x, lnc, accumulate, dX, st);
}

moe_status launch_bwd_dx(const moe_config& cfg, const float* dXp, const int* pos, const int* idx, const float* dl,
                         const void* Wr, const void* x, const float* lnc, int accumulate, float* dX, cudaStream_t st) {
  if (cfg.dtype == MOE_BF16)
    launch_bwd_dx_k<bf16>(cfg, dXp, pos, idx, dl, Wr, x, lnc, accumulate, dX, st);
  else
    launch_bwd_dx_k<float>(cfg, dXp, pos, idx, dl, Wr, x, lnc, accumulate, dX, st);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_group_colsum(const void* src, long long ld, const int* offsets, int G, int rows, int N,
                               const float* scale, float* out, cudaStream_t st) {
  dim3 grid((N + 255) / 256, G);
  launch_pdl(group_colsum_kernel, dim3(grid), dim3(256), 0, st, static_cast<const bf16*>(src), ld, offsets, rows, N,
             scale, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// Router: logits, top-k with lowest-index tie-break, renormalised weights,
// routed-slot histogram -- one fused kernel.
//
//   l[t,e]  = x[t] . Wr[e] (+ expert_bias[e]) (+ noise[t,e])
//   idx[t]  = the k largest l[t,:] (larger first; equal -> lower index)
//   w[t,j]  = exp(l[idx_j] - l[idx_0]) / sum_j' exp(l[idx_j'] - l[idx_0])
//   counts[e] += #{j : idx[t,j] = e}
// Sources: [P1] "'More parameters is better' is not the story..." 3.1
// (logits = h W_r, softmax, top-k), 3.3 (weights renormalised over the
// top-k, non-top-k logits masked); [P3] "MoE architecture revealed..." 2.3
// (Gumbel noise added to the router score before top-k).  Selecting on the
// logits equals selecting on softmax(l), which is monotone.
//
// bf16: a CTA owns 64 tokens; 4 warps compute the 64 x 128 logit block of
// an expert chunk with mma.sync m16n8k16 (fp32 accumulate) from
// double-buffered cp.async tiles of x and Wr, then 64 threads merge the
// chunk into each token's running top-k.  x is read from HBM once (the
// kernel is bound by that read); Wr stays in L2.
// fp32: one warp per token on the CUDA cores (tiny workloads).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int MAXK = 8;
constexpr int RT_TM = 64;         // tokens per CTA
constexpr int RT_NE = 128;        // experts per chunk
constexpr int RT_BK = 64;         // k per stage
constexpr int RT_LD = RT_BK + 8;  // padded smem row (bf16): conflict-free fragment loads

// Insert (val, e) into a descending top-k list; equal values keep the
// earlier (lower) index first because experts arrive in increasing order.
__device__ __forceinline__ void topk_insert(float (&v)[MAXK], int (&ix)[MAXK], int k, float val, int e) {
#pragma unroll
  for (int p = MAXK - 1; p > 0; --p) {
    if (p < k) {
      if (val > v[p - 1]) {
        v[p] = v[p - 1];
        ix[p] = ix[p - 1];
      } else if (val > v[p]) {
        v[p] = val;
        ix[p] = e;
      }
    }
  }
  if (val > v[0]) {
    v[0] = val;
    ix[0] = e;
  }
}

__device__ __forceinline__ void topk_finish(const float (&v)[MAXK], const int (&ix)[MAXK], int k, bool finite,
                                            int t, int* idx, float* w, int* hist) {
  if (!finite) {
    for (int j = 0; j < k; ++j) {
      idx[static_cast<size_t>(t) * k + j] = -1;
      w[static_cast<size_t>(t) * k + j] = 0.f;
    }
    return;
  }
  float ex[MAXK];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j < k) {
      ex[j] = expf(v[j] - v[0]);
      s += ex[j];
    }
  }
  const float inv = 1.0f / s;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j < k) {
      idx[static_cast<size_t>(t) * k + j] = ix[j];
      w[static_cast<size_t>(t) * k + j] = ex[j] * inv;
      atomicAdd(&hist[ix[j]], 1);
    }
  }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct RouteSmem {
  bf16 xs[2][RT_TM][RT_LD];
  bf16 ws[2][RT_NE][RT_LD];
  float L[RT_TM][RT_NE + 1];
};

__global__ void __launch_bounds__(128)
route_bf16_kernel(const bf16* __restrict__ x, const bf16* __restrict__ Wr, const float* __restrict__ ebias,
                  const float* __restrict__ noise, int T, int d, int E, int k, int* __restrict__ idx,
                  float* __restrict__ w, int* __restrict__ counts) {
  extern __shared__ uint8_t smem_raw[];
  RouteSmem& S = *reinterpret_cast<RouteSmem*>(smem_raw);
  int* hist = reinterpret_cast<int*>(smem_raw + sizeof(RouteSmem));

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int t0 = blockIdx.x * RT_TM;
  const int nk = (d + RT_BK - 1) / RT_BK;

  for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;

  float tv[MAXK];
  int tix[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    tv[j] = -INFINITY;
    tix[j] = -1;
  }
  bool finite = true;

  for (int e0 = 0; e0 < E; e0 += RT_NE) {
    const int ne = min(RT_NE, E - e0);
    const int nfrag = (ne + 7) / 8;
    float acc[RT_NE / 8][4];
#pragma unroll
    for (int f = 0; f < RT_NE / 8; ++f) acc[f][0] = acc[f][1] = acc[f][2] = acc[f][3] = 0.f;

    auto load_stage = [&](int stage, int kb) {
      const int k0 = kb * RT_BK;
      // x tile: 64 rows x 8 chunks of 16 B; out-of-range chunks are zero-filled
      for (int q = tid; q < RT_TM * 8; q += 128) {
        const int r = q >> 3, ch = q & 7;
        const int t = t0 + r, kk = k0 + ch * 8;
        const bool ok = t < T && kk < d;
        const bf16* src = ok ? x + static_cast<size_t>(t) * d + kk : x;
        cp_async16(&S.xs[stage][r][ch * 8], src, ok);
      }
      for (int q = tid; q < RT_NE * 8; q += 128) {
        const int r = q >> 3, ch = q & 7;
        const int e = e0 + r, kk = k0 + ch * 8;
        const bool ok = r < ne && kk < d;
        const bf16* src = ok ? Wr + static_cast<size_t>(e) * d + kk : Wr;
        cp_async16(&S.ws[stage][r][ch * 8], src, ok);
      }
      cp_async_commit();
    };

    load_stage(0, 0);
    for (int kb = 0; kb < nk; ++kb) {
      if (kb + 1 < nk) {
        load_stage((kb + 1) & 1, kb + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const int st = kb & 1;
      const int r0 = warp * 16;
#pragma unroll
      for (int kk = 0; kk < RT_BK / 16; ++kk) {
        uint32_t a[4];
        a[0] = *reinterpret_cast<const uint32_t*>(&S.xs[st][r0 + g][kk * 16 + 2 * c4]);
        a[1] = *reinterpret_cast<const uint32_t*>(&S.xs[st][r0 + g + 8][kk * 16 + 2 * c4]);
        a[2] = *reinterpret_cast<const uint32_t*>(&S.xs[st][r0 + g][kk * 16 + 2 * c4 + 8]);
        a[3] = *reinterpret_cast<const uint32_t*>(&S.xs[st][r0 + g + 8][kk * 16 + 2 * c4 + 8]);
#pragma unroll
        for (int f = 0; f < RT_NE / 8; ++f) {
          if (f < nfrag) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&S.ws[st][f * 8 + g][kk * 16 + 2 * c4]);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&S.ws[st][f * 8 + g][kk * 16 + 2 * c4 + 8]);
            mma_bf16_16816(acc[f], a, b0, b1);
          }
        }
      }
      __syncthreads();
    }

    // logits of this chunk (+ bias, + noise) -> smem
    {
      const int r0 = warp * 16;
#pragma unroll
      for (int f = 0; f < RT_NE / 8; ++f) {
        if (f < nfrag) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = r0 + g + ((q & 2) ? 8 : 0);
            const int col = f * 8 + 2 * c4 + (q & 1);
            const int e = e0 + col;
            const int t = t0 + r;
            float v = acc[f][q];
            if (e < E && t < T) {
              if (ebias) v += ebias[e];
              if (noise) v += noise[static_cast<size_t>(t) * E + e];
            }
            S.L[r][col] = v;
          }
        }
      }
    }
    __syncthreads();
    if (tid < RT_TM && t0 + tid < T) {
      for (int col = 0; col < ne; ++col) {
        const float v = S.L[tid][col];
        if (!isfinite(v)) finite = false;
        topk_insert(tv, tix, k, v, e0 + col);
      }
    }
    __syncthreads();
  }

  if (tid < RT_TM && t0 + tid < T) topk_finish(tv, tix, k, finite, t0 + tid, idx, w, hist);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&counts[e], hist[e]);
}

// fp32 storage: one warp per token, fp32 dot products on the CUDA cores.
__global__ void route_f32_kernel(const float* __restrict__ x, const float* __restrict__ Wr,
                                 const float* __restrict__ ebias, const float* __restrict__ noise, int T, int d,
                                 int E, int k, int* __restrict__ idx, float* __restrict__ w,
                                 int* __restrict__ counts) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const int t = warp;
  float tv[MAXK];
  int tix[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    tv[j] = -INFINITY;
    tix[j] = -1;
  }
  bool finite = true;
  const float* xr = x + static_cast<size_t>(t) * d;
  for (int e = 0; e < E; ++e) {
    const float* wr = Wr + static_cast<size_t>(e) * d;
    float s = 0.f;
    for (int i = lane; i < d; i += 32) s = fmaf(xr[i], wr[i], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (ebias) s += ebias[e];
    if (noise) s += noise[static_cast<size_t>(t) * E + e];
    if (!isfinite(s)) finite = false;
    topk_insert(tv, tix, k, s, e);
  }
  if (lane == 0) topk_finish(tv, tix, k, finite, t, idx, w, counts);
}

}  // namespace

moe_status launch_route(const moe_config& cfg, const void* x, const void* Wr, const float* expert_bias,
                        const float* noise, int* idx, float* w, int* counts, cudaStream_t stream) {
  if (cudaMemsetAsync(counts, 0, sizeof(int) * cfg.E, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cfg.dtype == MOE_BF16) {
    const size_t smem = sizeof(RouteSmem) + sizeof(int) * cfg.E;
    static thread_local int attr_dev = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (attr_dev != dev) {
      if (cudaFuncSetAttribute(route_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(RouteSmem) + sizeof(int) * 1024)) != cudaSuccess)
        return MOE_ERR_CUDA;
      attr_dev = dev;
    }
    const int grid = (cfg.T + RT_TM - 1) / RT_TM;
    route_bf16_kernel<<<grid, 128, smem, stream>>>(static_cast<const bf16*>(x), static_cast<const bf16*>(Wr),
                                                   expert_bias, noise, cfg.T, cfg.d, cfg.E, cfg.k, idx, w,
                                                   counts);
  } else {
    const int threads = 256;
    const long long grid = (static_cast<long long>(cfg.T) * 32 + threads - 1) / threads;
    route_f32_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(
        static_cast<const float*>(x), static_cast<const float*>(Wr), expert_bias, noise, cfg.T, cfg.d, cfg.E,
        cfg.k, idx, w, counts);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

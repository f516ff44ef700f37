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
// bf16 with a workspace: the logits x . Wr^T run on the tcgen05 grouped
// GEMM (one group of T rows, N = E rounded up to 8 with zero rows past E,
// fp32 out into the workspace; x streams from HBM through TMA), then
// route_topk_kernel takes each token's top-k with one warp.  bf16 without a
// workspace: a CTA owns 64 tokens; 4 warps compute the 64 x 128 logit block
// of an expert chunk with mma.sync m16n8k16 (fp32 accumulate) from a 3- to
// 5-stage cp.async ring of x and Wr tiles, then 64 threads merge the chunk
// into each token's running top-k.
// fp32: one warp per token on the CUDA cores (tiny workloads).
//
// LayerNorm before the router ([P2] "MoE mixture-of-experts architecture:
// principles and engineering practice" 5.2:
// a LayerNorm, then the linear router; identity scale and zero shift, eps
// 1e-5, biased variance).  With mu_t, r_t = 1/sqrt(var_t + eps) of row t
// and S_e = sum_i Wr[e,i]:
//   LN(x_t) . Wr[e] = r_t (x_t . Wr[e] - mu_t S_e),
// so the GEMM still contracts the stored x and the top-k kernel applies the
// row statistics (two passes over x_t in fp32) and S (one warp per expert).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int RT_TM = 64;         // tokens per CTA
constexpr int RT_NE = 128;        // experts per chunk
constexpr int RT_BK = 64;         // k per stage
constexpr int RT_LD = RT_BK + 8;  // padded smem row (bf16): conflict-free fragment loads

// Backup experts of a token for rerouting on overflow: its entries k .. kk-1
// of the sorted list (kk <= 2k), -1 past kk or for a non-finite token.
__device__ __forceinline__ void write_backup(const int (&ix)[MAXK], int k, int kk, bool finite, int t,
                                             int* backup) {
#pragma unroll
  for (int q = 0; q < MAXK; ++q)  // static indices keep ix in registers
    if (q >= k && q < 2 * k) backup[static_cast<size_t>(t) * k + (q - k)] = (finite && q < kk) ? ix[q] : -1;
}

constexpr float kLnEps = 1e-5f;

// mean and 1/sqrt(biased variance + eps) of a bf16 row of d (a multiple of 8)
// elements, one warp, two passes (the second centred on the mean).
__device__ __forceinline__ void row_stats_bf16(const bf16* __restrict__ row, int d, float& mu, float& r) {
  const uint4* v = reinterpret_cast<const uint4*>(row);
  const int nv = d >> 3;
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int i = lane; i < nv; i += 32) {
    const uint4 q = v[i];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) s += bf16lo(u[c]) + bf16hi(u[c]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  mu = s / static_cast<float>(d);
  float q2 = 0.f;
  for (int i = lane; i < nv; i += 32) {
    const uint4 q = v[i];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float a = bf16lo(u[c]) - mu, b = bf16hi(u[c]) - mu;
      q2 = fmaf(a, a, fmaf(b, b, q2));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q2 += __shfl_xor_sync(0xffffffffu, q2, o);
  r = 1.0f / sqrtf(q2 / static_cast<float>(d) + kLnEps);
}

__device__ __forceinline__ void row_stats_f32(const float* __restrict__ row, int d, float& mu, float& r) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int i = lane; i < d; i += 32) s += row[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  mu = s / static_cast<float>(d);
  float q2 = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float a = row[i] - mu;
    q2 = fmaf(a, a, q2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q2 += __shfl_xor_sync(0xffffffffu, q2, o);
  r = 1.0f / sqrtf(q2 / static_cast<float>(d) + kLnEps);
}

// S[e] = sum_i Wr[e,i] (fp32), one warp per expert; S[e] = 0 for E <= e < ld.
__global__ void weight_row_sum_kernel(const bf16* __restrict__ Wr, int E, int d, int ld, float* __restrict__ S) {
  pdl_entry();
  const int e = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= ld) return;
  float s = 0.f;
  if (e < E) {
    const uint4* v = reinterpret_cast<const uint4*>(Wr + static_cast<size_t>(e) * d);
    for (int i = lane; i < (d >> 3); i += 32) {
      const uint4 q = v[i];
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) s += bf16lo(u[c]) + bf16hi(u[c]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  if (lane == 0) S[e] = s;
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

// Shared-memory layout of route_bf16_kernel (dynamic): a ring of STAGES
// stages, each an x tile [64][RT_LD] and a Wr tile [nep][RT_LD] (nep = the
// expert chunk width, <= 128, a multiple of 8); after the K loop the ring
// is reused for the chunk's logits L[64][nep+1]; then E ints of histogram.
struct RouteLayout {
  int nep;
  size_t stage_bytes, ring_bytes, total;
  __host__ __device__ RouteLayout(int E, int stages) {
    nep = ((E < RT_NE ? E : RT_NE) + 7) / 8 * 8;
    stage_bytes = static_cast<size_t>(RT_TM + nep) * RT_LD * 2;
    const size_t lbytes = static_cast<size_t>(RT_TM) * (nep + 1) * 4;
    ring_bytes = stages * stage_bytes > lbytes ? stages * stage_bytes : lbytes;
    total = ring_bytes + static_cast<size_t>(E) * 4;
  }
};

// Logits of 64 tokens against all experts (chunks of 128) from a cp.async
// ring of STAGES stages, plus bias and noise; then each token's top-k and
// the block histogram.
template <int STAGES>
__global__ void __launch_bounds__(128)
route_bf16_kernel(const bf16* __restrict__ x, const bf16* __restrict__ Wr, const float* __restrict__ ebias,
                  const float* __restrict__ noise, int T, int d, int E, int k, int* __restrict__ idx,
                  float* __restrict__ w, int* __restrict__ counts, int raw, float* __restrict__ ent) {
  pdl_entry();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const RouteLayout Lay(E, STAGES);
  const int nep = Lay.nep;
  int* hist = reinterpret_cast<int*>(smem_raw + Lay.ring_bytes);
  float* L = reinterpret_cast<float*>(smem_raw);  // [64][nep+1], aliases the ring after the K loop
  auto xs = [&](int st) { return reinterpret_cast<bf16*>(smem_raw + st * Lay.stage_bytes); };
  auto wsm = [&](int st) { return reinterpret_cast<bf16*>(smem_raw + st * Lay.stage_bytes) + RT_TM * RT_LD; };

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
  const bool need_stat = raw || ent;
  SoftStat sst;

  for (int e0 = 0; e0 < E; e0 += RT_NE) {
    const int ne = min(RT_NE, E - e0);
    const int nfrag = (ne + 7) / 8;
    float acc[RT_NE / 8][4];
#pragma unroll
    for (int f = 0; f < RT_NE / 8; ++f) acc[f][0] = acc[f][1] = acc[f][2] = acc[f][3] = 0.f;

    auto load_stage = [&](int stage, int kb) {
      const int k0 = kb * RT_BK;
      bf16* xd = xs(stage);
      bf16* wd = wsm(stage);
      // x tile: 64 rows x 8 chunks of 16 B; out-of-range chunks are zero-filled
      for (int q = tid; q < RT_TM * 8; q += 128) {
        const int r = q >> 3, ch = q & 7;
        const int t = t0 + r, kk = k0 + ch * 8;
        const bool ok = t < T && kk < d;
        const bf16* src = ok ? x + static_cast<size_t>(t) * d + kk : x;
        cp_async16(xd + r * RT_LD + ch * 8, src, ok);
      }
      for (int q = tid; q < nep * 8; q += 128) {
        const int r = q >> 3, ch = q & 7;
        const int e = e0 + r, kk = k0 + ch * 8;
        const bool ok = r < ne && kk < d;
        const bf16* src = ok ? Wr + static_cast<size_t>(e) * d + kk : Wr;
        cp_async16(wd + r * RT_LD + ch * 8, src, ok);
      }
    };

    // multistage ring: STAGES-1 blocks in flight ahead of the one computed
#pragma unroll
    for (int s0 = 0; s0 < STAGES - 1; ++s0) {
      if (s0 < nk) load_stage(s0, s0);
      cp_async_commit();
    }
    for (int kb = 0; kb < nk; ++kb) {
      cp_async_wait<STAGES - 2>();
      __syncthreads();
      const int nxt = kb + STAGES - 1;
      if (nxt < nk) load_stage(nxt % STAGES, nxt);
      cp_async_commit();
      const bf16* xa = xs(kb % STAGES);
      const bf16* wb = wsm(kb % STAGES);
      const int r0 = warp * 16;
#pragma unroll
      for (int kk = 0; kk < RT_BK / 16; ++kk) {
        uint32_t a[4];
        a[0] = *reinterpret_cast<const uint32_t*>(xa + (r0 + g) * RT_LD + kk * 16 + 2 * c4);
        a[1] = *reinterpret_cast<const uint32_t*>(xa + (r0 + g + 8) * RT_LD + kk * 16 + 2 * c4);
        a[2] = *reinterpret_cast<const uint32_t*>(xa + (r0 + g) * RT_LD + kk * 16 + 2 * c4 + 8);
        a[3] = *reinterpret_cast<const uint32_t*>(xa + (r0 + g + 8) * RT_LD + kk * 16 + 2 * c4 + 8);
#pragma unroll
        for (int f = 0; f < RT_NE / 8; ++f) {
          if (f < nfrag) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wb + (f * 8 + g) * RT_LD + kk * 16 + 2 * c4);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wb + (f * 8 + g) * RT_LD + kk * 16 + 2 * c4 + 8);
            mma_bf16_16816(acc[f], a, b0, b1);
          }
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // the ring becomes L

    // logits of this chunk (+ bias, + noise) -> L
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
            L[r * (nep + 1) + col] = v;
          }
        }
      }
    }
    __syncthreads();
    if (tid < RT_TM && t0 + tid < T) {
      for (int col = 0; col < ne; ++col) {
        const float v = L[tid * (nep + 1) + col];
        if (!isfinite(v)) finite = false;
        topk_insert(tv, tix, k, v, e0 + col);
        if (need_stat && finite) sst.add(v);
      }
    }
    __syncthreads();  // L is the ring again for the next expert chunk
  }

  if (tid < RT_TM && t0 + tid < T) topk_finish(tv, tix, k, finite, t0 + tid, idx, w, hist, raw, sst, ent);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&counts[e], hist[e]);
}

// Top-k of precomputed logits (row stride ld), one warp per token:
// l[t,e] = logits[t,e] (+ bias[e]) (+ noise[t,e]); with S (LayerNorm before
// the router) the stored value is x_t . Wr[e] and l[t,e] = r_t (logits[t,e]
// - mu_t S[e]) (+ ...), mu_t and r_t from the row x_t.  Lane i holds the
// logits of experts i, i+32, ... (NV per lane, -inf past E).  The softmax
// statistics come from one warp max m and then sums of exp(l - m); the
// top-k from k rounds of a warp argmax by (value desc, index asc), each
// round retiring its winner.  Lane 0 writes idx, the weights and the block
// histogram.
template <int NV>
__global__ void __launch_bounds__(256)
route_topk_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ ebias,
                  const float* __restrict__ noise, int T, int E, int k, int* __restrict__ idx, float* __restrict__ w,
                  int* __restrict__ counts, int raw, float* __restrict__ ent, const bf16* __restrict__ x, int d,
                  const float* __restrict__ S, int* __restrict__ backup, float* __restrict__ out_logits) {
  pdl_entry();
  extern __shared__ int hist_s[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist_s[e] = 0;
  __syncthreads();
  // with backup: the 2k best (at most E), the last k of them the backups
  const int kk = backup ? min(2 * k, E) : k;
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (t < T) {
    float mu = 0.f, r = 1.f;
    if (S) row_stats_bf16(x + static_cast<size_t>(t) * d, d, mu, r);
    const float* lr = logits + static_cast<size_t>(t) * ld;
    const float* nr = noise ? noise + static_cast<size_t>(t) * E : nullptr;
    float v[NV];
    bool finite = true;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = -INFINITY;
      if (e < E) {
        float a = lr[e];
        if (S) a = r * fmaf(-mu, S[e], a);
        if (ebias) a += ebias[e];
        if (nr) a += nr[e];
        if (!isfinite(a)) finite = false;
        v[i] = a;
      }
    }
    finite = __all_sync(0xffffffffu, finite);
    if (out_logits) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i < E) out_logits[static_cast<size_t>(t) * E + lane + 32 * i] = v[i];
    }
    SoftStat sst;
    float sel_v[MAXK];
    int sel_i[MAXK];
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      sel_v[j] = -INFINITY;
      sel_i[j] = -1;
    }
    if (finite) {
      if (raw || ent) {
        float m = v[0];
#pragma unroll
        for (int i = 1; i < NV; ++i) m = fmaxf(m, v[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.f, sz = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          if (lane + 32 * i < E) {
            const float dv = v[i] - m;
            const float ex = expf(dv);
            z += ex;
            sz = fmaf(ex, dv, sz);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          z += __shfl_xor_sync(0xffffffffu, z, o);
          sz += __shfl_xor_sync(0xffffffffu, sz, o);
        }
        sst.m = m;
        sst.Z = z;
        sst.S = sz;
      }
#pragma unroll
      for (int j = 0; j < MAXK; ++j) {
        if (j < kk) {
          // this lane's best remaining (the first of equal values: lower expert)
          float bv = v[0];
          int bi = lane;
#pragma unroll
          for (int i = 1; i < NV; ++i)
            if (v[i] > bv) {
              bv = v[i];
              bi = lane + 32 * i;
            }
          if (bv == -INFINITY) bi = 0x7fffffff;  // nothing left in this lane
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
              bv = ov;
              bi = oi;
            }
          }
          sel_v[j] = bv;
          sel_i[j] = bi;
          // the lane that held the winner retires it
#pragma unroll
          for (int i = 0; i < NV; ++i)
            if (lane + 32 * i == bi) v[i] = -INFINITY;
        }
      }
    }
    if (lane == 0) {
      topk_finish(sel_v, sel_i, k, finite, t, idx, w, hist_s, raw, sst, ent);
      if (backup) write_backup(sel_i, k, kk, finite, t, backup);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist_s[e]) atomicAdd(&counts[e], hist_s[e]);
}

// fp32 storage: one warp per token, fp32 dot products on the CUDA cores.
__global__ void route_f32_kernel(const float* __restrict__ x, const float* __restrict__ Wr,
                                 const float* __restrict__ ebias, const float* __restrict__ noise, int T, int d,
                                 int E, int k, int* __restrict__ idx, float* __restrict__ w,
                                 int* __restrict__ counts, int raw, float* __restrict__ ent, int layernorm,
                                 int* __restrict__ backup) {
  pdl_entry();
  const int kk = backup ? min(2 * k, E) : k;
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
  const bool need_stat = raw || ent;
  SoftStat sst;
  const float* xr = x + static_cast<size_t>(t) * d;
  float mu = 0.f, r = 1.f;
  if (layernorm) row_stats_f32(xr, d, mu, r);
  for (int e = 0; e < E; ++e) {
    const float* wr = Wr + static_cast<size_t>(e) * d;
    float s = 0.f;
    for (int i = lane; i < d; i += 32) s = fmaf(xr[i] - mu, wr[i], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (layernorm) s *= r;
    if (ebias) s += ebias[e];
    if (noise) s += noise[static_cast<size_t>(t) * E + e];
    if (!isfinite(s)) finite = false;
    topk_insert(tv, tix, kk, s, e);
    if (need_stat && finite) sst.add(s);
  }
  if (lane == 0) {
    topk_finish(tv, tix, k, finite, t, idx, w, counts, raw, sst, ent);
    if (backup) write_backup(tix, k, kk, finite, t, backup);
  }
}

}  // namespace

namespace {

template <int STAGES>
moe_status launch_route_stages(const moe_config& cfg, const void* x, const void* Wr, const float* expert_bias,
                               const float* noise, int* idx, float* w, int* counts, float* ent, cudaStream_t stream) {
  const RouteLayout Lay(cfg.E, STAGES);
  static DeviceOnce attr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const moe_status sa = attr.run(dev, [&] {
    const RouteLayout Lmax(1024, STAGES);
    return cudaFuncSetAttribute(route_bf16_kernel<STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(Lmax.total)) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  });
  if (sa != MOE_OK) return sa;
  dim3 grid((cfg.T + RT_TM - 1) / RT_TM, 1);
  launch_pdl(route_bf16_kernel<STAGES>, dim3(grid), dim3(128), Lay.total, stream, static_cast<const bf16*>(x),
             static_cast<const bf16*>(Wr), expert_bias, noise, cfg.T, cfg.d, cfg.E, cfg.k, idx, w, counts,
             (cfg.route_flags & MOE_ROUTE_RAW_PROBS) ? 1 : 0, ent);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Row stride of the fp32 logits on the tensor-core path: E rounded up to
// the GEMM's 8-column granule (columns past E hold the logits of zero
// weight rows and are never read).
// The largest E whose top-k runs in the logits GEMM's epilogue.  There one
// thread walks its token's E logits alone, against a warp per token in
// route_topk_kernel: measured per router call, the epilogue wins at E = 16
// (small prefill 23.4 -> 21.0 us, training 79.9 -> 66.0 us) and ties at
// E = 64 (large prefill 52.2 -> 51.5 us), but loses at E = 128 (decode, 64
// tokens: 34.0 -> 55.5 us).
constexpr int kRouteFuseMaxE = 64;

int logit_ld(const moe_config& cfg) { return cfg.E < 8 ? 8 : (cfg.E + 7) / 8 * 8; }

}  // namespace

size_t route_scratch_bytes(const moe_config& cfg) {
  if (cfg.dtype != MOE_BF16) return 0;
  const size_t ld = logit_ld(cfg);
  const bool ln = (cfg.route_flags & MOE_ROUTE_LAYERNORM) != 0;
  return (static_cast<size_t>(cfg.T) + (ln ? 1 : 0)) * ld * sizeof(float);
}

moe_status launch_route(const moe_config& cfg, const void* x, const void* Wr, const float* expert_bias,
                        const float* noise, int* idx, float* w, int* counts, float* ent, void* scratch, int* backup,
                        float* out_logits, int* err, cudaStream_t stream) {
  const int raw = (cfg.route_flags & MOE_ROUTE_RAW_PROBS) ? 1 : 0;
  const bool ln = (cfg.route_flags & MOE_ROUTE_LAYERNORM) != 0;
  if (ln && cfg.dtype == MOE_BF16 && !scratch) return MOE_ERR_UNSUPPORTED;  // the fold needs the workspace path
  if ((cfg.route_flags & MOE_ROUTE_REROUTE) && (!backup || (cfg.dtype == MOE_BF16 && !scratch)))
    return MOE_ERR_UNSUPPORTED;  // the backups live in the workspace
  if (out_logits && !(cfg.dtype == MOE_BF16 && scratch)) return MOE_ERR_UNSUPPORTED;  // top-k kernel path only
  moe_status zs = launch_zero(counts, sizeof(int) * cfg.E, err, err ? kWsZeroBytes : 0, stream);
  if (zs != MOE_OK) return zs;
  if (cfg.dtype == MOE_BF16 && scratch && !ln && !backup && cfg.E <= kRouteFuseMaxE && cfg.k <= MAXK) {
    // logits = x . Wr^T on the tcgen05 grouped GEMM (one group of T rows,
    // N = E rounded up to 8; the TMA box reads zeros past row E), and the
    // top-k in its epilogue: each thread holds one token's logits in TMEM,
    // so no logit goes through HBM
    GemmParams g{};
    g.G = 1;
    g.rows = cfg.T;
    g.N = logit_ld(cfg);
    g.K = cfg.d;
    g.mode = kModeRouteTopK;
    g.err = err;
    g.sched = err ? err + 1 : nullptr;
    g.route = RouteEpilogue{expert_bias, noise, idx, w, counts, ent, out_logits, cfg.E, cfg.k, raw};
    return launch_grouped_gemm_tc(g, kKindFwd, x, cfg.T, Wr, nullptr, cfg.E, stream);
  }
  if (cfg.dtype == MOE_BF16 && scratch) {
    // logits = x . Wr^T on the tcgen05 grouped GEMM (one group of T rows,
    // N = E rounded up to 8, fp32 out; the TMA box reads zeros past row E),
    // then the top-k per token (a LayerNorm in front, backups for rerouting,
    // or more than kRouteFuseMaxE experts)
    const int ld = logit_ld(cfg);
    float* logits = static_cast<float*>(scratch);
    float* S = ln ? logits + static_cast<size_t>(cfg.T) * ld : nullptr;
    if (ln) {
      launch_pdl(weight_row_sum_kernel, dim3(static_cast<unsigned>((ld * 32 + 255) / 256)), dim3(256), 0, stream,
                 static_cast<const bf16*>(Wr), cfg.E, cfg.d, ld, S);
    }
    GemmParams g{};
    g.G = 1;
    g.rows = cfg.T;
    g.N = ld;
    g.K = cfg.d;
    g.mode = kModePlain;
    g.out_f32 = 1;
    g.out = logits;
    g.err = err;
    g.sched = err ? err + 1 : nullptr;
    moe_status s = launch_grouped_gemm_tc(g, kKindFwd, x, cfg.T, Wr, nullptr, cfg.E, stream);
    if (s != MOE_OK) return s;
    const unsigned grid = static_cast<unsigned>((static_cast<long long>(cfg.T) * 32 + 255) / 256);
    const bf16* xb = static_cast<const bf16*>(x);
    const size_t hs = sizeof(int) * cfg.E;
    const int nv = (cfg.E + 31) / 32;
#define MOE_TOPK(NVv)                                                                                          \
  launch_pdl(route_topk_kernel<NVv>, dim3(grid), dim3(256), hs, stream, logits, ld, expert_bias, noise, cfg.T, \
             cfg.E, cfg.k, idx, w, counts, raw, ent, xb, cfg.d, S, backup, out_logits)
    if (nv <= 1) MOE_TOPK(1);
    else if (nv <= 2) MOE_TOPK(2);
    else if (nv <= 4) MOE_TOPK(4);
    else if (nv <= 8) MOE_TOPK(8);
    else if (nv <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
  } else if (cfg.dtype == MOE_BF16) {
    const int nep = ((cfg.E < RT_NE ? cfg.E : RT_NE) + 7) / 8 * 8;
    return nep <= 64 ? launch_route_stages<5>(cfg, x, Wr, expert_bias, noise, idx, w, counts, ent, stream)
                     : launch_route_stages<3>(cfg, x, Wr, expert_bias, noise, idx, w, counts, ent, stream);
  } else {
    const int threads = 256;
    const long long grid = (static_cast<long long>(cfg.T) * 32 + threads - 1) / threads;
    launch_pdl(route_f32_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), 0, stream,
               static_cast<const float*>(x), static_cast<const float*>(Wr), expert_bias, noise, cfg.T, cfg.d, cfg.E,
               cfg.k, idx, w, counts, raw, ent, ln ? 1 : 0, backup);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

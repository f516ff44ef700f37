// Grouped expert GEMM for fp32 storage, on the CUDA cores in fp32.
//
// Same contract as the tensor-core path (out[r,:] = act(A[r,:] . B_g^T) for
// the rows r of each group g), one thread per output element.  It serves the
// fp32 workloads, which are small validation shapes; the bf16 path is the
// performance path.  Sources as for the expert loop: [P2] "MoE
// mixture-of-experts architecture..." 4.2 and [P3] "MoE architecture
// revealed..." 3.3 (Linear -> GELU -> Linear per expert).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void grouped_gemm_f32_kernel(const GemmParams p, const float* __restrict__ A,
                                        const float* __restrict__ B0, const float* __restrict__ B1) {
  pdl_entry();
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int r = blockIdx.y;
  const int rows_total = p.offsets ? p.offsets[p.G] : p.rows;
  if (n >= p.N || r >= rows_total || r >= p.rows_alloc) return;
  int g = 0;
  if (p.offsets) {
    int lo = 0, hi = p.G;  // largest g with offsets[g] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.offsets[mid] <= r) lo = mid; else hi = mid;
    }
    g = lo;
  }
  const float* a = A + static_cast<size_t>(r) * p.K;
  const size_t brow = (static_cast<size_t>(g) * p.N + n) * p.K;
  float acc = 0.f;
  for (int kk = 0; kk < p.K; ++kk) acc = fmaf(a[kk], B0[brow + kk], acc);
  float out;
  if (p.mode == kModeSwiGLU) {
    float up = 0.f;
    for (int kk = 0; kk < p.K; ++kk) up = fmaf(a[kk], B1[brow + kk], up);
    out = silu_f(acc) * up;
  } else {
    if (p.bias) acc += static_cast<const float*>(p.bias)[static_cast<size_t>(g) * p.N + n];
    out = p.mode == kModeGeLU ? gelu_f(acc) : acc;
  }
  static_cast<float*>(p.out)[static_cast<size_t>(r) * p.N + n] = out;
}

}  // namespace

moe_status launch_grouped_gemm_f32(const GemmParams& p_in, const void* A, long long a_rows, const void* B0,
                                   const void* B1, cudaStream_t stream) {
  GemmParams p = p_in;
  p.rows_alloc = a_rows;
  if (a_rows <= 0) return MOE_OK;
  const long long rows = p.offsets ? a_rows : p.rows;
  if (rows > 2147483647LL) return MOE_ERR_UNSUPPORTED;
  dim3 block(128);
  dim3 grid((p.N + 127) / 128, static_cast<unsigned>(rows));
  launch_pdl(grouped_gemm_f32_kernel, dim3(grid), dim3(block), 0, stream, p, static_cast<const float*>(A),
             static_cast<const float*>(B0), static_cast<const float*>(B1));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

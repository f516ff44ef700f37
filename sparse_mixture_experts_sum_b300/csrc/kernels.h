// Host-side declarations of the layer's kernel launchers (internal; the
// public C ABI is include/moe.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

enum GemmMode : int { kModePlain = 0, kModeSwiGLU = 1, kModeGeLU = 2 };

// One grouped GEMM: out[r, :] = act(A[r, :] . B_g^T) for the rows r of each group.
struct GemmParams {
  const int* offsets;    // [G+1] device row offsets, or nullptr: one group of `rows` rows
  int G;                 // groups (experts)
  int rows;              // rows of the single group when offsets == nullptr
  long long rows_alloc;  // rows allocated in A and out: no row at or past it is written (set by the launcher)
  int N;                 // output columns per group (rows of B per group)
  int K;                 // contraction length
  int mode;              // GemmMode
  void* out;             // [*, N] row-major, storage type of the path
  const void* bias;      // [G, N] nullable (GeLU / plain)
  int* err;              // workspace error word
};

// sm_103a tensor-core path (bf16 in, fp32 accumulate, bf16 out).
moe_status launch_grouped_gemm_tc(const GemmParams& p, const void* A, long long a_rows, const void* B0,
                                  const void* B1, long long b_rows, cudaStream_t stream);

// fp32 CUDA-core path (fp32 storage and arithmetic).
moe_status launch_grouped_gemm_f32(const GemmParams& p, const void* A, long long a_rows, const void* B0,
                                   const void* B1, cudaStream_t stream);

// Router: logits, top-k, weights, routed counts.
moe_status launch_route(const moe_config& cfg, const void* x, const void* Wr, const float* expert_bias,
                        const float* noise, int* idx, float* w, int* counts, cudaStream_t stream);

// Dispatch: slot-major capacity ranks, offsets, positions, statistics, permute.
size_t dispatch_scratch_bytes(const moe_config& cfg);
moe_status launch_dispatch(const moe_config& cfg, int C, const int* idx, const void* x, int* kept,
                           int* offsets, int* pos, void* Xp, moe_stats* stats, void* scratch,
                           cudaStream_t stream);

// Size of the library's own dispatch scratch (moe_dispatch_static): enough
// for T*k <= 2^20 slots (256 chunks of 4096) at any E <= 1024.
constexpr size_t kStaticDispatchScratchBytes = 256u * 1025u * 4u + 256u * 1024u * 4u + 256u;
// Device address of that scratch on the current device (looked up on the
// first call per device); MOE_ERR_UNSUPPORTED if `need` bytes do not fit.
moe_status static_dispatch_scratch(size_t need, void** ptr);

// Combine / un-permute.
moe_status launch_combine(const moe_config& cfg, const void* Yp, const int* pos, const float* w,
                          const void* Sx, void* y, cudaStream_t stream);

// TMA descriptor of a row-major bf16 matrix [rows, inner] with a
// (box_inner x box_rows) box and 128-byte swizzling.
bool make_tma_2d_bf16(CUtensorMap* map, const void* base, long long inner, long long rows, int box_inner,
                      int box_rows);
int device_sm_count(int dev);

}  // namespace moe

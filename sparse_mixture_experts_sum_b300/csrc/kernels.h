// Host-side declarations of the layer's kernel launchers (internal; the
// public C ABI is include/moe.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "moe.h"

namespace moe {

// A per-device set-up step (a kernel attribute, a cached device property)
// that must succeed once per device: the first call for a device runs fn
// and, on MOE_OK, records it.  One lock covers the flags, so first calls from
// several host threads do not race.
class DeviceOnce {
 public:
  template <typename F>
  moe_status run(int dev, F&& fn) {
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev]) return MOE_OK;
    const moe_status s = fn();
    if (s == MOE_OK) done_[dev] = true;
    return s;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
};

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic
// stream serialization: the kernel may be scheduled while its predecessor in
// the stream is still running, once the predecessor's CTAs have all
// triggered (pdl_trigger) or exited.  Every kernel of this library starts
// with pdl_entry() (the GEMM: its shared-memory and TMEM set-up, then
// pdl_wait()), so no thread reads or writes global memory before the
// predecessor has completed and its writes are visible; since every kernel
// waits so, a kernel also runs after all earlier ones in the stream.  What
// overlaps is the launch and, in the GEMM, the set-up.  Launch errors are
// also reported by cudaGetLastError().
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Epilogue of a grouped GEMM (acc = the fp32 accumulator of one output element).
enum GemmMode : int {
  kModePlain = 0,      // out = acc (+ bias)
  kModeSwiGLU = 1,     // out = silu(gate) * up (B tile pairs W1 and W3 rows); zsave: gate | up
  kModeGeLU = 2,       // out = gelu(acc + bias); zsave: acc + bias
  // Backward modes; s = row_scale[r] (1 when null), dH = s * acc:
  kModeSwiGLUBwd = 3,  // g = zin[r,n], u = zin[r,N+n]: out[r,n] = dH*u*silu'(g), out[r,N+n] = dH*silu(g);
                       // hout + hout_lo = s*silu(g)*u
  kModeGeLUBwd = 4,    // out = dH * gelu'(zin[r,n]); hout + hout_lo = s*gelu(zin[r,n])
  // Fwd, one group of T rows, N = E (<= 256): the router.  Row t's logits
  // l = acc (+ r_bias) (+ r_noise[t]) go through the top-k in the epilogue
  // (value desc, index asc); out is not written
  kModeRouteTopK = 5,
};

// The router's top-k epilogue (kModeRouteTopK): idx/w [T, k]; counts [E]
// gets each expert's selections added (atomics); ent [T] the entropy of the
// softmax over all E (nullable); logits [T, E] the final logits (nullable);
// raw: w = the selected entries of that softmax instead of the softmax over
// the k selected logits.  A token with a non-finite logit gets idx -1, w 0,
// entropy NaN.
struct RouteEpilogue {
  const float* bias;   // [E] nullable
  const float* noise;  // [T, E] nullable
  int* idx;
  float* w;
  int* counts;
  float* ent;
  float* logits;
  int E, k, raw;
};

// Operand geometry of a grouped GEMM launch.
enum GemmKind : int {
  kKindFwd = 0,    // out[r,:] = A[r,:] . B_g^T; A [rows,K] and B_g [N,K] both K-contiguous
  kKindDgrad = 1,  // out[r,:] = A[r,:] . B_g;   A [rows,K] K-contiguous, B_g [K,N] N-contiguous
  kKindWgrad = 2,  // out_g = A_g^T . B_g over the group's rows; A [rows,M], B [rows,N]
};

// One grouped GEMM.  Groups (experts) own the row ranges [offsets[g],
// offsets[g+1]) of the activation matrices: the output rows (Fwd, Dgrad) or
// the contraction (Wgrad).
struct GemmParams {
  const int* offsets;    // [G+1] device row offsets, or nullptr: one group of `rows` rows
  int G;                 // groups (experts)
  int rows;              // rows of the single group when offsets == nullptr
  long long rows_alloc;  // rows allocated in the activation operands (set by the launcher)
  int M;                 // Wgrad: output rows per group
  int N;                 // output columns (per group)
  int K;                 // Fwd/Dgrad: contraction length
  int k_split;           // Dgrad: k < k_split reads B0 rows, k >= k_split reads B1 rows k - k_split (0: B0 only)
  int m_split;           // Wgrad: output rows m >= m_split go to out2 (row m - m_split); 0: all to out
  int mode;              // GemmMode
  int out_f32;           // output element type: 1 fp32, 0 bf16
  void* out;             // Fwd/Dgrad: [rows, ldo]; Wgrad: [G, M or m_split, N]
  void* out2;            // Wgrad second output [G, M - m_split, N]
  long long ldo;         // Fwd/Dgrad row stride of out (elements); 0: N
  void* zsave;           // Fwd SwiGLU/GeLU: pre-activations out (fp32), nullable
  const void* zin;       // *Bwd modes: saved pre-activations (fp32)
  long long ldz;         // row stride of zsave / zin (elements)
  const float* row_scale;  // *Bwd modes: per output row factor of the accumulator, nullable (1)
  void* hout;            // *Bwd modes: s * act(z) per row, rounded to bf16 ([rows, N]), nullable
  void* hout_lo;         // *Bwd modes: the bf16 residual s * act(z) - hout ([rows, N]), nullable
  int b_lo;              // Wgrad: out_g = A_g^T . (B0_g + B1_g) -- the contraction runs over the
                         // group's rows twice, with B0 then with B1 (a hi/lo pair)
  int cta_pairs;         // Fwd: 256-row tiles on CTA pairs where the groups average >= 256 rows
  const void* bias;      // [G, N] nullable (GeLU / plain)
  int* err;              // workspace error word
  int* sched;            // [2] the workspace's tile scheduler words, zero at the launch (it leaves them
                         // zero); nullptr: a static round-robin schedule
  // Fwd only: one more group with its own operands (the shared expert):
  // xrows rows of its own A, its own weights, output xout [xrows, ldo],
  // pre-activations xzsave, bias xbias [N].  xrows = 0: none.
  int xrows;
  void* xout;
  void* xzsave;
  const void* xbias;
  RouteEpilogue route;  // kModeRouteTopK
};

// Operands of the extra group of a Fwd launch.
struct GemmExtra {
  const void* A;     // [xrows, K]
  const void* B0;    // [N, K]
  const void* B1;    // [N, K] (SwiGLU up), nullable
};

// sm_103a tensor-core path (bf16 in, fp32 accumulate).  A: the activation
// operand (a_rows rows); B0/B1: weights (b_rows rows each) for Fwd/Dgrad, or
// B0 = the second activation operand (a_rows rows) for Wgrad.
moe_status launch_grouped_gemm_tc(const GemmParams& p, int kind, const void* A, long long a_rows, const void* B0,
                                  const void* B1, long long b_rows, cudaStream_t stream,
                                  const GemmExtra* extra = nullptr);

// fp32 CUDA-core path (fp32 storage and arithmetic).
moe_status launch_grouped_gemm_f32(const GemmParams& p, const void* A, long long a_rows, const void* B0,
                                   const void* B1, cudaStream_t stream);

// Router: logits, top-k, weights, routed counts.  scratch (nullable, at
// least route_scratch_bytes) holds the fp32 logits of the tensor-core path;
// err: the workspace error word (nullable), zeroed here with counts.
// backup [T,k] (MOE_ROUTE_REROUTE, else nullable): each token's next-best
// experts, ranks k .. 2k-1, -1 where none.  out_logits [T,E] (nullable; bf16
// with scratch only): the final logits the top-k saw.
size_t route_scratch_bytes(const moe_config& cfg);
moe_status launch_route(const moe_config& cfg, const void* x, const void* Wr, const float* expert_bias,
                        const float* noise, int* idx, float* w, int* counts, float* ent, void* scratch, int* backup,
                        float* out_logits, int* err, cudaStream_t stream);

// Dispatch: slot-major capacity ranks, offsets, positions, statistics, permute.
size_t dispatch_scratch_bytes(const moe_config& cfg);
// backup: the router's backup experts (MOE_ROUTE_REROUTE: a second pass
// offers the dropped slots to them), else nullptr.  ent (with stats): the
// router's per-token entropies; stats->router_entropy = the mean of their
// finite entries (an exact sum in 2^-40 fixed point), else NaN.
moe_status launch_dispatch(const moe_config& cfg, int C, const int* idx, const void* x, int* kept,
                           int* offsets, int* pos, void* Xp, moe_stats* stats, void* scratch,
                           const int* backup, cudaStream_t stream, const float* ent = nullptr);

// Size of the library's own dispatch scratch (moe_dispatch_static): enough
// for T*k <= 2^20 slots (256 chunks of 4096) at any E <= 1024.
constexpr size_t kStaticDispatchScratchBytes = 256u * 1025u * 4u + 256u * 1024u * 4u + 256u;
// Device address of that scratch on the current device (looked up on the
// first call per device); MOE_ERR_UNSUPPORTED if `need` bytes do not fit.
moe_status static_dispatch_scratch(size_t need, void** ptr);

// Expert parallelism: per-(slot, expert) routed counts [k, E] (zeroed here);
// the dispatch of one rank's slots with global ranks (adj) and send-buffer
// rows (send), both [k, E], and the global capacity C (slot-major priority;
// scratch >= dispatch_ep_scratch_bytes); and a row permutation (scatter:
// dst[map[i]] = src[i]; gather: dst[i] = src[map[i]]; map[i] < 0 skips).
moe_status launch_slot_counts(const moe_config& cfg, const int* idx, int* counts, cudaStream_t stream);
size_t dispatch_ep_scratch_bytes(const moe_config& cfg);
moe_status launch_dispatch_ep(const moe_config& cfg, const int* idx, const void* x, const int* adj, const int* send,
                              int C, int* pos, void* Xsend, void* scratch, cudaStream_t stream);
moe_status launch_permute_rows(const void* src, const int* map, long long n, long long row_bytes, int scatter,
                               void* dst, cudaStream_t stream);

// Combine / un-permute.
moe_status launch_combine(const moe_config& cfg, const void* Yp, const int* pos, const float* w,
                          const void* Sx, void* y, cudaStream_t stream);

// Backward pieces outside the expert GEMMs (backward.cu).
size_t router_wgrad_partial_bytes(const moe_config& cfg);
// Per kept slot (t,j): dYg[pos] = dY[t] (the rows as stored), wp[pos] =
// w[t,j], dot[t,j] = <dY[t], Yp[pos]> (0 when dropped).
moe_status launch_bwd_gather(const moe_config& cfg, const void* dY, const void* Yp, const int* pos, const float* w,
                             void* dYg, float* wp, float* dot, cudaStream_t st);
// imp (E words of 8 bytes) must be zero on entry.  With LayerNorm before
// the router (lnc = 3T floats: mu, A, B per token, else nullptr) dl leaves
// scaled by each token's 1/sqrt(var + eps) and lnc holds the per-token terms
// of the normalisation's backward.
moe_status launch_router_bwd(const moe_config& cfg, const void* x, const void* Wr, const int* idx, const float* w,
                             const int* counts, const float* dot, unsigned long long* imp, float* coef, float* dl,
                             float* lnc, cudaStream_t st);
// Raw softmax weights: the dense logit gradient dlD [T, E] from the forward's
// logits, the saved weights, the dots and the balance coefficients.
moe_status launch_router_bwd_raw(const moe_config& cfg, const float* logits, const int* idx, const float* w,
                                 const float* dot, const float* coef, float* dlD, cudaStream_t st);
// stats->balance_stat of MOE_BALANCE_SWITCH: lambda * sum_e (counts[e]/T) (I[e]/T)
// (imp: E scratch words, zeroed here).
moe_status launch_balance_stat_switch(const moe_config& cfg, const int* idx, const float* w, const int* counts,
                                      unsigned long long* imp, moe_stats* stats, cudaStream_t st);
moe_status launch_router_wgrad(const moe_config& cfg, const void* x, const int* idx, const float* dl,
                               const float* lnc, float* partial, float* dWr, cudaStream_t st);
moe_status launch_bwd_dx(const moe_config& cfg, const float* dXp, const int* pos, const int* idx, const float* dl,
                         const void* Wr, const void* x, const float* lnc, int accumulate, float* dX, cudaStream_t st);
// out[g][n] = sum over group g's rows r of scale[r] * src[r][n] (scale nullable: 1).
moe_status launch_group_colsum(const void* src, long long ld, const int* offsets, int G, int rows, int N,
                               const float* scale, float* out, cudaStream_t st);

// TMA descriptor of a row-major bf16 matrix [rows, inner] with a
// (box_inner x box_rows) box and 128-byte swizzling.
bool make_tma_2d_bf16(CUtensorMap* map, const void* base, long long inner, long long rows, int box_inner,
                      int box_rows);
int device_sm_count(int dev);
// One kernel whose bounded wait runs out (~1 s): kErrSelfTest lands in *err.
moe_status launch_selftest_wait(int* err, cudaStream_t stream);
// Zero a_bytes at a and b_bytes at b (multiples of 4; either may be null)
// with one small kernel on `stream`.
moe_status launch_zero(void* a, size_t a_bytes, void* b, size_t b_bytes, cudaStream_t stream);

}  // namespace moe

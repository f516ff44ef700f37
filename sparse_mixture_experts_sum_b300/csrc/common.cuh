// Device helpers shared by the layer's kernels: bf16 packing, the
// workspace error word, and inline-PTX wrappers for mbarrier, TMA
// (cp.async.bulk.tensor), and the 5th-generation tensor cores (tcgen05 /
// TMEM) of sm_100-family GPUs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// workspace layout: the first 256 bytes are a header.  Word 0 is the error
// word; words 1-2 are the grouped GEMM's dynamic tile scheduler (the next
// tile to hand out, the CTAs finished), which every launch leaves at zero.
// Each entry point zeroes the first kWsZeroBytes before its first launch.
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;
constexpr size_t kWsZeroBytes = 3 * sizeof(int);

// error codes written by bounded waits (nonzero = a wait gave up)
enum : int {
  kErrNone = 0,
  kErrWaitProducer = 0x101,  // TMA producer waited too long for a free stage
  kErrWaitMma = 0x102,       // MMA issuer waited too long for data / accumulator
  kErrWaitEpilogue = 0x103,  // epilogue waited too long for an accumulator
  kErrWaitDrain = 0x104,     // teardown could not drain in-flight copies / MMAs
  kErrSelfTest = 0x1ff,      // the self-test's wait on a barrier that nothing completes
};

// 1 second: every legitimate wait in these kernels is microseconds long
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// small numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);  // a -> low half
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ float gelu_f(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
// d/dz gelu(z) = Phi(z) + z phi(z)
__device__ __forceinline__ float gelu_grad_f(float z) {
  return 0.5f * (1.0f + erff(z * 0.70710678118654752f)) + z * 0.39894228040143268f * expf(-0.5f * z * z);
}
// sigmoid, and d/dz silu(z) = s (1 + z (1 - s))
__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }
// The same two functions with the hardware exponential (__expf) and the fast
// division: for values that are stored as bf16 next (a 2^-9 rounding), the
// few-ulp error of these intrinsics does not show.
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ---------------------------------------------------------------------------
// router top-k, shared by the router kernels and the GEMM's top-k epilogue
// ---------------------------------------------------------------------------
constexpr int MAXK = 8;  // the largest k

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

// Running softmax statistics over a token's logits (any order):
//   m = max l,  Z = sum exp(l - m),  S = sum exp(l - m) (l - m),
// so that p_e = exp(l_e - m) / Z and the entropy -sum p ln p = ln Z - S/Z.
struct SoftStat {
  float m, Z, S;
  __device__ __forceinline__ SoftStat() : m(-INFINITY), Z(0.f), S(0.f) {}
  __device__ __forceinline__ void add(float v) { merge(v, 1.f, 0.f); }
  __device__ __forceinline__ void merge(float m2, float Z2, float S2) {
    if (Z2 == 0.f) return;
    if (Z == 0.f) {
      m = m2;
      Z = Z2;
      S = S2;
      return;
    }
    if (m2 > m) {
      const float sc = expf(m - m2);
      S = sc * (S + (m - m2) * Z) + S2;
      Z = sc * Z + Z2;
      m = m2;
    } else {
      const float sc = expf(m2 - m);
      S += sc * (S2 + (m2 - m) * Z2);
      Z += sc * Z2;
    }
  }
  __device__ __forceinline__ float entropy() const { return logf(Z) - S / Z; }
};

// Weights, indices, entropy and histogram of one token from its sorted
// top-k (v descending, ix).  raw: w_j = p_{ix_j} from the softmax over all
// experts (st holds its statistics); otherwise the softmax over the k
// selected logits.  ent (nullable) receives the token's router entropy (NaN
// for a token with a non-finite logit, which is routed nowhere).
__device__ __forceinline__ void topk_finish(const float (&v)[MAXK], const int (&ix)[MAXK], int k, bool finite,
                                            int t, int* idx, float* w, int* hist, bool raw, const SoftStat& st,
                                            float* ent) {
  if (!finite) {
    for (int j = 0; j < k; ++j) {
      idx[static_cast<size_t>(t) * k + j] = -1;
      w[static_cast<size_t>(t) * k + j] = 0.f;
    }
    if (ent) ent[t] = __int_as_float(0x7fc00000);
    return;
  }
  float ex[MAXK];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j < k) {
      ex[j] = expf(v[j] - (raw ? st.m : v[0]));
      s += ex[j];
    }
  }
  const float inv = 1.0f / (raw ? st.Z : s);
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    if (j < k) {
      idx[static_cast<size_t>(t) * k + j] = ix[j];
      w[static_cast<size_t>(t) * k + j] = ex[j] * inv;
      atomicAdd(&hist[ix[j]], 1);
    }
  }
  if (ent) ent[t] = st.entropy();
}

// ---------------------------------------------------------------------------
// programmatic dependent launch (kernels launched by launch_pdl)
// ---------------------------------------------------------------------------
// Lets the next kernel in the stream be scheduled now; it still waits for
// this one in its own pdl_wait().
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Returns once the preceding kernel in the stream has completed and its
// memory operations are visible (at once for a kernel launched without
// programmatic serialization).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The first statement of every kernel but the GEMM: before any global
// memory access and before any thread can return.  A grid of at most one
// CTA per SM runs in one wave, so it lets the next kernel be scheduled at
// once; a larger grid does not (the next kernel's CTAs would take SM room
// from its later waves while they wait) and triggers as its CTAs exit.
__device__ __forceinline__ void pdl_entry() {
  uint32_t nsm;
  asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
  if (static_cast<unsigned long long>(gridDim.x) * gridDim.y * gridDim.z <= nsm) pdl_trigger();
  pdl_wait();
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 127u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load: box at (c0 = innermost element index, c1 = row) into smem,
// completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 / TMEM
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every previously issued tcgen05.mma of this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 4 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// CTA pairs (a cluster of two CTAs on two SMs sharing one tcgen05 MMA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster: release this CTA's prior writes,
// then wait for everyone (co-scheduled CTAs of one cluster always arrive).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of `p` (a variable of this CTA's shared
// memory) in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Arrive once on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Wait about `ns` nanoseconds (a bounded grace period, not a synchronisation).
__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_ns();
  while (global_ns() - t0 < ns) {
  }
}

// 2-D tiled load whose completion is counted on an mbarrier of the other CTA
// of the pair (bar_cluster: a shared::cluster address from mapa_shared); the
// data lands in this CTA's shared memory.
__device__ __forceinline__ void tma_load_2d_to_peer_bar(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int c0,
                                                        int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

// Pair forms of the TMEM allocation: one warp of each CTA of the pair
// performs them together; the same columns are allocated on both SMs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A * B^T over the CTA pair, issued by one thread of the even
// CTA: A's M rows come half from each CTA's shared memory, B's N columns
// half from each (both at the descriptors' addresses), and each CTA's TMEM
// receives its M/2 rows of D.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once, on the barrier at `bar`'s offset in every CTA of `cta_mask`,
// when the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row (1024-byte) swizzle
// atoms stacked along M/N.  Fields: start address >> 4 (bits 0-13), leading
// byte offset (unused for swizzled K-major, 0), stride byte offset = 1024 >> 4
// (bits 32-45), descriptor version 1 (bit 46), swizzle mode 2 = 128B
// (bits 61-63).  The tile base must be 1024-byte aligned; advancing along K
// inside the 128-byte row adds the byte offset to the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory matrix descriptor for an MN-major operand tile written by
// TMA with 128-byte swizzling: each K row holds 64 consecutive M (or N)
// elements in one 128-byte line; 8 K rows form a 1024-byte swizzle atom;
// the tile stores 64-element MN blocks of 64 K rows (8 KB each) one after
// another.  Leading byte offset = 8192 (bits 16-29, between MN blocks),
// stride byte offset = 1024 (bits 32-45, between 8-row K groups), version 1
// (bit 46), swizzle mode 2 = 128B (bits 61-63).  Advancing K by 16 rows
// adds 2048 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(8192u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A bf16 (bits 7-9 = 1), B bf16 (bits 10-12 = 1), A major (bit 15) and B
// major (bit 16): 0 = K-major, 1 = MN-major; N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn = 0, int b_mn = 0) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn & 1) << 15) |
         (static_cast<uint32_t>(b_mn & 1) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace moe

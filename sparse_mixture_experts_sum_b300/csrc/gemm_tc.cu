// Grouped expert GEMM on the sm_103a tensor cores (tcgen05 + TMEM, fed by TMA).
//
// out[r, :] = act( A[r, :] . B_g^T )   for every group g and row r of g,
// where the rows of group g are [offsets[g], offsets[g+1]) of the
// expert-contiguous activation matrix A, and B_g is group g's weight block.
// This is the expert loop of the MoE layer: "[P2] 4.2 / [P3] 3.3 Linear ->
// GELU -> Linear" per expert, with all experts' weights in one contiguous
// tensor ([P2] 4.1 expert fusion) sliced by the group index.
//
// Design (one persistent CTA per SM, 192 threads):
//   warp 0  : TMA producer -- A tile 128x64 and B tile 256x64 (bf16, 128-byte
//             swizzle) per k-block into a 4-stage shared-memory ring;
//   warp 1  : owns 512 TMEM columns; one lane issues tcgen05.mma
//             (M=128, N=256, K=16) into one of two 128x256 fp32 accumulators;
//   warps 2-5: epilogue -- tcgen05.ld the accumulator, apply the activation,
//             round to bf16, store the rows that belong to the group.
// Accumulators are double-buffered so the epilogue of tile i overlaps the
// MMAs of tile i+1.  The tile list (group, n-tile, m-tile) is derived on the
// device from offsets[], so no host round-trip is needed for the
// data-dependent per-expert row counts; m is the fastest index so that the
// CTAs running at the same time share each weight tile through L2.
//
// Modes:
//   SwiGLU: B rows [0,128) come from W1 (gate) and [128,256) from W3 (up) at
//           the same 128 output columns; out = silu(gate) * up.
//   GeLU  : out = gelu(acc + bias);  Plain: out = acc (+ bias).
//
// Every wait on a barrier is bounded (1 s); on expiry the kernel records an
// error code in the workspace error word, drains its in-flight copies and
// MMAs (again bounded), frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_TILE_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_HALF_BYTES = 128 * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_TILE_BYTES + 2 * B_HALF_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_GROUPS = 1024;

struct __align__(8) Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int grp_row[MAX_GROUPS + 1];     // first row of each group (+ end)
  int tile_start[MAX_GROUPS + 1];  // first tile of each group (+ total)
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + sizeof(Ctl);

struct Tile {
  int g, n, m;
};

__device__ __forceinline__ Tile tile_coords(const Ctl& c, int G, int n_tiles, int tile) {
  int lo = 0, hi = G;  // largest g with tile_start[g] <= tile (always a non-empty group)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  const int local = tile - c.tile_start[lo];
  const int mt = (c.tile_start[lo + 1] - c.tile_start[lo]) / n_tiles;
  Tile t;
  t.g = lo;
  t.n = local / mt;
  t.m = local - t.n * mt;
  return t;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                       const __grid_constant__ CUtensorMap mapB1, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl& c = *reinterpret_cast<Ctl*>(tiles + static_cast<size_t>(STAGES) * STAGE_BYTES);
  volatile int* abort_flag = &c.abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const bool swiglu = p.mode == kModeSwiGLU;
  const int n_tiles = swiglu ? (p.N + 127) / 128 : (p.N + BN - 1) / BN;
  const int nk = (p.K + BK - 1) / BK;

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c.tmem_full[a], 1);
      mbar_init(&c.tmem_empty[a], 128);
    }
    mbar_init(&c.drain, 1);
    c.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB0);
    tma_prefetch_desc(&mapB1);
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    // per-group tile counts -> exclusive prefix (one warp, 32 groups a step)
    int carry = 0;
    for (int g0 = 0; g0 <= G; g0 += 32) {
      const int g = g0 + lane;
      int row = 0;
      if (g <= G) row = p.offsets ? p.offsets[g] : (g == 0 ? 0 : p.rows);
      int tiles_g = 0;
      if (g < G) {
        const int r1 = p.offsets ? p.offsets[g + 1] : p.rows;
        const int rows = r1 - row;
        tiles_g = rows > 0 ? ((rows + BM - 1) / BM) * n_tiles : 0;
      }
      int incl = tiles_g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g <= G) {
        c.grp_row[g] = row;
        c.tile_start[g] = carry + incl - tiles_g;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) c.total_tiles = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int total = c.total_tiles;
  const uint32_t tmem_base = c.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
        const Tile t = tile_coords(c, G, n_tiles, tile);
        const int a_row = c.grp_row[t.g] + t.m * BM;
        int b_row0, b_row1;
        const CUtensorMap* mb1;
        if (swiglu) {
          b_row0 = t.g * p.N + t.n * 128;
          b_row1 = b_row0;
          mb1 = &mapB1;
        } else {
          b_row0 = t.g * p.N + t.n * BN;
          b_row1 = b_row0 + 128;
          mb1 = &mapB0;
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&c.empty[s], ph ^ 1u)) {
            record_error(p.err, kErrWaitProducer);
            *abort_flag = 1;
            break;
          }
          uint8_t* sa = tiles + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&c.full[s], STAGE_BYTES);
          tma_load_2d(sa, &mapA, &c.full[s], kb * BK, a_row);
          tma_load_2d(sa + A_TILE_BYTES, &mapB0, &c.full[s], kb * BK, b_row0);
          tma_load_2d(sa + A_TILE_BYTES + B_HALF_BYTES, mb1, &c.full[s], kb * BK, b_row1);
        }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA goes away
        const uint32_t n = it < STAGES ? it : STAGES;
        for (uint32_t q = it - n; q < it; ++q) {
          if (!mbar_wait(&c.full[q % STAGES], (q / STAGES) & 1u)) record_error(p.err, kErrWaitDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
      uint32_t it = 0, local = 0;
      bool issued = false;
      for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++local) {
        const uint32_t acc = local & 1u;
        const uint32_t aph = (local >> 1) & 1u;
        if (!mbar_wait(&c.tmem_empty[acc], aph ^ 1u)) {
          record_error(p.err, kErrWaitMma);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&c.full[s], ph)) {
            record_error(p.err, kErrWaitMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(tiles + s * STAGE_BYTES);
          const uint32_t b_base = a_base + A_TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sw128_kmajor_desc(a_base + kk * 32);
            const uint64_t bd = sw128_kmajor_desc(b_base + kk * 32);
            tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(&c.empty[s]);
        }
        if (!ok) break;
        tc_commit(&c.tmem_full[acc]);
      }
      if (*abort_flag && issued) {
        tc_commit(&c.drain);
        if (!mbar_wait(&c.drain, 0)) record_error(p.err, kErrWaitDrain);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter+32)
    uint32_t local = 0;
    for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++local) {
      const Tile t = tile_coords(c, G, n_tiles, tile);
      const long long row_end = min(static_cast<long long>(c.grp_row[t.g + 1]), p.rows_alloc);
      const uint32_t acc = local & 1u;
      const uint32_t aph = (local >> 1) & 1u;
      if (!mbar_wait(&c.tmem_full[acc], aph)) {
        record_error(p.err, kErrWaitEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int row = c.grp_row[t.g] + t.m * BM + quarter * 32 + lane;
      const bool valid = row < row_end;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      bf16* orow = static_cast<bf16*>(p.out) + static_cast<size_t>(row) * p.N;
      if (swiglu) {
        const int col0 = t.n * 128;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t gr[32], ur[32];
          tmem_ld_32x32b_x32(taddr + cc * 32, gr);
          tmem_ld_32x32b_x32(taddr + 128 + cc * 32, ur);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
            const float u0 = __uint_as_float(ur[2 * i]), u1 = __uint_as_float(ur[2 * i + 1]);
            pk[i] = pack_bf16(silu_f(g0) * u0, silu_f(g1) * u1);
          }
          if (valid) {
            const int col = col0 + cc * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (col + q * 8 + 8 <= p.N)
                *reinterpret_cast<uint4*>(orow + col + q * 8) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
      } else {
        const int col0 = t.n * BN;
        const bool gelu = p.mode == kModeGeLU;
        const bf16* brow = p.bias ? static_cast<const bf16*>(p.bias) + static_cast<size_t>(t.g) * p.N : nullptr;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + cc * 32, r);
          tmem_ld_wait();
          const int col = col0 + cc * 32;
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float v0 = __uint_as_float(r[2 * i]), v1 = __uint_as_float(r[2 * i + 1]);
            if (brow) {
              const int c0 = col + 2 * i;
              if (c0 < p.N) v0 += __bfloat162float(brow[c0]);
              if (c0 + 1 < p.N) v1 += __bfloat162float(brow[c0 + 1]);
            }
            if (gelu) {
              v0 = gelu_f(v0);
              v1 = gelu_f(v1);
            }
            pk[i] = pack_bf16(v0, v1);
          }
          if (valid) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (col + q * 8 + 8 <= p.N)
                *reinterpret_cast<uint4*>(orow + col + q * 8) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c.tmem_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
moe_status launch_grouped_gemm_tc(const GemmParams& p_in, const void* A, long long a_rows, const void* B0,
                                  const void* B1, long long b_rows, cudaStream_t stream) {
  GemmParams p = p_in;
  p.rows_alloc = a_rows;
  if (p.G < 1 || p.G > MAX_GROUPS || p.N < 8 || p.K < 8 || (p.N % 8) || (p.K % 8)) return MOE_ERR_UNSUPPORTED;
  if (a_rows <= 0) return MOE_OK;
  CUtensorMap mA, mB0, mB1;
  if (!make_tma_2d_bf16(&mA, A, p.K, a_rows, BK, BM)) return MOE_ERR_CUDA;
  if (!make_tma_2d_bf16(&mB0, B0, p.K, b_rows, BK, 128)) return MOE_ERR_CUDA;
  if (!make_tma_2d_bf16(&mB1, B1 ? B1 : B0, p.K, b_rows, BK, 128)) return MOE_ERR_CUDA;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  static thread_local int attr_set_dev = -1;
  if (attr_set_dev != dev) {
    if (cudaFuncSetAttribute(grouped_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set_dev = dev;
  }
  const bool swiglu = p.mode == kModeSwiGLU;
  const long long n_tiles = swiglu ? (p.N + 127) / 128 : (p.N + BN - 1) / BN;
  const long long rows_bound = p.offsets ? a_rows : p.rows;
  const long long m_tiles_bound = (rows_bound + BM - 1) / BM + (p.offsets ? p.G : 0);
  long long grid = m_tiles_bound * n_tiles;
  if (grid > sms) grid = sms;
  if (grid < 1) grid = 1;
  grouped_gemm_tc_kernel<<<static_cast<unsigned>(grid), NUM_THREADS, kSmemBytes, stream>>>(mA, mB0, mB1, p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// Grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM, fed by TMA).
//
// The expert loop of the MoE layer -- "[P2] 4.2 / [P3] 3.3 Linear -> GELU ->
// Linear" per expert, with all experts' weights in one contiguous tensor
// ([P2] 4.1 expert fusion) sliced by the group index -- and the same loop's
// backward ([P1] 3.3: gradients flow back to the chosen experts).  Group g
// (an expert) owns rows [offsets[g], offsets[g+1]) of the expert-contiguous
// activation matrices.  Three operand geometries share one kernel:
//
//   Fwd   out[r,:] = act( A[r,:] . B_g^T )   A [rows,K], B_g [N,K]  (K-major)
//   Dgrad out[r,:] = act( A[r,:] . B_g )     A [rows,K] K-major, B_g [K,N] (MN-major)
//   Wgrad out_g    = A_g^T . B_g             A_g [rows_g,M], B_g [rows_g,N] (both MN-major),
//                                             contraction over the group's rows
//
// Dgrad reads the weights in their stored layout (W2 [E,d,h] as B_g [K=d, N=h];
// W1/W3 [E,h,d] as [K=h, N=d]) through MN-major shared-memory descriptors, so
// no transposed copy of any weight is made.  Its K range may be split
// between two weight tensors (dXp = dA.W1 + dB.W3 with A = [dA | dB]).
//
// Design (one persistent CTA per SM; the 128-row tile shown, TileCfg below
// has the 256-row and CTA-pair forms):
//   warp 0  : TMA producer -- A tile 128x64 and B tile 256x64 (bf16, 128-byte
//             swizzle) per k-block into a 4-stage shared-memory ring;
//   warp 1  : owns 512 TMEM columns; one lane issues tcgen05.mma
//             (M=128, N=256, K=16) into one of two 128x256 fp32 accumulators;
//             for Wgrad the warp first clears the rows of a group's last
//             k-block that belong to the next group;
//   warps 2-5: epilogue -- tcgen05.ld the accumulator, apply the epilogue
//             mode, store the rows / columns inside the output.
// Accumulators are double-buffered so the epilogue of tile i overlaps the
// MMAs of tile i+1.  Every launch is a programmatic dependent launch: the
// barrier and TMEM set-up runs before griddepcontrol.wait, and the producer
// lets the next kernel be scheduled once its last load is issued.  The tile
// list is derived on the device from offsets[],
// so no host round-trip is needed for the data-dependent per-expert row
// counts.  Fwd/Dgrad tiles run m fastest, so the CTAs running together share
// each weight tile through L2; Wgrad tiles run along the smaller of M and N
// fastest, so that operand stays in L2 while the other streams once.
//
// Epilogue modes (GemmMode): plain (+bias), SwiGLU (B rows [0,128) from W1
// and [128,256) from W3 at the same 128 output columns: silu(gate) * up),
// GeLU (gelu(acc + bias)), the backward of both activations, and the
// router's top-k (each thread takes its token's logits from TMEM).  The
// forward saves the pre-activations in fp32; the backward reads them, scales
// the accumulator by the row's routing weight (so the GEMM contracts the
// upstream gradient rows as stored, not a rounded weighted copy) and can
// write the weighted activation s * act(z) for the W2 gradient.
//
// Every wait on a barrier is bounded (1 s); on expiry the kernel records an
// error code in the workspace error word, drains its in-flight copies and
// MMAs (again bounded), frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BN = 256;
constexpr int BK = 64;
constexpr int B_HALF_BYTES = 128 * BK * 2;   // 16 KB
constexpr int MN_BLOCK_BYTES = 64 * BK * 2;  // one 64-wide MN block of 64 K rows: 8 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_GROUPS = 1024;
constexpr int SCHED_DEPTH = 8;  // tiles the producer may hand out ahead of the last epilogue warp

// Tile shape per BM (output rows per CTA) and PAIR:
//   BM = 128: 4-stage ring of 48 KB, two 128x256 accumulators (the epilogue
//             of one tile overlaps the MMAs of the next), 4 epilogue warps;
//   BM = 256: 3-stage ring of 64 KB, one 256x256 accumulator (two M=128
//             MMAs per K step share the B tile: 2x the MACs per byte of
//             shared memory filled), 8 epilogue warps;
//   PAIR (BM = 128 per CTA, Fwd): a cluster of two CTAs on two SMs runs
//             256-row tiles with one M=256 tcgen05 MMA per K step
//             (cta_group::2).  Each CTA stages its own 128 A rows and half of
//             the 256 B rows (32 KB per stage, 6 stages), and keeps two
//             128x256 accumulators for its rows: the B bytes staged per MAC
//             halve against BM = 128, and the epilogue still overlaps.  Both
//             CTAs' copies of a stage complete on the even CTA's barrier.
template <int BM_, bool PAIR = false>
struct TileCfg {
  static constexpr int BM = BM_;                        // output rows per CTA
  static constexpr int TILE_M = PAIR ? 2 * BM_ : BM_;   // output rows per tile
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = PAIR ? B_HALF_BYTES : 2 * B_HALF_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = PAIR ? 6 : (BM == 128 ? 4 : 3);
  static constexpr int NACC = BM == 128 ? 2 : 1;
  static constexpr int EPI_WARPS = BM / 32;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static_assert(!PAIR || BM_ == 128, "pair tiles are two 128-row halves");
};

template <int STAGES>
struct __align__(8) Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  // dynamic schedule: the producer writes the tile of its j-th turn to
  // sched_tile[j % SCHED_DEPTH] and arrives on sched_full; the MMA warp and
  // each epilogue warp read it and arrive on sched_empty
  uint64_t sched_full[SCHED_DEPTH];
  uint64_t sched_empty[SCHED_DEPTH];
  int sched_tile[SCHED_DEPTH];
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int x_tile0;  // first tile of the extra group (= tiles of the routed groups)
  int grp_row[MAX_GROUPS + 1];     // first row of each group (+ end)
  int tile_start[MAX_GROUPS + 1];  // first tile of each group (+ total)
  int hist[256];                   // kModeRouteTopK: this CTA's selections per expert
};

// A Wgrad epilogue warp stages 32 rows x 64 bytes of output here (see
// warp_store_rows64), after the control block.
constexpr int STAGE_OUT_BYTES = 32 * 64;

template <int KIND, int BM_, bool PAIR = false>
constexpr size_t smem_bytes() {
  return 1024 + static_cast<size_t>(TileCfg<BM_, PAIR>::STAGES) * TileCfg<BM_, PAIR>::STAGE_BYTES +
         (sizeof(Ctl<TileCfg<BM_, PAIR>::STAGES>) + 15) / 16 * 16 +
         (KIND == kKindWgrad ? static_cast<size_t>(TileCfg<BM_, PAIR>::EPI_WARPS) * STAGE_OUT_BYTES : 0);
}

struct Tile {
  int g, n, m;
};

// Tile index -> (group, n-tile, m-tile).  Fwd/Dgrad: a group has
// ceil(rows/BM) m-tiles per n-tile, m fastest, so the CTAs running together
// share each weight tile through L2.  Wgrad: every group has m_tiles x
// n_tiles tiles, n fastest when n_fast.  The extra group's X tiles (the
// shared expert: many rows on one weight set, so bound by the tensor cores
// where the routed groups stream weights) are spread evenly through the
// schedule of N tiles: slot s holds extra tile floor(s X / N) when that
// count steps at s, else routed tile s - floor(s X / N).  They run n
// fastest: the shared weights are small enough to stay in L2, while its T
// input rows are not, so each block of rows is read once for all n-tiles.
template <int KIND, int BM, typename C>
__device__ __forceinline__ Tile tile_coords(const C& c, int G, int n_tiles, int m_tiles, bool n_fast, int tile) {
  if (KIND == kKindFwd && c.total_tiles > c.x_tile0) {
    const long long NT = c.total_tiles, XT = NT - c.x_tile0;
    const long long before = static_cast<long long>(tile) * XT / NT;
    if ((static_cast<long long>(tile) + 1) * XT / NT > before) {
      const int local = static_cast<int>(before);
      Tile t;
      t.g = G;
      t.m = local / n_tiles;
      t.n = local - t.m * n_tiles;
      return t;
    }
    tile -= static_cast<int>(before);
  }
  int lo = 0, hi = G;  // largest g with tile_start[g] <= tile (a group with tiles)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  const int local = tile - c.tile_start[lo];
  Tile t;
  t.g = lo;
  if (KIND == kKindWgrad) {
    if (n_fast) {
      t.m = local / n_tiles;
      t.n = local - t.m * n_tiles;
    } else {
      t.n = local / m_tiles;
      t.m = local - t.n * m_tiles;
    }
  } else {
    const int mt = (c.tile_start[lo + 1] - c.tile_start[lo]) / n_tiles;
    t.n = local / mt;
    t.m = local - t.n * mt;
  }
  return t;
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, int col, int N, const uint32_t (&pk)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (col + q * 8 + 8 <= N)
      *reinterpret_cast<uint4*>(dst + col + q * 8) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
}

__device__ __forceinline__ void store_f32x32(float* dst, int col, int N, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (col + q * 4 + 4 <= N)
      *reinterpret_cast<float4*>(dst + col + q * 4) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// The warp's 32 rows (one per lane) each hand 64 bytes (words w(0..15)) to dst, this
// lane's destination (nullptr: the row is not stored); the first `bytes` of
// them (a multiple of 16, the same in every lane) are stored.  The rows go
// through the warp's 2 KB of shared memory, so that each store instruction
// writes 8 rows of 64 contiguous bytes rather than 16 bytes in each of 32
// rows: a quarter of the L1 wavefronts, and whole 32-byte sectors.  Used for
// the weight gradients (fp32).  In the forward kernels the same staging
// raised register use past the 256-row tile's ceiling (spills), and the
// small prefill's layer went from 0.176 to 0.182-0.184 ms.  Granule
// q of row r sits in slot q ^ ((r >> 1) & 3), so neither the row-wise
// writes nor the column-wise reads conflict on banks.  Warp-collective.
template <typename W>
__device__ __forceinline__ void warp_store_rows64(uint4* stage, const W& w, void* dst, int bytes, int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    stage[lane * 4 + (q ^ ((lane >> 1) & 3))] = make_uint4(w(4 * q), w(4 * q + 1), w(4 * q + 2), w(4 * q + 3));
  __syncwarp();
  const int q = lane & 3;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2);
    uint8_t* d = reinterpret_cast<uint8_t*>(
        __shfl_sync(0xffffffffu, static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(dst)), r));
    if (d && q * 16 < bytes) *reinterpret_cast<uint4*>(d + q * 16) = stage[r * 4 + (q ^ ((r >> 1) & 3))];
  }
  __syncwarp();
}

// 32 fp32 of this lane's row, in two 16-column halves; warp-collective
__device__ __forceinline__ void warp_store_f32x32(uint4* stage, float* rowp, int col, int N, const float (&v)[32],
                                                  int lane) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int c = col + 16 * hf;
    warp_store_rows64(stage, [&](int i) { return __float_as_uint(v[16 * hf + i]); }, rowp ? rowp + c : nullptr,
                      min(64, (N - c) * 4), lane);
  }
}

// 32 consecutive fp32 (16-byte aligned); groups of 4 past N read as 0.
__device__ __forceinline__ void load_f32x32(const float* src, int col, int N, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col + q * 4 + 4 <= N) f = *reinterpret_cast<const float4*>(src + col + q * 4);
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
}

template <int KIND, int BM_, bool PAIR>
__global__ void __launch_bounds__(TileCfg<BM_, PAIR>::THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                       const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapXA,
                       const __grid_constant__ CUtensorMap mapXB0, const __grid_constant__ CUtensorMap mapXB1,
                       const GemmParams p) {
  static_assert(!PAIR || KIND == kKindFwd, "pair tiles are for the forward geometry");
  using TC = TileCfg<BM_, PAIR>;
  constexpr int BM = TC::BM;
  constexpr int TM = TC::TILE_M;
  constexpr int STAGES = TC::STAGES;
  constexpr int STAGE_BYTES = TC::STAGE_BYTES;
  constexpr int A_TILE_BYTES = TC::A_BYTES;
  constexpr int NACC = TC::NACC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl<STAGES>& c = *reinterpret_cast<Ctl<STAGES>*>(tiles + static_cast<size_t>(STAGES) * STAGE_BYTES);
  uint4* const stage_out = reinterpret_cast<uint4*>(tiles + static_cast<size_t>(STAGES) * STAGE_BYTES +
                                                    (sizeof(Ctl<STAGES>) + 15) / 16 * 16);
  volatile int* abort_flag = &c.abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const bool swiglu_fwd = KIND == kKindFwd && p.mode == kModeSwiGLU;
  const int n_tiles = swiglu_fwd ? (p.N + 127) / 128 : (p.N + BN - 1) / BN;
  const int m_tiles_w = KIND == kKindWgrad ? (p.M + BM - 1) / BM : 1;
  const bool n_fast = KIND == kKindWgrad && p.M > p.N;
  const int nk_fixed = (p.K + BK - 1) / BK;
  // PAIR: this CTA's rank in its cluster (0 issues the MMAs) and the tile
  // stream of the cluster; otherwise one CTA per tile stream
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  // ---------------- set-up ----------------
  // the barriers, TMEM and descriptor prefetches below touch no global
  // memory, so they overlap the preceding kernel's tail; pdl_wait() comes
  // before the first read
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c.tmem_full[a], 1);
      // PAIR: one arrival per epilogue warp of both CTAs; else every thread
      mbar_init(&c.tmem_empty[a], PAIR ? 2 * TC::EPI_WARPS : 32 * TC::EPI_WARPS);
    }
    mbar_init(&c.drain, 1);
    for (int q = 0; q < SCHED_DEPTH; ++q) {
      mbar_init(&c.sched_full[q], 1);
      mbar_init(&c.sched_empty[q], 1 + TC::EPI_WARPS);
    }
    c.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB0);
    tma_prefetch_desc(&mapB1);
  }
  if (KIND == kKindFwd && p.mode == kModeRouteTopK)
    for (int i = threadIdx.x; i < 256; i += blockDim.x) c.hist[i] = 0;
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&c.tmem_base, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&c.tmem_base, TMEM_COLS);
      tmem_relinquish();
    }
  }
  pdl_wait();
  if (warp == 2) {
    // per-group tile counts -> exclusive prefix (one warp, 32 groups a step)
    int carry = 0;
    for (int g0 = 0; g0 <= G; g0 += 32) {
      const int g = g0 + lane;
      int row = 0;
      if (g <= G) row = p.offsets ? p.offsets[g] : (g == 0 ? 0 : p.rows);
      int tiles_g = 0;
      if (g < G) {
        if (KIND == kKindWgrad) {
          tiles_g = m_tiles_w * n_tiles;
        } else {
          const int r1 = p.offsets ? p.offsets[g + 1] : p.rows;
          const int rows = r1 - row;
          tiles_g = rows > 0 ? ((rows + TM - 1) / TM) * n_tiles : 0;
        }
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
    if (lane == 0) {
      c.x_tile0 = carry;
      c.total_tiles = carry + (KIND == kKindFwd && p.xrows > 0 ? ((p.xrows + TM - 1) / TM) * n_tiles : 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  // PAIR: both CTAs' barriers are initialised before either signals the other's
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();

  const int total = c.total_tiles;
  const uint32_t tmem_base = c.tmem_base;
  // Dynamic schedule, for the launches whose tiles differ in cost (256-row
  // tiles, where a group's last tile may be a half tile; Wgrad, where a
  // tile's k-blocks are its group's rows), given the scheduler words: a
  // CTA's first tile is its block index, and each further one comes from a
  // counter in the workspace (tiles gridDim.x, gridDim.x + 1, ... in order).
  // A CTA whose tiles ran short takes more of them, while the tiles in
  // flight at any time stay neighbours in the order above and share their
  // weight tiles through L2.  Otherwise CTA b runs tiles b, b + tstep, ...
  // (equal tiles gain nothing from the counter's round trips).
  const bool dyn = !PAIR && (BM == 256 || KIND == kKindWgrad) && p.sched != nullptr;
  // a consumer warp's tile for its j-th turn (warp-uniform); total once the
  // schedule has ended, or when the wait gave up (the abort flag is then set)
  auto take_tile = [&](uint32_t j, int err_code) -> int {
    if (!dyn) return tile0 + static_cast<int>(j) * tstep;
    const uint32_t q = j % SCHED_DEPTH;
    int tile = total;
    if (lane == 0) {
      if (mbar_wait(&c.sched_full[q], (j / SCHED_DEPTH) & 1u)) {
        tile = c.sched_tile[q];
        mbar_arrive(&c.sched_empty[q]);
      } else {
        record_error(p.err, err_code);
        *abort_flag = 1;
      }
    }
    return __shfl_sync(0xffffffffu, tile, 0);
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      int next = tile0;
      for (uint32_t j = 0; !*abort_flag; ++j) {
        const int tile = next < total ? next : total;
        if (dyn) {
          // fetch the tile after this one now, so that its latency hides
          // behind this tile's loads; then hand this one to the consumers
          if (tile < total) next = static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
          const uint32_t q = j % SCHED_DEPTH;
          if (!mbar_wait(&c.sched_empty[q], ((j / SCHED_DEPTH) & 1u) ^ 1u)) {
            record_error(p.err, kErrWaitProducer);
            *abort_flag = 1;
            break;
          }
          c.sched_tile[q] = tile;
          mbar_arrive(&c.sched_full[q]);
        } else {
          next = tile + tstep;
        }
        if (tile >= total) break;
        const Tile t = tile_coords<KIND, TM>(c, G, n_tiles, m_tiles_w, n_fast, tile);
        const bool xg = KIND == kKindFwd && t.g == G;  // the extra group
        const int grow = xg ? 0 : c.grp_row[t.g];
        // Wgrad: k-blocks of the group's rows (twice over with a hi/lo B pair)
        const int nk1 = KIND == kKindWgrad ? (c.grp_row[t.g + 1] - grow + BK - 1) / BK : nk_fixed;
        const int nk = KIND == kKindWgrad && p.b_lo ? 2 * nk1 : nk1;
        // a 256-row tile holding at most 128 of its group's rows stages and
        // multiplies only its first half
        const int gend_p = xg ? p.xrows : c.grp_row[t.g + 1];
        const bool half_tile = KIND != kKindWgrad && !PAIR && BM == 256 && gend_p - (grow + t.m * TM) <= 128;
        // every box of k-block kb, handed to emit(dst offset in the stage, map, x, y)
        auto boxes = [&](int kb, auto&& emit) {
          if (KIND == kKindFwd) {
            const CUtensorMap* ma = xg ? &mapXA : &mapA;
            const CUtensorMap* mb0 = xg ? &mapXB0 : &mapB0;
            const CUtensorMap* mb1 = xg ? &mapXB1 : &mapB1;
            const int g_row = xg ? 0 : t.g * p.N;
            // this CTA's rows of the tile, 128-row boxes (PAIR: the odd CTA
            // stages the upper half; BM = 256: two boxes, one for a half tile)
            const int a_row = grow + t.m * TM + static_cast<int>(crank) * (PAIR ? BM : 0);
            emit(0, ma, kb * BK, a_row);
            if (BM == 256 && !half_tile) emit(16384, ma, kb * BK, a_row + 128);
            if constexpr (PAIR) {
              // this CTA's half of the 256 B rows: SwiGLU W1 (even) or W3
              // (odd) rows of the tile's 128 hidden units; plain rows
              // [128 crank, 128 crank + 128) of the tile's 256 columns
              if (swiglu_fwd)
                emit(A_TILE_BYTES, crank ? mb1 : mb0, kb * BK, g_row + t.n * 128);
              else
                emit(A_TILE_BYTES, mb0, kb * BK, g_row + t.n * BN + static_cast<int>(crank) * 128);
            } else if (swiglu_fwd) {
              const int b_row = g_row + t.n * 128;
              emit(A_TILE_BYTES, mb0, kb * BK, b_row);
              emit(A_TILE_BYTES + B_HALF_BYTES, mb1, kb * BK, b_row);
            } else {
              const int b_row = g_row + t.n * BN;
              emit(A_TILE_BYTES, mb0, kb * BK, b_row);
              emit(A_TILE_BYTES + B_HALF_BYTES, mb0, kb * BK, b_row + 128);
            }
          } else if (KIND == kKindDgrad) {
            emit(0, &mapA, kb * BK, grow + t.m * BM);
            if (BM == 256 && !half_tile) emit(16384, &mapA, kb * BK, grow + t.m * BM + 128);
            int k0 = kb * BK;
            const CUtensorMap* mb = &mapB0;
            const int kb_rows = p.k_split ? p.k_split : p.K;
            if (p.k_split && k0 >= p.k_split) {
              mb = &mapB1;
              k0 -= p.k_split;
            }
            const int y = t.g * kb_rows + k0;
#pragma unroll
            for (int i = 0; i < 4; ++i) emit(A_TILE_BYTES + i * MN_BLOCK_BYTES, mb, t.n * BN + 64 * i, y);
          } else {
            const bool lo = kb >= nk1;  // second pass: the B1 (lo) rows
            const int y = grow + (lo ? kb - nk1 : kb) * BK;
            const CUtensorMap* mb = lo ? &mapB1 : &mapB0;
#pragma unroll
            for (int i = 0; i < BM / 64; ++i) emit(i * MN_BLOCK_BYTES, &mapA, t.m * BM + 64 * i, y);
#pragma unroll
            for (int i = 0; i < 4; ++i) emit(A_TILE_BYTES + i * MN_BLOCK_BYTES, mb, t.n * BN + 64 * i, y);
          }
        };
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          // (PAIR: the even CTA's commit frees the stage on both SMs)
          if (!mbar_wait(&c.empty[s], ph ^ 1u)) {
            record_error(p.err, kErrWaitProducer);
            *abort_flag = 1;
            break;
          }
          uint8_t* st_base = tiles + s * STAGE_BYTES;
          if (PAIR && crank == 1) {
            // the odd CTA's half of the stage counts on the even CTA's
            // barrier, which expects both halves
            const uint32_t bar0 = mapa_shared(&c.full[s], 0);
            boxes(kb, [&](int off, const CUtensorMap* m, int x, int y) {
              tma_load_2d_to_peer_bar(st_base + off, m, bar0, x, y);
            });
          } else {
            mbar_arrive_expect_tx(&c.full[s], PAIR ? 2 * STAGE_BYTES : STAGE_BYTES - (half_tile ? 16384 : 0));
            boxes(kb, [&](int off, const CUtensorMap* m, int x, int y) { tma_load_2d(st_base + off, m, &c.full[s], x, y); });
          }
        }
      }
      if (dyn) {
        // this CTA fetches no more tiles (on every way out of the loop): the
        // last CTA to get here leaves the scheduler words at zero for the
        // next launch, while its MMAs and epilogue still run
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
          atomicExch(p.sched, 0);
          atomicExch(p.sched + 1, 0);
        }
      }
      // every load of this CTA is issued: the next kernel in the stream may
      // be scheduled (its CTAs wait in pdl_wait() until this grid completes)
      pdl_trigger();
      if (*abort_flag && PAIR && crank == 1) {
        // the copies already issued count on the other CTA's barriers, which
        // this CTA cannot wait on: give them a bounded grace period to land
        spin_ns(100000);
      } else if (*abort_flag) {
        // let the copies already issued land before the CTA goes away
        const uint32_t n = it < STAGES ? it : STAGES;
        for (uint32_t q = it - n; q < it; ++q) {
          if (!mbar_wait(&c.full[q % STAGES], (q / STAGES) & 1u)) record_error(p.err, kErrWaitDrain);
        }
      }
    }
  } else if (warp == 1 && PAIR) {
    // ---------------- PAIR: MMA issuer (even CTA only) ----------------
    // The even CTA waits until both CTAs' halves of a stage have landed (one
    // barrier counts both), issues one M=256 x N=256 x K=16 MMA per K step
    // over both, and commits with a multicast so that both CTAs see the
    // stage freed and the accumulator full.
    const uint32_t IDESC2 = idesc_bf16_f32(256, BN, 0, 0);
    uint32_t it = 0, local = 0;
    bool issued = false;
    for (int tile = tile0; tile < total && crank == 0; tile += tstep, ++local) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const uint32_t acc = local % NACC;
      const uint32_t aph = (local / NACC) & 1u;
      // both CTAs' epilogues have drained this accumulator
      bool ok = lane == 0 ? mbar_wait(&c.tmem_empty[acc], aph ^ 1u) : true;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) record_error(p.err, kErrWaitMma);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < nk_fixed; ++kb, ++it) {
        const uint32_t s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        bool okf = lane == 0 ? mbar_wait(&c.full[s], ph) : true;
        okf = __shfl_sync(0xffffffffu, okf, 0);
        if (!okf) {
          if (lane == 0) record_error(p.err, kErrWaitMma);
          *abort_flag = 1;
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_base = smem_u32(tiles + s * STAGE_BYTES);
          const uint32_t b_base = a_base + A_TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16_pair(d_tmem, sw128_kmajor_desc(a_base + kk * 32), sw128_kmajor_desc(b_base + kk * 32),
                             IDESC2, (kb | kk) != 0 ? 1u : 0u);
          tc_commit_pair_mc(&c.empty[s], 0x3);
        }
        __syncwarp();
        issued = true;
      }
      if (!ok) break;
      if (lane == 0) tc_commit_pair_mc(&c.tmem_full[acc], 0x3);
      __syncwarp();
    }
    if (*abort_flag && issued && crank == 0 && lane == 0) {
      tc_commit_pair_mc(&c.drain, 0x1);
      if (!mbar_wait(&c.drain, 0)) record_error(p.err, kErrWaitDrain);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (lane 0 issues; the warp clears Wgrad tails) ----------------
    // every MMA is M=128 x N=256 (a BM=256 tile issues two per K step); a
    // problem narrower than one tile (e.g. the router's N = E logits) uses
    // N = its width rounded up to 16, so no MMA work is spent on columns
    // that are never stored
    const int n_mma = (p.N < BN && !swiglu_fwd) ? ((p.N + 15) / 16) * 16 : BN;
    const uint32_t IDESC = idesc_bf16_f32(128, n_mma, KIND == kKindWgrad ? 1 : 0, KIND == kKindFwd ? 0 : 1);
    uint32_t it = 0;
    bool issued = false;
    for (uint32_t local = 0;; ++local) {
      // one read of the abort flag for the whole warp keeps its lanes together
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const int tile = take_tile(local, kErrWaitMma);
      if (tile >= total) break;
      const Tile t = tile_coords<KIND, TM>(c, G, n_tiles, m_tiles_w, n_fast, tile);
      const int grows = KIND == kKindWgrad ? c.grp_row[t.g + 1] - c.grp_row[t.g] : 0;
      const int nk1 = KIND == kKindWgrad ? (grows + BK - 1) / BK : nk_fixed;
      const int nk = KIND == kKindWgrad && p.b_lo ? 2 * nk1 : nk1;
      int n_half = BM / 128;  // M=128 MMAs per K step
      if (KIND != kKindWgrad && BM == 256) {
        const bool xt = KIND == kKindFwd && t.g == G;
        const int g0 = xt ? 0 : c.grp_row[t.g], g1 = xt ? p.xrows : c.grp_row[t.g + 1];
        if (g1 - (g0 + t.m * TM) <= 128) n_half = 1;
      }
      const uint32_t acc = local % NACC;
      const uint32_t aph = (local / NACC) & 1u;
      bool ok = lane == 0 ? mbar_wait(&c.tmem_empty[acc], aph ^ 1u) : true;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) record_error(p.err, kErrWaitMma);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const uint32_t s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        bool okf = lane == 0 ? mbar_wait(&c.full[s], ph) : true;
        okf = __shfl_sync(0xffffffffu, okf, 0);
        if (!okf) {
          if (lane == 0) record_error(p.err, kErrWaitMma);
          *abort_flag = 1;
          ok = false;
          break;
        }
        uint8_t* sa = tiles + s * STAGE_BYTES;
        uint8_t* sb = sa + A_TILE_BYTES;
        if (KIND == kKindWgrad) {
          const int valid = grows - (kb >= nk1 ? kb - nk1 : kb) * BK;  // in (0, BK]
          if (valid < BK) {
            // rows [valid, BK) of this k-block belong to the next group (or
            // lie past the tensor): clear them in all six 64-row MN blocks.
            // The phase completed already, so this wait returns at once and
            // makes the copy's data visible to every lane.
            mbar_wait(&c.full[s], ph);
            constexpr int ABLK = BM / 64;  // MN blocks of the A tile (the B tile has 4)
            const int nrow = BK - valid;
            const int per_block = nrow * 8;  // 16-byte chunks
            for (int q = lane; q < (ABLK + 4) * per_block; q += 32) {
              const int blk = q / per_block;
              const int rem = q - blk * per_block;
              const int r = valid + (rem >> 3);
              uint8_t* base = blk < ABLK ? sa + blk * MN_BLOCK_BYTES : sb + (blk - ABLK) * MN_BLOCK_BYTES;
              *reinterpret_cast<uint4*>(base + r * 128 + (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_base = smem_u32(sa);
          const uint32_t b_base = smem_u32(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t a_k = KIND == kKindWgrad ? a_base + kk * 2048 : a_base + kk * 32;
            const uint64_t bd =
                KIND == kKindFwd ? sw128_kmajor_desc(b_base + kk * 32) : sw128_mnmajor_desc(b_base + kk * 2048);
            // rows 128h..128h+127 of A: +16 KB in both layouts (128 rows of
            // 128 B K-major, or two 64-wide MN blocks)
#pragma unroll
            for (int hh = 0; hh < BM / 128; ++hh) {
              if (hh >= n_half) break;
              const uint64_t ad = KIND == kKindWgrad ? sw128_mnmajor_desc(a_k + hh * 16384)
                                                     : sw128_kmajor_desc(a_k + hh * 16384);
              tc_mma_bf16(d_tmem + hh * BN, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&c.empty[s]);
        }
        __syncwarp();
        issued = true;
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&c.tmem_full[acc]);
      __syncwarp();
    }
    if (*abort_flag && issued && lane == 0) {
      tc_commit(&c.drain);
      if (!mbar_wait(&c.drain, 0)) record_error(p.err, kErrWaitDrain);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;          // TMEM lanes [32*quarter, 32*quarter+32)
    const int half = (warp - 2) >> 2;      // BM = 256: accumulator rows 128*half.. (columns 256*half..)
    uint4* const stg = stage_out + (warp - 2) * (STAGE_OUT_BYTES / 16);  // this warp's output staging
    for (uint32_t local = 0;; ++local) {
      // tcgen05.ld is warp-collective: the warp decides to stop as one
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const int tile = take_tile(local, kErrWaitEpilogue);
      if (tile >= total) break;
      const Tile t = tile_coords<KIND, TM>(c, G, n_tiles, m_tiles_w, n_fast, tile);
      const bool xg = KIND == kKindFwd && t.g == G;  // the extra group
      const int grow = xg ? 0 : c.grp_row[t.g];
      const int gend = xg ? p.xrows : c.grp_row[t.g + 1];
      void* const out_p = xg ? p.xout : p.out;
      void* const zsave_p = xg ? p.xzsave : p.zsave;
      const uint32_t acc = local % NACC;
      const uint32_t aph = (local / NACC) & 1u;
      // (PAIR: the even CTA's commit arrives here on both SMs)
      if (!__all_sync(0xffffffffu, mbar_wait(&c.tmem_full[acc], aph))) {
        if (lane == 0) record_error(p.err, kErrWaitEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      // hand the accumulator back to the MMA warp.  The branches below call
      // this as soon as their last TMEM load of the tile has completed, so
      // that the next tile's MMAs overlap the last chunk's arithmetic and
      // stores; otherwise it runs at the end of the tile.  Warp-uniform.
      bool released = false;
      auto release = [&]() {
        tc_fence_before();
        if constexpr (PAIR) {
          // one arrival per warp, on the even CTA's barrier (it reuses the
          // accumulator of both CTAs)
          __syncwarp();
          if (lane == 0) {
            if (crank == 0) mbar_arrive(&c.tmem_empty[acc]);
            else mbar_arrive_cluster(mapa_shared(&c.tmem_empty[acc], 0));
          }
        } else {
          mbar_arrive(&c.tmem_empty[acc]);
        }
        released = true;
      };
      const int rt = half * 128 + quarter * 32 + lane;  // tile row of this thread
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + (acc + half) * BN;
      // the upper half of a half tile holds no rows and was not multiplied
      const bool idle_half = KIND != kKindWgrad && BM == 256 && half == 1 && gend - (grow + t.m * TM) <= 128;

      if (KIND == kKindWgrad) {
        // out_g[m, n] fp32; a group with no rows has a zero gradient
        const bool empty = gend == grow;
        const int m = t.m * BM + rt;
        const bool valid = m < p.M;
        float* orow = nullptr;
        if (valid) {
          const int M1 = p.m_split ? p.m_split : p.M;
          if (m < M1)
            orow = static_cast<float*>(p.out) + (static_cast<size_t>(t.g) * M1 + m) * p.N;
          else
            orow = static_cast<float*>(p.out2) + (static_cast<size_t>(t.g) * (p.M - M1) + (m - M1)) * p.N;
        }
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + cc * 32, r);
          tmem_ld_wait();
          if (cc == BN / 32 - 1) release();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = empty ? 0.f : __uint_as_float(r[i]);
          warp_store_f32x32(stg, orow, t.n * BN + cc * 32, p.N, v, lane);
        }
      } else if (!idle_half) {
        const long long row_end = xg ? static_cast<long long>(gend) : min(static_cast<long long>(gend), p.rows_alloc);
        const int row = grow + t.m * TM + static_cast<int>(crank) * BM + rt;
        const bool valid = row < row_end;
        if (KIND == kKindFwd && BM == 128 && !PAIR && p.mode == kModeRouteTopK) {
          // (the launcher runs this mode on single-CTA 128-row tiles only)
          // the router: this thread's token's E logits, 4 columns at a time
          // (a small loop body: the thread walks all E alone).  Pass 1 adds
          // bias and noise, checks finiteness and keeps a descending top-k
          // (experts in increasing order, so an equal value keeps the lower
          // index) and the max m; pass 2 (raw weights or the entropy) sums
          // exp(l - m) and exp(l - m) (l - m).
          const RouteEpilogue& R = p.route;
          float sv[MAXK];
          int si[MAXK];
#pragma unroll
          for (int j = 0; j < MAXK; ++j) {
            sv[j] = -INFINITY;
            si[j] = -1;
          }
          bool finite = true;
          float m = -INFINITY;
          const float* nrow = R.noise && valid ? R.noise + static_cast<size_t>(row) * R.E : nullptr;
          float* lrow = R.logits && valid ? R.logits + static_cast<size_t>(row) * R.E : nullptr;
          auto logit = [&](uint32_t raw_bits, int e) {
            float a = __uint_as_float(raw_bits);
            if (R.bias) a += R.bias[e];
            if (nrow) a += nrow[e];
            return a;
          };
          const int nq = (R.E + 3) / 4;
#pragma unroll 1
          for (int q = 0; q < nq; ++q) {
            uint32_t r[4];
            tmem_ld_32x32b_x4(taddr + q * 4, r);
            tmem_ld_wait();
            if (!valid) continue;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = q * 4 + i;
              if (e < R.E) {
                const float a = logit(r[i], e);
                if (!isfinite(a)) finite = false;
                if (lrow) lrow[e] = a;
                topk_insert(sv, si, R.k, a, e);
                m = fmaxf(m, a);
              }
            }
          }
          SoftStat st;
          // tcgen05.ld is warp-collective: the whole warp runs this pass
          // (the condition is the same for every lane); a row that is past
          // the end or not finite only skips the sums
          if (R.raw || R.ent) {
            float z = 0.f, sz = 0.f;
#pragma unroll 1
            for (int q = 0; q < nq; ++q) {
              uint32_t r[4];
              tmem_ld_32x32b_x4(taddr + q * 4, r);
              tmem_ld_wait();
              if (!valid || !finite) continue;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int e = q * 4 + i;
                if (e < R.E) {
                  const float dv = logit(r[i], e) - m;
                  const float ex = expf(dv);
                  z += ex;
                  sz = fmaf(ex, dv, sz);
                }
              }
            }
            st.m = m;
            st.Z = z;
            st.S = sz;
          }
          if (valid) topk_finish(sv, si, R.k, finite, row, R.idx, R.w, c.hist, R.raw != 0, st, R.ent);
        } else if (swiglu_fwd) {
          bf16* orow = static_cast<bf16*>(out_p) + static_cast<size_t>(row) * p.ldo;
          // the pre-activations are kept in fp32 for the backward: a bf16
          // copy would put a 2^-9 rounding inside silu'(gate) and up there
          float* zrow = zsave_p ? static_cast<float*>(zsave_p) + static_cast<size_t>(row) * p.ldz : nullptr;
          const int col0 = t.n * 128;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t gr[32], ur[32];
            tmem_ld_32x32b_x32(taddr + cc * 32, gr);
            tmem_ld_32x32b_x32(taddr + 128 + cc * 32, ur);
            tmem_ld_wait();
            if (cc == 3) release();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
              const float u0 = __uint_as_float(ur[2 * i]), u1 = __uint_as_float(ur[2 * i + 1]);
              pk[i] = pack_bf16(silu_fast(g0) * u0, silu_fast(g1) * u1);
            }
            const int col = col0 + cc * 32;
            if (valid) {
              store_bf16x32(orow, col, p.N, pk);
              if (zrow) {
                float zv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) zv[i] = __uint_as_float(gr[i]);
                store_f32x32(zrow, col, p.N, zv);
#pragma unroll
                for (int i = 0; i < 32; ++i) zv[i] = __uint_as_float(ur[i]);
                store_f32x32(zrow + p.N, col, p.N, zv);
              }
            }
          }
        } else {
          const int col0 = t.n * BN;
          const int mode = p.mode;
          const bf16* brow = xg ? static_cast<const bf16*>(p.xbias)
                                : (p.bias ? static_cast<const bf16*>(p.bias) + static_cast<size_t>(t.g) * p.N : nullptr);
          const bool bwd_mode = mode == kModeSwiGLUBwd || mode == kModeGeLUBwd;
          const float* zin = bwd_mode && valid ? static_cast<const float*>(p.zin) + static_cast<size_t>(row) * p.ldz
                                               : nullptr;
          // backward: dH = s * acc with s the row's routing weight, and the
          // weighted activation s * act(z) for the W2 gradient
          const float rs = bwd_mode && valid && p.row_scale ? p.row_scale[row] : 1.0f;
          bf16* hrow = bwd_mode && valid && p.hout ? static_cast<bf16*>(p.hout) + static_cast<size_t>(row) * p.N
                                                   : nullptr;
          bf16* lrow = hrow && p.hout_lo ? static_cast<bf16*>(p.hout_lo) + static_cast<size_t>(row) * p.N
                                         : nullptr;
          float* zrow = zsave_p && mode == kModeGeLU && valid
                            ? static_cast<float*>(zsave_p) + static_cast<size_t>(row) * p.ldz
                            : nullptr;
#pragma unroll 1
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + cc * 32, r);
            tmem_ld_wait();
            if (cc == BN / 32 - 1) release();
            const int col = col0 + cc * 32;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            if (!valid) continue;
            if (mode == kModeSwiGLUBwd) {
              // dH = s acc; gate g, up u: dA = dH u silu'(g), dB = dH silu(g), H' = s silu(g) u
              float g[32], u[32];
              load_f32x32(zin, col, p.N, g);
              load_f32x32(zin + p.N, col, p.N, u);
              uint32_t pa[16], pb[16], ph[16], pl[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float da[2], db[2], hh[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                  const int e = 2 * i + h2;
                  const float sg = sigmoid_fast(g[e]);
                  const float sl = g[e] * sg;
                  const float dh = rs * v[e];
                  da[h2] = dh * u[e] * (sg * (1.0f + g[e] * (1.0f - sg)));
                  db[h2] = dh * sl;
                  hh[h2] = rs * sl * u[e];
                }
                pa[i] = pack_bf16(da[0], da[1]);
                pb[i] = pack_bf16(db[0], db[1]);
                ph[i] = pack_bf16(hh[0], hh[1]);
                pl[i] = pack_bf16(hh[0] - bf16lo(ph[i]), hh[1] - bf16hi(ph[i]));
              }
              bf16* orow = static_cast<bf16*>(p.out) + static_cast<size_t>(row) * p.ldo;
              store_bf16x32(orow, col, p.N, pa);
              store_bf16x32(orow + p.N, col, p.N, pb);
              if (hrow) store_bf16x32(hrow, col, p.N, ph);
              if (lrow) store_bf16x32(lrow, col, p.N, pl);
              continue;
            }
            if (mode == kModeGeLUBwd) {
              float z[32];
              load_f32x32(zin, col, p.N, z);
              if (hrow) {
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float h0 = rs * gelu_f(z[2 * i]), h1 = rs * gelu_f(z[2 * i + 1]);
                  ph[i] = pack_bf16(h0, h1);
                  pl[i] = pack_bf16(h0 - bf16lo(ph[i]), h1 - bf16hi(ph[i]));
                }
                store_bf16x32(hrow, col, p.N, ph);
                if (lrow) store_bf16x32(lrow, col, p.N, pl);
              }
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= rs * gelu_grad_f(z[i]);
            } else {
              if (brow) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (col + i < p.N) v[i] += __bfloat162float(brow[col + i]);
              }
              if (mode == kModeGeLU) {
                if (zrow) store_f32x32(zrow, col, p.N, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i]);
              }
            }
            if (p.out_f32) {
              store_f32x32(static_cast<float*>(out_p) + static_cast<size_t>(row) * p.ldo, col, p.N, v);
            } else {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
              store_bf16x32(static_cast<bf16*>(out_p) + static_cast<size_t>(row) * p.ldo, col, p.N, pk);
            }
          }
        }
      }
      if (!released) release();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (KIND == kKindFwd && p.mode == kModeRouteTopK)
    for (int e = threadIdx.x; e < p.route.E; e += blockDim.x)
      if (c.hist[e]) atomicAdd(&p.route.counts[e], c.hist[e]);
  // PAIR: neither CTA leaves (or frees its TMEM) while the other may still
  // signal its barriers or the MMAs may still read its shared memory
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int KIND, int BM_, bool PAIR>
moe_status launch_kind(const GemmParams& p, const CUtensorMap& mA, const CUtensorMap& mB0, const CUtensorMap& mB1,
                       const CUtensorMap& mXA, const CUtensorMap& mXB0, const CUtensorMap& mXB1, long long tiles_bound,
                       cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  constexpr size_t smem = smem_bytes<KIND, BM_, PAIR>();
  constexpr int threads = TileCfg<BM_, PAIR>::THREADS;
  auto kern = grouped_gemm_tc_kernel<KIND, BM_, PAIR>;
  // pair launches: clusters of two CTAs; the kernel is persistent, so the
  // grid is no larger than the clusters that can be resident at once
  cudaLaunchAttribute cluster_attr[2];
  cluster_attr[0].id = cudaLaunchAttributeClusterDimension;
  cluster_attr[0].val.clusterDim.x = 2;
  cluster_attr[0].val.clusterDim.y = 1;
  cluster_attr[0].val.clusterDim.z = 1;
  // programmatic stream serialization, as launch_pdl gives every other launch
  cluster_attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cluster_attr[1].val.programmaticStreamSerializationAllowed = 1;
  static DeviceOnce attr;
  static int max_clusters[64] = {0};
  const moe_status sa = attr.run(dev, [&] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    if (PAIR) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(2, 1, 1);
      q.blockDim = dim3(threads, 1, 1);
      q.dynamicSmemBytes = smem;
      q.attrs = cluster_attr;
      q.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) return MOE_ERR_CUDA;
      max_clusters[dev] = n;
    }
    return MOE_OK;
  });
  if (sa != MOE_OK) return sa;
  long long grid = tiles_bound;
  if (PAIR) {
    if (grid > max_clusters[dev]) grid = max_clusters[dev];
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * grid), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = cluster_attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, mA, mB0, mB1, mXA, mXB0, mXB1, p) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, mA, mB0, mB1, mXA, mXB0, mXB1,
               p);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

// Tile shape for a launch: 256-row single-CTA tiles when the groups average
// at least 256 output rows, such tiles still give every SM one, and the
// epilogue is light -- plain, or any forward activation -- else 128-row
// tiles; a forward launch asked for CTA pairs (p.cta_pairs) runs 256-row
// tiles on pairs under the same rule.
template <int KIND>
moe_status launch_geometry(const GemmParams& p, const void* A, long long a_rows, const void* B0, const void* B1,
                           long long b_rows, long long avg_rows, const GemmExtra* extra, cudaStream_t stream) {
  // BM = 256 on one CTA feeds the tensor cores with 2/3 of the shared-memory
  // traffic per MAC but has a single accumulator, so its epilogue does not
  // overlap the next tile's MMAs.  On the power-capped part the saved
  // traffic outweighs the lost overlap for every forward epilogue: the large
  // prefill's SwiGLU GEMM-1 is 3% faster live (though 9% slower at uncapped
  // clocks), and the training forward's, which also stores the fp32
  // pre-activations, 6%.  The backward's activation epilogue (it reads those
  // pre-activations and writes four outputs) keeps 128-row tiles.  A CTA
  // pair halves the B bytes staged per MAC and keeps two accumulators per
  // CTA.  Either only when it still gives every SM a tile (a single-group
  // launch such as the router's logits would otherwise leave most SMs idle).
  const long long n_tiles = (KIND == kKindFwd && p.mode == kModeSwiGLU) ? (p.N + 127) / 128 : (p.N + BN - 1) / BN;
  auto tiles_for = [&](int bm) -> long long {
    if (KIND == kKindWgrad) return static_cast<long long>(p.G) * ((p.M + bm - 1) / bm) * n_tiles;
    const long long rows_bound = p.offsets ? a_rows : p.rows;
    long long tl = ((rows_bound + bm - 1) / bm + (p.offsets ? p.G : 0)) * n_tiles;
    if (KIND == kKindFwd && p.xrows > 0) tl += ((p.xrows + bm - 1) / bm) * n_tiles;
    return tl;
  };
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  const bool pair = KIND == kKindFwd && p.cta_pairs && avg_rows >= 256 && (p.mode == kModeSwiGLU || p.N >= BN) &&
                    2 * tiles_for(256) >= sms;
  const bool light = p.mode == kModePlain || (KIND == kKindFwd && p.mode != kModeRouteTopK);
  const bool tall = !pair && avg_rows >= 256 && light && tiles_for(256) >= sms;
  CUtensorMap mA, mB0, mB1, mXA, mXB0, mXB1;  // Fwd/Dgrad A boxes: 128 rows (two per 256-row tile)
  const long long tiles = tiles_for(pair || tall ? 256 : 128);
  if (KIND == kKindFwd) {
    if (!make_tma_2d_bf16(&mA, A, p.K, a_rows, BK, 128)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mB0, B0, p.K, b_rows, BK, 128)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mB1, B1 ? B1 : B0, p.K, b_rows, BK, 128)) return MOE_ERR_CUDA;
  } else if (KIND == kKindDgrad) {
    if (!make_tma_2d_bf16(&mA, A, p.K, a_rows, BK, 128)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mB0, B0, p.N, b_rows, 64, BK)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mB1, B1 ? B1 : B0, p.N, b_rows, 64, BK)) return MOE_ERR_CUDA;
  } else {
    if (!make_tma_2d_bf16(&mA, A, p.M, a_rows, 64, BK)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mB0, B0, p.N, a_rows, 64, BK)) return MOE_ERR_CUDA;
    if (p.b_lo) {
      if (!make_tma_2d_bf16(&mB1, B1, p.N, a_rows, 64, BK)) return MOE_ERR_CUDA;
    } else {
      mB1 = mB0;
    }
  }
  if (KIND == kKindFwd && p.xrows > 0) {
    const long long n_rows = p.N;  // rows of the extra group's weights [N, K]
    if (!make_tma_2d_bf16(&mXA, extra->A, p.K, p.xrows, BK, 128)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mXB0, extra->B0, p.K, n_rows, BK, 128)) return MOE_ERR_CUDA;
    if (!make_tma_2d_bf16(&mXB1, extra->B1 ? extra->B1 : extra->B0, p.K, n_rows, BK, 128)) return MOE_ERR_CUDA;
  } else {
    mXA = mA;
    mXB0 = mB0;
    mXB1 = mB1;
  }
  if constexpr (KIND == kKindFwd) {
    if (pair) return launch_kind<KIND, 128, true>(p, mA, mB0, mB1, mXA, mXB0, mXB1, tiles, stream);
  }
  return tall ? launch_kind<KIND, 256, false>(p, mA, mB0, mB1, mXA, mXB0, mXB1, tiles, stream)
              : launch_kind<KIND, 128, false>(p, mA, mB0, mB1, mXA, mXB0, mXB1, tiles, stream);
}

}  // namespace

moe_status launch_grouped_gemm_tc(const GemmParams& p_in, int kind, const void* A, long long a_rows, const void* B0,
                                  const void* B1, long long b_rows, cudaStream_t stream, const GemmExtra* extra) {
  GemmParams p = p_in;
  if (p.xrows < 0 || (p.xrows > 0 && (kind != kKindFwd || !extra || !extra->A || !extra->B0 || !p.xout)))
    return MOE_ERR_INVALID_ARG;
  if (p.xrows == 0) extra = nullptr;
  p.rows_alloc = a_rows;
  if (p.ldo == 0) p.ldo = p.N;
  if (p.G < 1 || p.G > MAX_GROUPS || p.N < 8 || (p.N % 8) || (!p.out && p.mode != kModeRouteTopK))
    return MOE_ERR_UNSUPPORTED;
  if (a_rows <= 0) return MOE_OK;
  if (a_rows > 2147483647LL || b_rows > 2147483647LL) return MOE_ERR_UNSUPPORTED;
  // output rows per group on average (Wgrad: M, the same for every group)
  const long long avg_rows = kind == kKindWgrad ? p.M : (p.offsets ? a_rows / p.G : p.rows);
  if (kind == kKindFwd) {
    if (p.K < 8 || (p.K % 8)) return MOE_ERR_UNSUPPORTED;
    if (p.mode == kModeSwiGLUBwd || p.mode == kModeGeLUBwd) return MOE_ERR_UNSUPPORTED;
    if (p.mode == kModeRouteTopK) {
      // one group of T rows, all E logits in one 256-column tile
      const RouteEpilogue& R = p.route;
      if (p.offsets || p.G != 1 || p.xrows || p.cta_pairs || p.N > BN || R.E < 1 || R.E > p.N || R.k < 1 ||
          R.k > MAXK || R.k > R.E || !R.idx || !R.w || !R.counts)
        return MOE_ERR_INVALID_ARG;
    }
    return launch_geometry<kKindFwd>(p, A, a_rows, B0, B1, b_rows, avg_rows, extra, stream);
  }
  if (kind == kKindDgrad) {
    // whole 64-deep k-blocks per weight tensor, so a block never mixes groups or tensors
    if (p.K < BK || (p.K % BK) || (p.k_split && (p.k_split % BK || p.K != 2 * p.k_split))) return MOE_ERR_UNSUPPORTED;
    if (p.k_split && !B1) return MOE_ERR_INVALID_ARG;
    if (p.mode == kModeSwiGLU || p.mode == kModeGeLU) return MOE_ERR_UNSUPPORTED;
    if ((p.mode == kModeSwiGLUBwd || p.mode == kModeGeLUBwd) && !p.zin) return MOE_ERR_INVALID_ARG;
    return launch_geometry<kKindDgrad>(p, A, a_rows, B0, B1, b_rows, avg_rows, nullptr, stream);
  }
  if (kind == kKindWgrad) {
    if (p.M < 8 || (p.M % 8) || !p.out_f32 || p.mode != kModePlain) return MOE_ERR_UNSUPPORTED;
    if (p.m_split && (p.m_split % 8 || p.m_split >= p.M || !p.out2)) return MOE_ERR_UNSUPPORTED;
    if (p.b_lo && !B1) return MOE_ERR_INVALID_ARG;
    return launch_geometry<kKindWgrad>(p, A, a_rows, B0, B1, b_rows, avg_rows, nullptr, stream);
  }
  return MOE_ERR_INVALID_ARG;
}

}  // namespace moe

// Capacity-limited dispatch and the weighted combine.
//
// Dispatch ([P3] "MoE architecture revealed..." 2.3: every expert has a
// capacity C and the tokens beyond it are dropped; [P1] "'More parameters is
// better' is not the story..." 4.2 step 2: the tokens bound for the same
// expert are grouped together).  Slots are ordered slot-major -- s = j*T + t,
// every token's first choice in token order, then every second choice -- and
// a slot's rank is the number of earlier slots routed to the same expert.
// A slot is kept iff rank < C; kept rows are laid out expert by expert:
//   offsets = exclusive scan of kept[e] = min(routed[e], C)
//   pos[t,j] = offsets[e] + rank, or -1 when dropped / unrouted
//   Xp[pos[t,j]] = x[t]
// Four launches, all integer and deterministic (no order-visible atomics):
//   slot_hist   per chunk of 1024 (or 4096) slots, per-expert counts (+ unrouted)
//   scan        per-expert exclusive scan over chunks (several lanes per
//               expert), kept, offsets, stats from integer sums
//   assign      in-chunk ranks (warp match + per-warp counts), pos
//   permute     one warp per token copies its row to its k destinations
// Token-major priority orders the slots s = t*k + j instead.  Rerouting on
// overflow ([P3] 2.3: the next-best expert) runs slot_hist, scan and assign
// a second time over the slots the first pass dropped, each asking for its
// token's backup expert against the room left.
//
// Combine ([P5] "Training a 200B LLM from scratch 5/25", "Who decides which
// experts to call?": y = 0.75*E1(x) + 0.25*E3(x); "Shared experts": the
// always-on path is added):
//   y[t] = sum_{j: pos >= 0} w[t,j] * Yp[pos[t,j]]  (+ Sx[t]), fp32, j ascending.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int DT = 256;      // threads of the chunk kernels
constexpr int DW = DT / 32;  // warps of the chunk kernels

// Slots per chunk of the histogram/rank kernels: 1024 for up to 2^18 slots
// (enough blocks to fill the GPU), 4096 beyond (so that T*k <= 2^20 slots
// need at most 256 chunks of scratch).
inline int chunk_slots(long long nslots) { return nslots <= (1LL << 18) ? 1024 : 4096; }

// Slot s in priority order -> (t, j) and its expert.  Slot-major: s = j*T + t;
// token-major: s = t*k + j (the row-major order of idx).
__device__ __forceinline__ int slot_expert(const int* idx, int T, int k, bool token_major, long long s, int& t,
                                           int& j) {
  if (token_major) {
    t = static_cast<int>(s / k);
    j = static_cast<int>(s - static_cast<long long>(t) * k);
  } else {
    j = static_cast<int>(s / T);
    t = static_cast<int>(s - static_cast<long long>(j) * T);
  }
  return idx[static_cast<size_t>(t) * k + j];
}

// The slots of one capacity pass.  Pass 1 (rank1 == nullptr): each slot
// asks for its chosen expert.  Pass 2 (rerouting on overflow): a slot the
// first pass dropped asks for backup[t, r], r = the number of the token's
// earlier slots (j' < j) that were dropped too; every other slot asks for
// none (-1).  rank1 holds the first pass's ranks (-1 = not kept).
struct SlotSrc {
  const int* idx;
  const int* rank1;
  const int* backup;
};

// Expert slot s asks for in this pass; e0 receives its chosen expert.
__device__ __forceinline__ int pass_expert(const SlotSrc& S, int T, int k, bool token_major, long long s, int& t,
                                           int& j, int& e0) {
  e0 = slot_expert(S.idx, T, k, token_major, s, t, j);
  if (!S.rank1) return e0;
  const size_t row = static_cast<size_t>(t) * k;
  if (e0 < 0 || S.rank1[row + j] >= 0) return -1;
  int r = 0;
  for (int q = 0; q < j; ++q)
    if (S.idx[row + q] >= 0 && S.rank1[row + q] < 0) ++r;
  return S.backup[row + r];
}

__global__ void __launch_bounds__(DT) slot_hist_kernel(SlotSrc S, int T, int k, int E, bool token_major, int CH,
                                                       int* __restrict__ blockhist) {
  pdl_entry();
  extern __shared__ int hist[];  // E + 1 (last: unrouted)
  for (int e = threadIdx.x; e <= E; e += DT) hist[e] = 0;
  __syncthreads();
  const long long nslots = static_cast<long long>(T) * k;
  const long long s0 = static_cast<long long>(blockIdx.x) * CH;
  for (int i = threadIdx.x; i < CH; i += DT) {
    const long long s = s0 + i;
    if (s >= nslots) break;
    int t, j, e0;
    const int e = pass_expert(S, T, k, token_major, s, t, j, e0);
    atomicAdd(&hist[(e >= 0 && e < E) ? e : E], 1);
  }
  __syncthreads();
  int* out = blockhist + static_cast<size_t>(blockIdx.x) * (E + 1);
  for (int e = threadIdx.x; e <= E; e += DT) out[e] = hist[e];
}

// v 2^40 truncated toward zero, as an integer, for a finite |v| < 2^23 (an
// entropy is at most ln E); integer operations only.  v = m 2^(e - 150) for
// the 24-bit significand m and biased exponent e, so v 2^40 = m 2^(e - 110);
// subnormals (|v| < 2^-126) count as 0.
__device__ __forceinline__ long long fixed40(float v) {
  const uint32_t u = __float_as_uint(v);
  const int e = static_cast<int>((u >> 23) & 0xFFu);
  if (e == 0) return 0;
  const long long m = static_cast<long long>((u & 0x7FFFFFu) | 0x800000u);
  const int sh = min(e - 110, 39);
  const long long mag = sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0);
  return (u >> 31) ? -mag : mag;
}

// Integer totals of the load statistics: routed and kept slots, sum of
// c_e^2, the entropy sum in units of 2^-40, max c_e, finite entropies,
// unrouted slots.
struct StatSums {
  long long rc, kc, s2, ts;
  int mx, tc, unrouted, pad;
};

// Parameters of the statistics' fp64 finish.
struct StatsFinish {
  const StatSums* sums;  // nullptr: none to finish
  moe_stats* stats;
  int T, k, E, C, balance;
  float lam, gamma;
};

// The statistics from their integer totals, by one whole warp.  With f =
// c/T,
//   sum_e (f_e - mean f)^2 = (E sum c^2 - (sum c)^2) / (E T^2)
// from an exact 128-bit numerator.  fp64 runs at a small fraction of fp32's
// rate on this part, so the five independent quotients run on five lanes at
// once: the longest dependent fp64 chain is a division, a square root and a
// division.
__device__ __forceinline__ void stats_finish_warp(const StatSums& S, const StatsFinish& F, int lane) {
  const long long nslots = static_cast<long long>(F.T) * F.k;
  const int E = F.E;
  // rc = sum c <= T k <= 2^30, so s2 <= rc^2 <= 2^60 and E s2 < 2^71
  const unsigned __int128 num = static_cast<unsigned __int128>(E) * static_cast<unsigned long long>(S.s2) -
                                static_cast<unsigned __int128>(S.rc) * static_cast<unsigned long long>(S.rc);
  const double Td = static_cast<double>(F.T);
  // lane 0: the variance sum / (E (E-1) T^2); 1: mean f = sum c / (E T);
  // 2: the drop rate; 3: the mean entropy; 4: max f = max c / T
  double a = 0.0, b = 1.0;
  if (lane == 0) {
    a = static_cast<double>(static_cast<unsigned long long>(num >> 64)) * 18446744073709551616.0 +
        static_cast<double>(static_cast<unsigned long long>(num));
    b = E > 1 ? static_cast<double>(E) * static_cast<double>(E - 1) * (Td * Td) : 1.0;
  } else if (lane == 1) {
    a = static_cast<double>(S.rc);
    b = static_cast<double>(E) * Td;
  } else if (lane == 2) {
    a = static_cast<double>(nslots - S.kc);
    b = static_cast<double>(nslots);
  } else if (lane == 3) {
    a = static_cast<double>(S.ts) * 0x1p-40;
    b = static_cast<double>(S.tc > 0 ? S.tc : 1);
  } else if (lane == 4) {
    a = static_cast<double>(S.mx);
    b = Td;
  }
  const double q = a / b;
  const double var = __shfl_sync(0xffffffffu, q, 0), mean = __shfl_sync(0xffffffffu, q, 1);
  const double drop = __shfl_sync(0xffffffffu, q, 2), emean = __shfl_sync(0xffffffffu, q, 3);
  const double fmax = __shfl_sync(0xffffffffu, q, 4);
  if (lane == 0) {
    const double sd = E > 1 ? sqrt(var) : 0.0;
    moe_stats st;
    st.routed_slots = S.rc;
    st.kept_slots = S.kc;
    st.dropped_slots = nslots - S.kc;
    st.capacity = F.C;
    st.numeric_error = S.unrouted / F.k;
    st.drop_rate = drop;
    if (F.balance == MOE_BALANCE_STD_MAX)
      st.balance_stat = static_cast<double>(F.lam) * (sd + static_cast<double>(F.gamma) * fmax);
    else if (F.balance == MOE_BALANCE_SWITCH)
      st.balance_stat = __longlong_as_double(0x7ff8000000000000LL);  // needs the weights: set by the layer
    else
      st.balance_stat = E > 1 ? static_cast<double>(F.lam) * sd / (mean + 1e-8) : 0.0;
    st.router_entropy = S.tc > 0 ? emean : __longlong_as_double(0x7ff8000000000000LL);
    st.rerouted_slots = 0;
    *F.stats = st;
  }
}

// The capacity scan of a whole block of 1024 threads (every thread calls
// it; it synchronises the block): per-expert bases across chunks, kept,
// offsets and the statistics.  blockhist [nb][E+1] may be in global or
// shared memory.
__device__ __forceinline__ void capacity_scan_block(const int* __restrict__ blockhist, int nb, int T, int k, int E,
                                                    int C, float lam, int balance, float gamma,
                                                    const int* __restrict__ used, int* __restrict__ base,
                                                    int* __restrict__ kept, int* __restrict__ offsets,
                                                    moe_stats* stats, const float* __restrict__ ent,
                                                    StatSums* defer) {
  __shared__ int tot[1024];
  __shared__ int warp_sums[32];
  __shared__ int unrouted;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  // per expert, exclusive scan of its chunk counts across chunks; expert E
  // is the "unrouted" column.  L lanes per expert (as many as fit all E+1
  // columns into the block at once, at most a warp) take L chunks a step;
  // the loops are uniform per warp, lanes past column E carry zeros.
  int L = 32;
  while (L > 1 && (E + 1) * L > static_cast<int>(blockDim.x)) L >>= 1;
  const int gpw = 32 / L;  // experts per warp
  const int sub = lane / L, gl = lane - (lane / L) * L;
  const int nwarps = blockDim.x >> 5;
  for (int e0 = warp * gpw; e0 <= E; e0 += nwarps * gpw) {
    const int e = e0 + sub;
    const bool ev = e <= E;
    int carry = 0;
    for (int b0 = 0; b0 < nb; b0 += L) {
      const int b = b0 + gl;
      const int v = (ev && b < nb) ? blockhist[static_cast<size_t>(b) * (E + 1) + e] : 0;
      int incl = v;
      for (int o = 1; o < L; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o, L);
        if (gl >= o) incl += u;
      }
      if (ev && e < E && b < nb) base[static_cast<size_t>(b) * E + e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, L - 1, L);
    }
    if (ev && gl == 0) {
      if (e < E) tot[e] = carry;
      else unrouted = carry;
    }
  }
  __syncthreads();
  // pass 2 (used != nullptr): the room left after the first pass's rows,
  // and kept[e] counts both passes
  int my_kept = 0, my_new = 0;
  if (tid < E) {
    const int u = used ? used[tid] : 0;
    my_new = tot[tid] < C - u ? tot[tid] : C - u;
    my_kept = u + my_new;
  }
  // exclusive scan of kept over experts (block-wide, experts in index order)
  int incl = my_kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = warp_sums[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - ws;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int excl = warp_sums[warp] + incl - my_kept;
  if (tid < E) {
    kept[tid] = my_kept;
    offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + my_kept;
  }
  if (stats && used) {
    // pass 2: the rerouted rows move from dropped to kept
    __shared__ long long rer_s[32];
    long long v = my_new;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) rer_s[warp] = v;
    __syncthreads();
    if (tid == 0) {
      long long rer = 0;
      for (int w2 = 0; w2 < ((blockDim.x + 31) >> 5); ++w2) rer += rer_s[w2];
      const long long nslots = static_cast<long long>(T) * k;
      stats->kept_slots += rer;
      stats->dropped_slots -= rer;
      stats->drop_rate = static_cast<double>(stats->dropped_slots) / static_cast<double>(nslots);
      stats->rerouted_slots = rer;
    }
  } else if (stats) {
    // load statistics from integer sums (exact in any order): routed and
    // kept slots, sum and max of the counts c_e, and sum of c_e^2.
    //
    // With ent (the layer forward): router_entropy = the mean of the finite
    // entries of ent[0..T), summed exactly in fixed point (units of 2^-40,
    // each entry truncated by less than 2^-40, so the mean is within 2^-40
    // of the fp32 entries' exact mean).
    //
    // The sums run in the integer pipes; stats_finish_warp forms the fp64
    // statistics from them, here or (defer) in an extra block of the
    // assignment kernel, where it runs beside the placement instead of
    // between the scan and it.
    __shared__ long long redl[32][4];
    __shared__ int redmax[32];
    __shared__ int redec[32];
    const int nwarps = (blockDim.x + 31) >> 5;
    long long es = 0;
    int ec = 0;
    if (ent) {
#pragma unroll 8
      for (int t = tid; t < T; t += blockDim.x) {
        const float v = ent[t];
        if (isfinite(v)) {
          es += fixed40(v);
          ++ec;
        }
      }
    }
    long long r_cnt = tid < E ? tot[tid] : 0, k_cnt = tid < E ? my_kept : 0;
    long long sq = tid < E ? static_cast<long long>(tot[tid]) * tot[tid] : 0;
    int cmax = tid < E ? tot[tid] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      r_cnt += __shfl_xor_sync(0xffffffffu, r_cnt, o);
      k_cnt += __shfl_xor_sync(0xffffffffu, k_cnt, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      es += __shfl_xor_sync(0xffffffffu, es, o);
      ec += __shfl_xor_sync(0xffffffffu, ec, o);
    }
    if (lane == 0) {
      redl[warp][0] = r_cnt;
      redl[warp][1] = k_cnt;
      redl[warp][2] = sq;
      redl[warp][3] = es;
      redmax[warp] = cmax;
      redec[warp] = ec;
    }
    __syncthreads();
    if (warp == 0) {
      // block totals on every lane of warp 0 (lane w holds warp w's partials)
      long long rc = lane < nwarps ? redl[lane][0] : 0, kc = lane < nwarps ? redl[lane][1] : 0;
      long long s2 = lane < nwarps ? redl[lane][2] : 0, ts = lane < nwarps ? redl[lane][3] : 0;
      int mx = lane < nwarps ? redmax[lane] : 0, tc = lane < nwarps ? redec[lane] : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        rc += __shfl_xor_sync(0xffffffffu, rc, o);
        kc += __shfl_xor_sync(0xffffffffu, kc, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        ts += __shfl_xor_sync(0xffffffffu, ts, o);
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        tc += __shfl_xor_sync(0xffffffffu, tc, o);
      }
      const StatSums S{rc, kc, s2, ts, mx, tc, unrouted, 0};
      if (defer) {
        // an extra block of the assignment kernel that follows finishes them
        if (lane == 0) *defer = S;
      } else {
        stats_finish_warp(S, StatsFinish{nullptr, stats, T, k, E, C, balance, lam, gamma}, lane);
      }
    }
  }
}

__global__ void __launch_bounds__(1024) capacity_scan_kernel(const int* __restrict__ blockhist, int nb, int T,
                                                             int k, int E, int C, float lam, int balance,
                                                             float gamma, const int* __restrict__ used,
                                                             int* __restrict__ base, int* __restrict__ kept,
                                                             int* __restrict__ offsets, moe_stats* stats,
                                                             const float* __restrict__ ent, StatSums* defer) {
  pdl_entry();
  capacity_scan_block(blockhist, nb, T, k, E, C, lam, balance, gamma, used, base, kept, offsets, stats, ent, defer);
}

// Expert-parallel placement of a rank's slots (adj == nullptr: none).  With
// experts split over ranks, a slot's rank among all ranks' slots routed to
// its expert is its local slot-major rank plus adj[j*E + e] (the earlier
// slots of the other ranks, from the exchanged counts); it is kept iff that
// global rank is below C, and then goes to row rank + send[j*E + e] of the
// rank's send buffer (rows grouped by owner rank, expert, slot, token).
struct EpMap {
  const int* adj;
  const int* send;
  int C;
};

// Ranks of one pass and the slots' places.  Pass 1: p = offsets[e] + rank
// (offsets == nullptr: the bare rank, kept for a second pass).  Pass 2
// (used = the first pass's kept rows): a rerouted slot lands after its new
// expert's first-pass rows, p = offsets[e] + used[e] + rank; a slot the
// first pass kept gets p = offsets[e0] + rank1.  Expert parallel (ep.adj):
// p = rank + ep.send[j*E + e] when rank + ep.adj[j*E + e] < ep.C.
// Synchronisation of the DT threads that place one chunk: the whole block
// (assign_kernel), or one named barrier for a 256-thread group of a larger
// block (dispatch_small_kernel).
struct BlockSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
struct GroupSync {
  int id;
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory"); }
};

// The placement of chunk `chunk` by DT threads (gtid = 0 .. DT-1 among
// them); sm = their E * (DW + 1) ints of shared memory.
template <typename Sync>
__device__ __forceinline__ void assign_chunk(const SlotSrc& S, int T, int k, int E, bool token_major, int CH,
                                             int chunk, int gtid, int* sm, const int* __restrict__ base,
                                             const int* __restrict__ kept, const int* __restrict__ offsets,
                                             const int* __restrict__ used, int* __restrict__ pos, const EpMap& ep,
                                             Sync sync) {
  int* runcnt = sm;       // [E]
  int* warpcnt = sm + E;  // [DW][E]
  for (int i = gtid; i < E * (DW + 1); i += DT) sm[i] = 0;
  sync();
  const int lane = gtid & 31, warp = gtid >> 5;
  const long long nslots = static_cast<long long>(T) * k;
  const long long s0 = static_cast<long long>(chunk) * CH;
  const int* bbase = base + static_cast<size_t>(chunk) * E;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < CH / DT; ++r) {
    if (s0 + static_cast<long long>(r) * DT >= nslots) break;  // uniform across the DT threads
    const long long s = s0 + static_cast<long long>(r) * DT + gtid;
    int t = 0, j = 0, e = -1, e0 = -1;
    const bool in = s < nslots;
    if (in) {
      e = pass_expert(S, T, k, token_major, s, t, j, e0);
      if (e >= E) e = -1;
    }
    const int key = in ? e : -2;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    const int lrank = __popc(same & lt_mask);
    if (e >= 0 && lane == __ffs(same) - 1) warpcnt[warp * E + e] = __popc(same);
    sync();
    if (in) {
      int p = -1;
      if (e >= 0) {
        int prefix = 0;
        for (int w2 = 0; w2 < warp; ++w2) prefix += warpcnt[w2 * E + e];
        const int rank = bbase[e] + runcnt[e] + prefix + lrank;
        if (ep.adj) {
          const int je = j * E + e;
          if (rank + ep.adj[je] < ep.C) p = rank + ep.send[je];
        } else {
          // kept[e] = min(routed[e], C) (+ the first pass's rows): a slot is
          // kept iff its rank is below its pass's share, which also keeps
          // every position inside [offsets[e], offsets[e+1])
          const int u = used ? used[e] : 0;
          if (rank < kept[e] - u) p = (offsets ? offsets[e] : 0) + u + rank;
        }
      } else if (used && e0 >= 0 && e0 < E) {
        const int r1 = S.rank1[static_cast<size_t>(t) * k + j];
        if (r1 >= 0) p = offsets[e0] + r1;
      }
      pos[static_cast<size_t>(t) * k + j] = p;
    }
    sync();
    for (int e2 = gtid; e2 < E; e2 += DT) {
      int add = 0;
      for (int w2 = 0; w2 < DW; ++w2) {
        add += warpcnt[w2 * E + e2];
        warpcnt[w2 * E + e2] = 0;
      }
      runcnt[e2] += add;
    }
    sync();
  }
}

__global__ void __launch_bounds__(DT) assign_kernel(SlotSrc S, int T, int k, int E, bool token_major, int CH,
                                                    const int* __restrict__ base, const int* __restrict__ kept,
                                                    const int* __restrict__ offsets, const int* __restrict__ used,
                                                    int* __restrict__ pos, EpMap ep, StatsFinish fin) {
  pdl_entry();
  if (fin.sums && blockIdx.x == gridDim.x - 1) {
    // the extra block: the statistics' fp64 finish, beside the placement
    if (threadIdx.x < 32) stats_finish_warp(*fin.sums, fin, static_cast<int>(threadIdx.x));
    return;
  }
  extern __shared__ int sm[];
  assign_chunk(S, T, k, E, token_major, CH, blockIdx.x, threadIdx.x, sm, base, kept, offsets, used, pos, ep,
               BlockSync{});
}

// Pass 1 of a small batch in one CTA of 1024 threads: the slot histogram per
// 1024-slot chunk (at most kSmallChunks chunks, at most kSmallMaxE experts)
// in shared memory, the capacity scan over it, then the placement, one
// chunk per 256-thread group.  The same integer steps as slot_hist_kernel,
// capacity_scan_kernel and assign_kernel, so the same results, in one
// launch instead of three.  Measured per layer step: tiny fp32 (128 slots)
// 0.044-0.049 -> 0.039 ms; with 8 chunks (small prefill, 8192 slots) one
// CTA was 3% slower than the three kernels' 8 CTAs, hence 4 chunks at most.
constexpr int kSmallChunks = 4;
constexpr int kSmallMaxE = 128;

__global__ void __launch_bounds__(1024) dispatch_small_kernel(SlotSrc S, int T, int k, int E, bool token_major,
                                                              int C, float lam, int balance, float gamma,
                                                              int* __restrict__ base, int* __restrict__ kept,
                                                              int* __restrict__ offsets, int* __restrict__ pos,
                                                              moe_stats* stats, const float* __restrict__ ent) {
  pdl_entry();
  extern __shared__ int sm[];  // hist [nb][E+1], then four groups' E * (DW + 1)
  constexpr int CH = 1024;
  const long long nslots = static_cast<long long>(T) * k;
  const int nb = static_cast<int>((nslots + CH - 1) / CH);
  int* hist = sm;
  for (int i = threadIdx.x; i < nb * (E + 1); i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (long long s = threadIdx.x; s < nslots; s += blockDim.x) {
    int t, j, e0;
    const int e = pass_expert(S, T, k, token_major, s, t, j, e0);
    atomicAdd(&hist[static_cast<int>(s / CH) * (E + 1) + ((e >= 0 && e < E) ? e : E)], 1);
  }
  __syncthreads();
  capacity_scan_block(hist, nb, T, k, E, C, lam, balance, gamma, nullptr, base, kept, offsets, stats, ent, nullptr);
  __syncthreads();  // the bases, kept and offsets it wrote are visible to the block
  const int g = threadIdx.x / DT;
  int* scratch = sm + nb * (E + 1) + g * E * (DW + 1);
  for (int b = g; b < nb; b += 1024 / DT)
    assign_chunk(S, T, k, E, token_major, CH, b, threadIdx.x % DT, scratch, base, kept, offsets, nullptr, pos,
                 EpMap{nullptr, nullptr, 0}, GroupSync{1 + g});
}

// One warp per (token, column chunk): copy row x[t] to its kept
// destinations in Xp.  Small batches split each row into `chunks` pieces so
// that enough warps are in flight.
template <typename V>
__global__ void permute_kernel(const V* __restrict__ x, int T, int k, int vec_per_row, int chunks,
                               const int* __restrict__ pos, V* __restrict__ Xp) {
  pdl_entry();
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int t = static_cast<int>(wid / chunks);
  const int ch = static_cast<int>(wid - static_cast<long long>(t) * chunks);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) p[j] = j < k ? pos[static_cast<size_t>(t) * k + j] : -1;
  const V* src = x + static_cast<size_t>(t) * vec_per_row;
  const int per = (vec_per_row + chunks - 1) / chunks;
  const int v1 = min(vec_per_row, (ch + 1) * per);
  for (int v = ch * per + lane; v < v1; v += 32) {
    const V val = src[v];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (p[j] >= 0) Xp[static_cast<size_t>(p[j]) * vec_per_row + v] = val;
  }
}

// One warp per (token, column chunk): y[t] = sum_j w[t,j] Yp[pos[t,j]]
// (+ Sx[t]); 8 bf16 per lane step.
template <int KM>  // slots per token rounded up to 2, 4 or 8 (register arrays)
__global__ void combine_bf16_kernel(const uint4* __restrict__ Yp, const int* __restrict__ pos,
                                    const float* __restrict__ w, const uint4* __restrict__ Sx, int T, int k,
                                    int vec_per_row, int chunks, uint4* __restrict__ y) {
  pdl_entry();
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int t = static_cast<int>(wid / chunks);
  const int ch = static_cast<int>(wid - static_cast<long long>(t) * chunks);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int p[KM];
  float wt[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    p[j] = j < k ? pos[static_cast<size_t>(t) * k + j] : -1;
    wt[j] = j < k ? w[static_cast<size_t>(t) * k + j] : 0.f;
  }
  const int per = (vec_per_row + chunks - 1) / chunks;
  const int v1 = min(vec_per_row, (ch + 1) * per);
  for (int v = ch * per + lane; v < v1; v += 32) {
    // every row's 16 bytes are requested before the first is used
    uint4 q[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j)
      q[j] = p[j] >= 0 ? Yp[static_cast<size_t>(p[j]) * vec_per_row + v] : make_uint4(0, 0, 0, 0);
    const uint4 qs = Sx ? Sx[static_cast<size_t>(t) * vec_per_row + v] : make_uint4(0, 0, 0, 0);
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (p[j] >= 0) {
        const uint32_t u[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[2 * i] = fmaf(wt[j], bf16lo(u[i]), a[2 * i]);
          a[2 * i + 1] = fmaf(wt[j], bf16hi(u[i]), a[2 * i + 1]);
        }
      }
    }
    if (Sx) {
      const uint32_t u[4] = {qs.x, qs.y, qs.z, qs.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[2 * i] += bf16lo(u[i]);
        a[2 * i + 1] += bf16hi(u[i]);
      }
    }
    y[static_cast<size_t>(t) * vec_per_row + v] =
        make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]), pack_bf16(a[6], a[7]));
  }
}

__global__ void combine_f32_kernel(const float* __restrict__ Yp, const int* __restrict__ pos,
                                   const float* __restrict__ w, const float* __restrict__ Sx, int T, int k, int d,
                                   float* __restrict__ y) {
  pdl_entry();
  const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  for (int c = lane; c < d; c += 32) {
    float a = 0.f;
    for (int j = 0; j < k; ++j) {
      const int p = pos[static_cast<size_t>(t) * k + j];
      if (p >= 0) a = fmaf(w[static_cast<size_t>(t) * k + j], Yp[static_cast<size_t>(p) * d + c], a);
    }
    if (Sx) a += Sx[static_cast<size_t>(t) * d + c];
    y[static_cast<size_t>(t) * d + c] = a;
  }
}

// counts[j*E + e] = the slots (t, j) routed to expert e: the per-slot
// histogram that expert-parallel ranks exchange.  Integer atomics, so the
// result does not depend on their order.
__global__ void slot_counts_kernel(const int* __restrict__ idx, int T, int k, int E, int* __restrict__ counts) {
  pdl_entry();
  extern __shared__ int hc[];  // k * E
  for (int i = threadIdx.x; i < k * E; i += blockDim.x) hc[i] = 0;
  __syncthreads();
  const long long n = static_cast<long long>(T) * k;
  for (long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; s < n;
       s += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = idx[s];
    if (e >= 0 && e < E) atomicAdd(&hc[static_cast<int>(s % k) * E + e], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k * E; i += blockDim.x)
    if (hc[i]) atomicAdd(&counts[i], hc[i]);
}

// One warp per row: dst[map[i]] = src[i] (scatter) or dst[i] = src[map[i]]
// (gather), rows of vec_per_row 16-byte vectors; map[i] < 0 skips row i.
__global__ void permute_rows_kernel(const uint4* __restrict__ src, const int* __restrict__ map, long long n,
                                    int vec_per_row, int scatter, uint4* __restrict__ dst) {
  pdl_entry();
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const int m = map[i];
  if (m < 0) return;
  const uint4* s = src + (scatter ? i : static_cast<long long>(m)) * vec_per_row;
  uint4* d = dst + (scatter ? static_cast<long long>(m) : i) * vec_per_row;
  for (int v = lane; v < vec_per_row; v += 32) d[v] = s[v];
}

inline int n_chunks(const moe_config& cfg) {
  const long long n = static_cast<long long>(cfg.T) * cfg.k;
  const int ch = chunk_slots(n);
  return static_cast<int>((n + ch - 1) / ch);
}

inline unsigned warp_grid(int T, int chunks = 1) {
  return static_cast<unsigned>((static_cast<long long>(T) * chunks * 32 + 255) / 256);
}

// Column chunks per row for the per-token copy kernels: enough warps to
// keep the memory system busy when the batch is small.
inline int row_chunks(int T, int vec_per_row) {
  int c = 1;
  while (c < 8 && static_cast<long long>(T) * c < 4096 && vec_per_row / (2 * c) >= 32) c *= 2;
  return c;
}

}  // namespace

size_t dispatch_scratch_bytes(const moe_config& cfg) {
  const size_t nb = n_chunks(cfg);
  size_t b = align_up(nb * (cfg.E + 1) * sizeof(int), 256) + align_up(nb * cfg.E * sizeof(int), 256);
  b += align_up(sizeof(StatSums), 256);  // the statistics' integer totals (no rerouting)
  if (cfg.route_flags & MOE_ROUTE_REROUTE)
    b += align_up(static_cast<size_t>(cfg.E) * sizeof(int), 256) +
         align_up(static_cast<size_t>(cfg.T) * cfg.k * sizeof(int), 256);
  return b;
}

moe_status launch_dispatch(const moe_config& cfg, int C, const int* idx, const void* x, int* kept, int* offsets,
                           int* pos, void* Xp, moe_stats* stats, void* scratch, const int* backup,
                           cudaStream_t stream, const float* ent) {
  const int nb = n_chunks(cfg);
  uint8_t* sp = static_cast<uint8_t*>(scratch);
  int* blockhist = reinterpret_cast<int*>(sp);
  sp += align_up(static_cast<size_t>(nb) * (cfg.E + 1) * sizeof(int), 256);
  int* base = reinterpret_cast<int*>(sp);
  sp += align_up(static_cast<size_t>(nb) * cfg.E * sizeof(int), 256);
  const bool tm = (cfg.route_flags & MOE_ROUTE_TOKEN_MAJOR) != 0;
  const bool reroute = (cfg.route_flags & MOE_ROUTE_REROUTE) != 0;
  if (reroute && !backup) return MOE_ERR_UNSUPPORTED;
  const int CH = chunk_slots(static_cast<long long>(cfg.T) * cfg.k);
  const size_t asmem = static_cast<size_t>(cfg.E) * (DW + 1) * sizeof(int);
  const SlotSrc S1{idx, nullptr, nullptr};
  const long long nslots = static_cast<long long>(cfg.T) * cfg.k;
  if (!reroute && nslots <= static_cast<long long>(kSmallChunks) * 1024 && cfg.E <= kSmallMaxE) {
    // a small batch: histogram, scan and placement in one CTA
    const int nbs = static_cast<int>((nslots + 1023) / 1024);
    const size_t smem = sizeof(int) * (static_cast<size_t>(nbs) * (cfg.E + 1) +
                                       static_cast<size_t>(1024 / DT) * cfg.E * (DW + 1));
    launch_pdl(dispatch_small_kernel, dim3(1), dim3(1024), smem, stream, S1, cfg.T, cfg.k, cfg.E, tm, C,
               cfg.lambda_balance, cfg.balance, cfg.balance_gamma, base, kept, offsets, pos, stats, ent);
  } else if (!reroute) {
    launch_pdl(slot_hist_kernel, dim3(nb), dim3(DT), (cfg.E + 1) * sizeof(int), stream, S1, cfg.T, cfg.k, cfg.E, tm, CH,
               blockhist);
    // with statistics the scan hands their integer totals to an extra block
    // of the assignment kernel, which forms the fp64 figures beside the
    // placement (13.1 -> 10.0 us of scan on the small prefill went to
    // integer sums; the rest of the fp64 leaves the chain here)
    StatSums* sums = stats ? reinterpret_cast<StatSums*>(sp) : nullptr;
    const StatsFinish fin{sums, stats, cfg.T, cfg.k, cfg.E, C, cfg.balance, cfg.lambda_balance, cfg.balance_gamma};
    launch_pdl(capacity_scan_kernel, dim3(1), dim3(1024), 0, stream, blockhist, nb, cfg.T, cfg.k, cfg.E, C,
               cfg.lambda_balance, cfg.balance, cfg.balance_gamma, nullptr, base, kept, offsets, stats, ent, sums);
    launch_pdl(assign_kernel, dim3(nb + (sums ? 1 : 0)), dim3(DT), asmem, stream, S1, cfg.T, cfg.k, cfg.E, tm, CH,
               base, kept, offsets, nullptr, pos, EpMap{nullptr, nullptr, 0}, fin);
  } else {
    // pass 1 keeps its ranks; pass 2 offers the dropped slots their backups
    // in the same priority order, then places every slot
    int* kept1 = reinterpret_cast<int*>(sp);
    sp += align_up(static_cast<size_t>(cfg.E) * sizeof(int), 256);
    int* rank1 = reinterpret_cast<int*>(sp);
    launch_pdl(slot_hist_kernel, dim3(nb), dim3(DT), (cfg.E + 1) * sizeof(int), stream, S1, cfg.T, cfg.k, cfg.E, tm, CH,
               blockhist);
    launch_pdl(capacity_scan_kernel, dim3(1), dim3(1024), 0, stream, blockhist, nb, cfg.T, cfg.k, cfg.E, C,
               cfg.lambda_balance, cfg.balance, cfg.balance_gamma, nullptr, base, kept1, offsets, stats, ent,
               nullptr);
    launch_pdl(assign_kernel, dim3(nb), dim3(DT), asmem, stream, S1, cfg.T, cfg.k, cfg.E, tm, CH, base, kept1, nullptr,
               nullptr, rank1, EpMap{nullptr, nullptr, 0}, StatsFinish{nullptr, nullptr, 0, 0, 0, 0, 0, 0.f, 0.f});
    const SlotSrc S2{idx, rank1, backup};
    launch_pdl(slot_hist_kernel, dim3(nb), dim3(DT), (cfg.E + 1) * sizeof(int), stream, S2, cfg.T, cfg.k, cfg.E, tm, CH,
               blockhist);
    launch_pdl(capacity_scan_kernel, dim3(1), dim3(1024), 0, stream, blockhist, nb, cfg.T, cfg.k, cfg.E, C,
               cfg.lambda_balance, cfg.balance, cfg.balance_gamma, kept1, base, kept, offsets, stats, nullptr,
               nullptr);
    launch_pdl(assign_kernel, dim3(nb), dim3(DT), asmem, stream, S2, cfg.T, cfg.k, cfg.E, tm, CH, base, kept, offsets,
               kept1, pos, EpMap{nullptr, nullptr, 0}, StatsFinish{nullptr, nullptr, 0, 0, 0, 0, 0, 0.f, 0.f});
  }
  if (Xp) {
    const int es = cfg.dtype == MOE_BF16 ? 2 : 4;
    const long long row_bytes = static_cast<long long>(cfg.d) * es;
    if (row_bytes % 16 == 0) {
      const int vpr = static_cast<int>(row_bytes / 16);
      const int ch = row_chunks(cfg.T, vpr);
      launch_pdl(permute_kernel<uint4>, dim3(warp_grid(cfg.T, ch)), dim3(256), 0, stream, static_cast<const uint4*>(x),
                 cfg.T, cfg.k, vpr, ch, pos, static_cast<uint4*>(Xp));
    } else {
      const int vpr = static_cast<int>(row_bytes / 4);
      const int ch = row_chunks(cfg.T, vpr);
      launch_pdl(permute_kernel<uint32_t>, dim3(warp_grid(cfg.T, ch)), dim3(256), 0, stream,
                 static_cast<const uint32_t*>(x), cfg.T, cfg.k, vpr, ch, pos, static_cast<uint32_t*>(Xp));
    }
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Fixed device scratch for moe_dispatch_static: the chunk histograms and
// per-chunk bases of the kernels above, held in a file-scope array of this
// library instead of caller workspace.  Every word a dispatch reads from it
// was written earlier in the same call (slot_hist writes all (E+1) counters
// of every chunk, the scan writes every base), so nothing needs clearing.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_dispatch_scratch[kStaticDispatchScratchBytes];

moe_status static_dispatch_scratch(size_t need, void** ptr) {
  if (need > kStaticDispatchScratchBytes) return MOE_ERR_UNSUPPORTED;
  // The array's name is a host-side stand-in in host code; its device
  // address on the current device is looked up on every call (the lookup
  // allocates nothing).  No address is cached, so a cudaDeviceReset that
  // reloads the module -- and may place the array elsewhere -- cannot leave
  // a stale pointer behind.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  *ptr = p;
  return MOE_OK;
}

moe_status launch_slot_counts(const moe_config& cfg, const int* idx, int* counts, cudaStream_t stream) {
  moe_status s = launch_zero(counts, static_cast<size_t>(cfg.k) * cfg.E * sizeof(int), nullptr, 0, stream);
  if (s != MOE_OK) return s;
  const long long n = static_cast<long long>(cfg.T) * cfg.k;
  long long blocks = (n + 255) / 256;
  if (blocks > 1184) blocks = 1184;
  launch_pdl(slot_counts_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256),
             static_cast<size_t>(cfg.k) * cfg.E * sizeof(int), stream, idx, cfg.T, cfg.k, cfg.E, counts);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t dispatch_ep_scratch_bytes(const moe_config& cfg) {
  return dispatch_scratch_bytes(cfg) + align_up(static_cast<size_t>(2 * cfg.E + 1) * sizeof(int), 256);
}

moe_status launch_dispatch_ep(const moe_config& cfg, const int* idx, const void* x, const int* adj, const int* send,
                              int C, int* pos, void* Xsend, void* scratch, cudaStream_t stream) {
  const int nb = n_chunks(cfg);
  uint8_t* sp = static_cast<uint8_t*>(scratch);
  int* blockhist = reinterpret_cast<int*>(sp);
  sp += align_up(static_cast<size_t>(nb) * (cfg.E + 1) * sizeof(int), 256);
  int* base = reinterpret_cast<int*>(sp);
  sp += align_up(static_cast<size_t>(nb) * cfg.E * sizeof(int), 256);
  int* kept = reinterpret_cast<int*>(sp);  // E local counts (no local capacity), then E+1 offsets: unused
  int* offsets = kept + cfg.E;
  const int CH = chunk_slots(static_cast<long long>(cfg.T) * cfg.k);
  const size_t asmem = static_cast<size_t>(cfg.E) * (DW + 1) * sizeof(int);
  const SlotSrc S1{idx, nullptr, nullptr};
  launch_pdl(slot_hist_kernel, dim3(nb), dim3(DT), (cfg.E + 1) * sizeof(int), stream, S1, cfg.T, cfg.k, cfg.E, false,
             CH, blockhist);
  // local slot-major ranks only: the capacity test is on the global rank
  launch_pdl(capacity_scan_kernel, dim3(1), dim3(1024), 0, stream, blockhist, nb, cfg.T, cfg.k, cfg.E, 0x7fffffff, 0.f,
             0, 0.f, nullptr, base, kept, offsets, nullptr, nullptr, nullptr);
  launch_pdl(assign_kernel, dim3(nb), dim3(DT), asmem, stream, S1, cfg.T, cfg.k, cfg.E, false, CH, base, kept, offsets,
             nullptr, pos, EpMap{adj, send, C}, StatsFinish{nullptr, nullptr, 0, 0, 0, 0, 0, 0.f, 0.f});
  if (Xsend) {
    const int es = cfg.dtype == MOE_BF16 ? 2 : 4;
    const long long row_bytes = static_cast<long long>(cfg.d) * es;
    if (row_bytes % 16) return MOE_ERR_UNSUPPORTED;
    const int vpr = static_cast<int>(row_bytes / 16);
    const int ch = row_chunks(cfg.T, vpr);
    launch_pdl(permute_kernel<uint4>, dim3(warp_grid(cfg.T, ch)), dim3(256), 0, stream, static_cast<const uint4*>(x),
               cfg.T, cfg.k, vpr, ch, pos, static_cast<uint4*>(Xsend));
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_permute_rows(const void* src, const int* map, long long n, long long row_bytes, int scatter,
                               void* dst, cudaStream_t stream) {
  if (n <= 0) return MOE_OK;
  if (row_bytes <= 0 || row_bytes % 16) return MOE_ERR_UNSUPPORTED;
  const long long blocks = (n * 32 + 255) / 256;
  if (blocks > 2147483647LL) return MOE_ERR_UNSUPPORTED;
  launch_pdl(permute_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
             static_cast<const uint4*>(src), map, n, static_cast<int>(row_bytes / 16), scatter,
             static_cast<uint4*>(dst));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}


moe_status launch_combine(const moe_config& cfg, const void* Yp, const int* pos, const float* w, const void* Sx,
                          void* y, cudaStream_t stream) {
  if (cfg.dtype == MOE_BF16) {
    const int ch = row_chunks(cfg.T, cfg.d / 8);
    const uint4* yp = static_cast<const uint4*>(Yp);
    const uint4* sx = static_cast<const uint4*>(Sx);
    uint4* yo = static_cast<uint4*>(y);
    if (cfg.k <= 2)
      launch_pdl(combine_bf16_kernel<2>, dim3(warp_grid(cfg.T, ch)), dim3(256), 0, stream, yp, pos, w, sx, cfg.T, cfg.k,
                 cfg.d / 8, ch, yo);
    else if (cfg.k <= 4)
      launch_pdl(combine_bf16_kernel<4>, dim3(warp_grid(cfg.T, ch)), dim3(256), 0, stream, yp, pos, w, sx, cfg.T, cfg.k,
                 cfg.d / 8, ch, yo);
    else
      launch_pdl(combine_bf16_kernel<8>, dim3(warp_grid(cfg.T, ch)), dim3(256), 0, stream, yp, pos, w, sx, cfg.T, cfg.k,
                 cfg.d / 8, ch, yo);
  } else {
    launch_pdl(combine_f32_kernel, dim3(warp_grid(cfg.T)), dim3(256), 0, stream, static_cast<const float*>(Yp), pos, w,
               static_cast<const float*>(Sx), cfg.T, cfg.k, cfg.d, static_cast<float*>(y));
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

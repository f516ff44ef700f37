/*
 * moe.h -- C ABI of the B300 (sm_103a) sparse Mixture-of-Experts FFN layer.
 *
 * One layer, forward (and backward for training): router -> softmax/top-k ->
 * capacity-limited dispatch -> k expert FFNs (GeLU or SwiGLU) + an optional
 * always-on shared expert -> weighted combine -> load statistics.
 *
 * Sources (page title -- section):
 *   [P1] "'More parameters is better' is not the story: the expert group
 *        quietly activated inside a large model" (mlqm.cn) -- 3.1 Router,
 *        3.3 Gate, 4.2 model definition, 4.3 training configuration.
 *   [P2] "MoE mixture-of-experts architecture: principles and engineering
 *        practice" (cnnetsun.cn) -- 3.2 router (and its auxiliary loss), 4.1
 *        expert fusion, 4.2 building an MoE model, 5.2 normalising the
 *        router's input.
 *   [P3] "MoE architecture revealed: why total parameters != active
 *        parameters" (rkmt.cn) -- 2.3 router design (noise, capacity,
 *        dropping or rerouting, the balance loss), 3.3 TinyMoE, 5.3 (k = 1
 *        first).
 *   [P4] "GPT-4 has 1.8 trillion parameters and uses 2% of them per token"
 *        (wmrh.cn) -- 2.2 dynamic routing, 5.1 MVP.
 *   [P5] "Training a 200B LLM from scratch 5/25: how does MoE compute with
 *        part of its parameters?" (shanhuang.net) -- "Who decides which
 *        experts to call?", "Shared experts".
 *
 * Conventions (every entry point):
 *  - Ownership: the caller allocates every buffer, the workspace included.
 *    The library never allocates or frees device memory and keeps no state
 *    between calls, apart from a per-process cache of driver entry points
 *    and the fixed scratch array behind moe_dispatch_static.
 *  - Pointers: device pointers unless stated, 16-byte aligned.  Tensors are
 *    dense row-major.  Storage type = cfg->dtype (fp32 or bf16) for
 *    activations and weights; routing weights, noise, the expert bias and
 *    statistics are always fp32; indices int32.
 *  - Weight layout ("out x in", the contraction dimension contiguous):
 *    Wr[E,d]; W1 (gate), W3 (up) [E,h,d]; W2 [E,d,h]; b1 [E,h]; b2 [E,d];
 *    shared Ws1, Ws3 [h,d]; Ws2 [d,h]; bs1 [h]; bs2 [d].
 *  - Asynchrony: work is enqueued on `stream`; no call synchronises the host
 *    except moe_check_error.  Statistics are written to device memory.
 *  - Workspace: it serves one call at a time -- calls that share one must be
 *    ordered (the same stream, or events).  Its first 256 bytes are a
 *    header: the error word and the grouped GEMMs' tile counter, which every
 *    entry point zeroes before its first launch, so a fresh workspace needs
 *    no set-up; the rest is scratch that each call writes before it reads.
 *  - Errors: argument checks happen before any launch and return
 *    MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE with no
 *    work enqueued.  A failed launch returns MOE_ERR_CUDA.  Non-finite router
 *    logits never trap: that token is routed to no expert (idx = -1, w = 0)
 *    and counted in moe_stats.numeric_error.  Kernels that wait on on-chip
 *    barriers give up after a bounded time and record a nonzero code in the
 *    workspace error word (read it with moe_check_error).
 *  - Fixed rules: top-k ties go to the lower expert index; capacity is
 *    granted in slot-major priority (every token's first choice in token
 *    order, then every second choice, ...) unless MOE_ROUTE_TOKEN_MAJOR.
 *  - Limits: 1 <= k <= min(E, 8); 1 <= E <= 1024; T >= 1; T*k <= 2^30; for
 *    bf16, d and h multiples of 8 (16-byte rows); moe_layer_bwd: bf16 with
 *    d and h multiples of 64, not with MOE_ROUTE_RAW_PROBS and
 *    MOE_ROUTE_LAYERNORM together; MOE_ROUTE_REROUTE: k <= 4.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* = cudaStream_t; NULL = legacy default */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_CUDA = 3,
  MOE_ERR_WORKSPACE = 4,
  MOE_ERR_TIMEOUT = 5
} moe_status;

enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 };
enum { MOE_F32 = 0, MOE_BF16 = 1 };

/* Routing variants (moe_config.route_flags, a bit set; 0 = the defaults).
 *  MOE_ROUTE_RAW_PROBS: the weights are the selected entries of the softmax
 *    over all E experts, not renormalised over the k ([P2] 3.2: output =
 *    p1*e1 + p2*e2; [P4] 5.1 uses the top-k probabilities as they are).
 *    moe_layer_bwd then gives every logit a gradient (the softmax's
 *    denominator) and needs the forward's saved logits (moe_saved.logits);
 *    not combined with MOE_ROUTE_LAYERNORM in the backward.
 *  MOE_ROUTE_TOKEN_MAJOR: capacity is granted token by token (all of token
 *    t's choices, in order, before token t+1's) instead of slot-major.
 *  MOE_ROUTE_LAYERNORM: the router sees LayerNorm(x[t]) = (x[t] - mean) /
 *    sqrt(biased variance + 1e-5), unit scale and zero shift ([P2] 5.2, a
 *    LayerNorm in front of the linear router); the experts still see x.
 *    bf16 needs the workspace path of moe_route (ws != NULL); moe_layer_bwd
 *    returns its gradient through the normalisation.
 *  MOE_ROUTE_REROUTE: a slot over capacity tries its token's next-best
 *    expert before it is dropped ([P3] 2.3).  The router also records each
 *    token's experts ranked k .. 2k-1 (its backups).  After the usual pass,
 *    the r-th dropped slot of token t (r in slot order) is offered
 *    backup r, in the same priority order.  It is kept if that expert has
 *    room left, and is placed after the expert's first-pass rows.  The
 *    slot keeps its weight w[t,j] and idx keeps the router's choice; pos
 *    and offsets show the serving expert.  Needs k <= 4 and a workspace:
 *    moe_route writes the backups into ws, moe_dispatch reads them from
 *    the same ws.  moe_dispatch_static returns MOE_ERR_UNSUPPORTED.  In
 *    moe_layer_bwd a rerouted slot's logit gradient goes to idx[t,j] and
 *    its expert gradients to the backup that served it. */
enum { MOE_ROUTE_RAW_PROBS = 1, MOE_ROUTE_TOKEN_MAJOR = 2, MOE_ROUTE_LAYERNORM = 4, MOE_ROUTE_REROUTE = 8 };

/* Tile choices of the forward expert GEMMs (moe_config.gemm_flags; no effect
 * on any result bit, only on speed; the pages have no counterpart).  CTA
 * pair tiles: groups averaging >= 256 rows run 256-row tiles on clusters of
 * two CTAs on two SMs, one tcgen05 M=256 MMA (cta_group::2) per K step,
 * each CTA staging half of the rows and half of the weight tile.  They raise
 * tensor-pipe activity per cycle, which pays in a short launch (the small
 * prefill, T=4096 d=1024 h=2816 E=16: 0.176 -> 0.169 ms per layer) but, in
 * a long one held at the power cap, draws the clock down by more (the
 * large prefill: ~10% slower).
 *  0 (default): pair tiles for an expert GEMM of under 2e11 FLOPs (counted
 *    over the T k routed rows and the shared expert's T rows), single-CTA
 *    tiles above;
 *  MOE_GEMM_CTA_PAIRS: pair tiles for every expert GEMM;
 *  MOE_GEMM_SINGLE_CTA: single-CTA tiles for every expert GEMM.
 * Setting both is MOE_ERR_INVALID_ARG. */
enum { MOE_GEMM_CTA_PAIRS = 1, MOE_GEMM_SINGLE_CTA = 2 };

/* Load-balance term (moe_config.balance).  f[e] = counts[e]/T (pre-capacity
 * usage), g[e] = I[e]/T with I[e] the sum of the routing weights of the
 * slots routed to e (the importance of [P4] 2.2).  moe_stats.balance_stat
 * is the form on f; the backward differentiates the form on g (the counts
 * are piecewise constant).
 *  MOE_BALANCE_CV (0): lambda * std_{n-1}(f) / (mean(f) + 1e-8)  ([P1] 3.1).
 *  MOE_BALANCE_STD_MAX (1): lambda * (std_{n-1}(f) + gamma * max(f)), gamma =
 *    balance_gamma ([P2] 3.2: gamma = 100); the max's gradient goes to the
 *    lowest-index expert among the largest g.
 *  MOE_BALANCE_SWITCH (2): lambda * sum_e f[e] * g[e] ([P3] 2.3's product of
 *    two per-expert batch sums, read as usage fraction times mean routing
 *    weight); the backward holds f constant.  moe_dispatch alone cannot
 *    form it (it has no weights) and reports NaN; moe_layer_fwd fills it. */
enum { MOE_BALANCE_CV = 0, MOE_BALANCE_STD_MAX = 1, MOE_BALANCE_SWITCH = 2 };

/* Layer shape and routing rule.  [P2] 4.2 (capacity_factor, min_capacity),
 * [P1] 4.3 (load_balancing_loss_coef 0.01). */
typedef struct {
  int T;                 /* tokens in the batch                                */
  int d;                 /* model width                                        */
  int h;                 /* expert hidden width                                */
  int E;                 /* routed experts                                     */
  int k;                 /* experts per token                                  */
  int act;               /* MOE_ACT_GELU | MOE_ACT_SWIGLU                      */
  int dtype;             /* MOE_F32 | MOE_BF16                                 */
  float capacity_factor; /* C = max(min_capacity, ceil(cf*T*k/E)); <= 0: C = T */
  int min_capacity;      /* floor on C (0 = none)                              */
  float lambda_balance;  /* lambda of the usage statistic (0.01)               */
  int has_shared;        /* 1: add the always-on shared expert                 */
  int route_flags;       /* MOE_ROUTE_* bits, 0 = renormalised, slot-major     */
  int balance;           /* MOE_BALANCE_*, 0 = the CV form                     */
  float balance_gamma;   /* gamma of MOE_BALANCE_STD_MAX (100 in [P2] 3.2)     */
  int gemm_flags;        /* MOE_GEMM_* bits, 0 = the default tiles             */
} moe_config;

typedef struct {
  const void* Wr;            /* [E,d]                                   */
  const void* W1;            /* [E,h,d] gate (GeLU: the only input proj) */
  const void* W3;            /* [E,h,d] up (SwiGLU only)                 */
  const void* W2;            /* [E,d,h]                                  */
  const void* b1;            /* [E,h] GeLU only, nullable                */
  const void* b2;            /* [E,d] GeLU only, nullable                */
  const void* Ws1;           /* [h,d] shared expert                      */
  const void* Ws3;           /* [h,d]                                    */
  const void* Ws2;           /* [d,h]                                    */
  const void* bs1;           /* [h] nullable                             */
  const void* bs2;           /* [d] nullable                             */
  const float* expert_bias;  /* [E] fp32 added to every token's logits, nullable */
} moe_weights;

/* Activations a training forward keeps for the backward (device, caller-owned). */
typedef struct {
  int* idx;      /* [T,k]  selected experts (-1: none)                     */
  float* w;      /* [T,k]  routing weights                                 */
  int* counts;   /* [E]    slots routed to each expert (before capacity)   */
  int* kept;     /* [E]    slots kept after capacity                       */
  int* offsets;  /* [E+1]  first row of each expert in Xp/H/Yp             */
  int* pos;      /* [T,k]  row of slot (t,j) in Xp/H/Yp, -1 if dropped     */
  void* Xp;      /* [T*k, d] tokens permuted to expert-contiguous order    */
  void* H;       /* [T*k, h] activated hidden rows                         */
  void* Yp;      /* [T*k, d] expert outputs, permuted order                */
  void* Sx;      /* [T, d]   shared-expert output (has_shared)             */
  /* Pre-activations and the shared hidden rows, written by a training
   * forward when non-NULL and read by moe_layer_bwd (bf16 layers only).
   * Z and Zs are fp32, whatever the storage type: the backward evaluates
   * silu'/gelu' on them, and a bf16 copy would put a 2^-9 rounding there. */
  float* Z;      /* [T*k, 2h] SwiGLU gate | up  (GeLU: [T*k, h], W1 v + b1) */
  void* Hs;      /* [T, h]   shared expert's activated hidden rows          */
  float* Zs;     /* [T, 2h]  shared expert's pre-activations (GeLU [T, h])  */
  float* logits; /* [T, E]   the router's final logits (bias, noise and the
                              LayerNorm applied), fp32: written by a bf16
                              forward when non-NULL; moe_layer_bwd reads them
                              with MOE_ROUTE_RAW_PROBS                       */
} moe_saved;

/* Gradients written by moe_layer_bwd (device, fp32, caller-owned).  Every
 * listed tensor is overwritten, including the experts that received no
 * rows (zero). */
typedef struct {
  float* dX;    /* [T,d]                                                    */
  float* dWr;   /* [E,d]                                                    */
  float* dW1;   /* [E,h,d]                                                  */
  float* dW3;   /* [E,h,d] SwiGLU                                           */
  float* dW2;   /* [E,d,h]                                                  */
  float* db1;   /* [E,h] GeLU, nullable                                     */
  float* db2;   /* [E,d] GeLU, nullable                                     */
  float* dWs1;  /* [h,d] has_shared                                         */
  float* dWs3;  /* [h,d] has_shared, SwiGLU                                 */
  float* dWs2;  /* [d,h] has_shared                                         */
  float* dbs1;  /* [h] has_shared, GeLU, nullable                           */
  float* dbs2;  /* [d] has_shared, GeLU, nullable                           */
} moe_grads;

/* Load statistics ([P1] 3.1, 4.2; [P3] 2.3 drop monitoring). */
typedef struct {
  long long routed_slots;  /* sum of counts                                 */
  long long kept_slots;    /* sum of kept                                   */
  long long dropped_slots; /* T*k - kept_slots                              */
  int capacity;            /* C                                             */
  int numeric_error;       /* tokens with a non-finite logit                */
  double drop_rate;        /* dropped_slots / (T*k)                         */
  double balance_stat;     /* cfg->balance's form on counts/T (MOE_BALANCE_*) */
  double router_entropy;   /* mean over tokens with finite logits of
                              -sum_e p_e ln p_e, p = softmax over all E
                              ([P3] monitoring: alert below 0.3); written by
                              moe_layer_fwd; moe_dispatch alone leaves NaN  */
  long long rerouted_slots; /* slots kept by a backup expert
                               (MOE_ROUTE_REROUTE; counted in kept_slots)  */
} moe_stats;

/* C = max(min_capacity, ceil(cf*T*k/E)) or T when cf <= 0 ([P3] 2.3:
 * (1024*2)/16 = 128).  Host only.  MOE_ERR_INVALID_ARG on a bad config. */
moe_status moe_capacity(const moe_config* cfg, int* C_out);

/* Bytes of workspace the entry points below need for this config.
 * training = 0: moe_layer_fwd with saved == NULL keeps every intermediate in
 * the workspace.  training = 1: intermediates live in moe_saved; the
 * workspace holds scratch only (also enough for moe_dispatch and
 * moe_expert_ffn).  training = 2: moe_layer_bwd's scratch. */
moe_status moe_workspace_size(const moe_config* cfg, int training, size_t* bytes);

/* Router ([P1] 3.1 "logits = h W_r", softmax, top-k; [P1] 3.3 weights
 * renormalised over the top-k; [P3] 2.3 Gumbel noise on the router score).
 *   l[t,e] = x[t].Wr[e] (+ expert_bias[e]) (+ noise[t,e])  (fp32 accumulate)
 *   idx[t,:] = the k largest l[t,:], larger first, ties -> lower index
 *   w[t,j]   = exp(l[idx_j] - l[idx_0]) / sum_j' exp(l[idx_j'] - l[idx_0])
 *   counts[e] = #slots routed to e (zeroed by this call)
 * (cfg->route_flags MOE_ROUTE_RAW_PROBS: w[t,j] = softmax over all E of
 * l[t,:] at idx_j.)
 * x [T,d], Wr [E,d] in cfg->dtype; expert_bias [E], noise [T,E] fp32,
 * both nullable.  Outputs idx [T,k] int32, w [T,k] fp32, counts [E] int32,
 * entropy [T] fp32 (nullable): -sum_e p_e ln p_e of each token's softmax
 * over all experts, NaN for a token with a non-finite logit.
 * (MOE_ROUTE_LAYERNORM: l uses LayerNorm(x[t]) in place of x[t];
 * MOE_ROUTE_REROUTE: each token's experts ranked k .. 2k-1 are also left in
 * ws for moe_dispatch.)
 * ws: NULL, or >= moe_workspace_size(cfg, 1) bytes.  bf16 with ws: the
 * logits run on the tcgen05 tensor cores; up to 64 experts the top-k is
 * taken in the same kernel's epilogue, else (or with MOE_ROUTE_LAYERNORM or
 * MOE_ROUTE_REROUTE) the logits go through the workspace to a top-k pass.
 * Without ws a fused mma.sync kernel (MOE_ROUTE_LAYERNORM and
 * MOE_ROUTE_REROUTE then return MOE_ERR_UNSUPPORTED).  All sum in a fixed
 * order, so results repeat bit for bit; the paths may differ in the last
 * bits of l (and of w and the entropy). */
moe_status moe_route(const moe_config* cfg, const void* x, const void* Wr,
                     const float* expert_bias, const float* noise, int* idx,
                     float* w, int* counts, float* entropy, void* ws,
                     moe_stream_t stream);

/* Capacity and dispatch ([P3] 2.3 capacity and dropped tokens; [P1] 4.2
 * step 2, grouping the tokens bound for the same expert).
 *   slot-major ranks -> kept[e] = min(routed to e, C), offsets = exclusive
 *   scan of kept, pos[t,j] = offsets[e] + rank or -1, Xp[pos[t,j]] = x[t].
 * idx [T,k] int32 from moe_route; x [T,d].  Outputs kept [E], offsets [E+1],
 * pos [T,k] int32; Xp [T*k, d] (rows >= offsets[E] untouched); stats:
 * device moe_stats*, nullable (balance_stat in cfg->balance's form; NaN for
 * MOE_BALANCE_SWITCH, which needs the weights).  ws: >= moe_workspace_size(
 * cfg, 1) bytes; with MOE_ROUTE_REROUTE it must hold the backups moe_route
 * left there, and a second pass offers the dropped slots to them (kept[e]
 * then counts both passes). */
moe_status moe_dispatch(const moe_config* cfg, const int* idx, const void* x,
                        int* kept, int* offsets, int* pos, void* Xp,
                        moe_stats* stats, void* ws, moe_stream_t stream);

/* moe_dispatch without a workspace argument.  The pages have no counterpart
 * of this call: it exists for callers that cannot allocate device memory
 * at the point where they dispatch -- for example a plugin or custom-op
 * host that hands an operator only its input and output buffers, or a
 * serving loop that reserves all of its device memory up front and forbids
 * cudaMalloc afterwards.  Same arguments, results and rules as moe_dispatch
 * (kept, offsets, pos, Xp, stats are bit-identical), minus `ws`.
 *   Scratch: a fixed array of 2,098,432 bytes inside this library, which
 *   every GPU that loads the library holds until the process exits.  A
 *   call whose scratch need exceeds it returns MOE_ERR_UNSUPPORTED before
 *   any launch; every T*k <= 2^20 (1,048,576 slots) fits at any E <= 1024.
 *   Allocation: none -- no cudaMalloc, cudaFree or allocating library call.
 *   Set-up: every call looks up the array's device address on the current
 *   device (cudaGetSymbolAddress, which allocates nothing) instead of
 *   keeping it from an earlier call, so an address cannot go stale across a
 *   cudaDeviceReset.  The first call on a device also loads the library's
 *   module there: make that first call before any stream capture.
 *   Sharing: all calls on a device share the one array and it keeps the
 *   last call's contents; nothing in it has to start at zero (each call
 *   writes every word it later reads).  Calls whose work overlaps on the
 *   GPU -- on different streams, or from different host threads -- race
 *   on it: order them on one stream or with events. */
moe_status moe_dispatch_static(const moe_config* cfg, const int* idx, const void* x,
                               int* kept, int* offsets, int* pos, void* Xp,
                               moe_stats* stats, moe_stream_t stream);

/* Expert parallelism ([P1] 4.2-4.3 and [P2] 4.1: experts on different GPUs,
 * tokens sent to them and back with all-to-all; [P5] "Experts on different
 * GPUs: a new kind of waiting").  R ranks each hold their own tokens and the
 * weights of a contiguous block of experts.  The layer keeps the one-GPU
 * result on the ranks' batches concatenated in rank order: the capacity C
 * is the global one, and slot-major priority runs over all ranks' first
 * choices (rank 0's tokens, then rank 1's, ...) before any second choice.
 * The ranks exchange their per-(slot, expert) counts (moe_slot_counts); from
 * all of them every rank derives the same plan -- for each of its slots
 * (j, e), the earlier slots of the other ranks routed to e (rank_adjust)
 * and the row where the slot's run starts in its send buffer (send_adjust);
 * the host computes the plan (the binding's ep module).  Rows then travel
 * by all-to-all: the send buffer holds each owner's rows, expert by expert,
 * each expert's rows in slot-major order. */

/* counts[j*E + e] = #{t : idx[t,j] = e}, int32 [k, E] (zeroed by this
 * call); idx [T,k] from moe_route. */
moe_status moe_slot_counts(const moe_config* cfg, const int* idx, int* counts, moe_stream_t stream);

/* moe_dispatch for one rank of an expert-parallel layer (slot-major
 * priority only; MOE_ROUTE_TOKEN_MAJOR and MOE_ROUTE_REROUTE return
 * MOE_ERR_UNSUPPORTED).  A slot (t,j) routed to e with local slot-major
 * rank L (the number of this rank's earlier slots routed to e) is kept iff
 * L + rank_adjust[j*E + e] < capacity, the global capacity; then pos[t,j] =
 * L + send_adjust[j*E + e] and Xsend[pos[t,j]] = x[t]; else pos[t,j] = -1.
 * rank_adjust, send_adjust: device int32 [k, E] from the plan.  Xsend: the
 * send buffer, as many rows as the plan sends (nullable: positions only).
 * ws: >= moe_workspace_size(cfg, 1) bytes. */
moe_status moe_dispatch_ep(const moe_config* cfg, const int* idx, const void* x, const int* rank_adjust,
                           const int* send_adjust, int capacity, int* pos, void* Xsend, void* ws,
                           moe_stream_t stream);

/* Row permutation on the device, rows of row_bytes (a multiple of 16):
 * scatter != 0: dst[map[i]] = src[i]; scatter == 0: dst[i] = src[map[i]];
 * for i < n, skipping map[i] < 0.  An expert-parallel owner scatters the
 * rows it received into expert-contiguous order (map: each row's place from
 * the plan), runs moe_expert_ffn there, and gathers the outputs back into
 * the received order for the return all-to-all. */
moe_status moe_permute_rows(const void* src, const int* map, long long n, long long row_bytes, int scatter,
                            void* dst, moe_stream_t stream);

/* Grouped expert FFN over expert-contiguous rows ([P2] 4.2 and [P3] 3.3:
 * Linear -> GELU -> Linear; SwiGLU gate/up; [P2] 4.1 all experts' weights
 * in one contiguous tensor).  For every expert e and row r in
 * [offsets[e], offsets[e+1]):
 *   GeLU:   H[r] = gelu(W1[e] Xp[r] + b1[e]);   Yp[r] = W2[e] H[r] + b2[e]
 *   SwiGLU: H[r] = silu(W1[e] Xp[r]) * (W3[e] Xp[r]);  Yp[r] = W2[e] H[r]
 * offsets is a device array of E+1 nondecreasing int32 with offsets[0] = 0
 * (rows past T*k are never written).  Xp, Yp [T*k, d], H [T*k, h] in
 * cfg->dtype; rows past offsets[E] are not written.  bf16 runs on the
 * tcgen05 tensor cores with fp32 accumulation; fp32 runs on the CUDA cores
 * in fp32.  ws: >= moe_workspace_size(cfg, 1) bytes (its error word is
 * reset here). */
moe_status moe_expert_ffn(const moe_config* cfg, const void* Xp, const int* offsets,
                          const void* W1, const void* W3, const void* b1,
                          const void* W2, const void* b2, void* H, void* Yp,
                          void* ws, moe_stream_t stream);

/* moe_expert_ffn plus the always-on shared expert ([P5] "Shared experts":
 * every token also passes through one more FFN), in the same two launches:
 * the shared expert is one more group of T rows with its own operands, so
 * its weight streaming overlaps the routed experts'.  In addition to
 * moe_expert_ffn's outputs:
 *   Hs[t] = act(Ws1 x[t] ...) [T,h];   Sx[t] = Ws2 Hs[t] (+ bs2)  [T,d]
 * bf16 only (MOE_ERR_UNSUPPORTED otherwise).  wts supplies W1, W3, b1, W2,
 * b2 and Ws1, Ws3, Ws2, bs1, bs2 (Wr and expert_bias are not read).
 * ws: >= moe_workspace_size(cfg, 1) bytes. */
moe_status moe_expert_ffn_shared(const moe_config* cfg, const void* Xp, const int* offsets,
                                 const moe_weights* wts, void* H, void* Yp, const void* x,
                                 void* Hs, void* Sx, void* ws, moe_stream_t stream);

/* Weighted combine / un-permute ([P5] "Who decides which experts to call?":
 * 0.75*[0.8,0.2,-0.4] + 0.25*[0.4,0.6,0.8] = [0.7,0.3,-0.1]; [P5] "Shared
 * experts": the shared path is added).
 *   y[t] = sum_{j: pos[t,j] >= 0} w[t,j] * Yp[pos[t,j]]  (+ Sx[t])
 * summed in fp32 in slot order j = 0..k-1, stored in cfg->dtype.  pos
 * entries index rows of Yp (< T*k).  Sx nullable. */
moe_status moe_combine(const moe_config* cfg, const void* Yp, const int* pos,
                       const float* w, const void* Sx, void* y, moe_stream_t stream);

/* The whole forward: route, dispatch, experts, shared expert, combine,
 * statistics.  noise [T,E] fp32 nullable.  saved: NULL (inference: every
 * intermediate lives in ws) or the buffers a backward needs.  stats:
 * device moe_stats*, nullable.  ws_bytes >= moe_workspace_size(cfg, saved
 * != NULL). */
moe_status moe_layer_fwd(const moe_config* cfg, const moe_weights* wts, const void* x,
                         const float* noise, void* y, moe_saved* saved,
                         moe_stats* stats, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* The whole backward of the layer (bf16; d and h multiples of 64), for the
 * loss L = <dY, y> + lambda * CV(I / T) where I[e] is the sum of the routing
 * weights of the slots routed to e ([P4] 2.2's importance, in [P1] 3.1's
 * std/mean form: std with n-1, mean + 1e-8); gradients reach the router and
 * the chosen experts ([P1] 3.3).  Per routed slot (t,j) -> e:
 *   G[t,j]  = [kept] <dY[t], Yp[pos[t,j]]> + d(lambda CV)/dw[t,j]
 *   dl[t,j] = w[t,j] (G[t,j] - sum_j' w[t,j'] G[t,j'])  (other logits: 0)
 *   dWr = sum_t dl[t]^T x[t];   dX[t] = sum_j dl[t,j] Wr[idx_j]
 *         + sum_{kept j} J_e(x[t])^T (w[t,j] dY[t]) + J_shared(x[t])^T dY[t]
 *   expert weights: the chain rule through W2 (act(...)) with
 *   silu'(z) = s (1 + z (1 - s)) and gelu'(z) = Phi(z) + z phi(z).
 * Noise and the expert bias are additive constants of the logits and get no
 * gradient.  x, wts: the forward's inputs; saved: the forward's moe_saved
 * with Z (and Zs with a shared expert) filled -- H and Hs are not read:
 * the backward forms w * act(z) again from the fp32 pre-activations, in
 * bf16 plus its bf16 residual, for the W2 gradients; dY [T,d] bf16.  The
 * expert GEMMs contract dY as stored and apply the routing weight in fp32.
 * Sums run in a fixed order (integers for the importance), so repeated
 * calls give the same bits.  ws_bytes >= moe_workspace_size(cfg, 2). */
moe_status moe_layer_bwd(const moe_config* cfg, const moe_weights* wts, const void* x,
                         const moe_saved* saved, const void* dY, const moe_grads* grads,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronises `stream`, then reads the workspace error word left by the
 * last call that used `ws`: MOE_OK, or MOE_ERR_TIMEOUT if a kernel gave up
 * a bounded wait (code_out receives the raw word, nullable). */
moe_status moe_check_error(const void* ws, int* code_out, moe_stream_t stream);

/* Self-test of the failure-detection path; the pages have no counterpart.
 * Enqueues one kernel whose single thread waits on a shared-memory barrier
 * that nothing completes.  The wait gives up after its bound (1 s), records
 * code 0x1ff in the workspace error word and returns, so the context stays
 * usable and moe_check_error(ws) then reports MOE_ERR_TIMEOUT.  The kernel
 * holds one SM for about a second.  ws: >= 256 bytes of device memory (the
 * error word is its first int, zeroed by this call). */
moe_status moe_selftest_wait_timeout(void* ws, moe_stream_t stream);

const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */

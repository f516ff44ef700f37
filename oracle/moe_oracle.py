"""Plain fp64 CPU oracle of the sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  This module is the checker the CUDA path is
compared against.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the library itself never calls
it, and it shares no code with the CUDA path.

Everything is numpy float64, single pass, written in the order the pages
state the method.  Library primitives used as single steps: ``@`` (matmul),
``np.lexsort`` (a sort), ``math.erf``/``np.exp``.  Inputs arrive as the
stored bits the GPU reads (fp32 or bf16 decoded exactly to fp64), so both
sides start from identical values.

Sources (page title -- section):
  [P1] "'More parameters is better' is not the story: the expert group
       quietly activated inside a large model" (mlqm.cn) -- 3.1 Router,
       3.3 Gate, 4.2 model definition, 4.3 training configuration.
  [P2] "MoE mixture-of-experts architecture: principles and engineering
       practice" (cnnetsun.cn) -- 3.2 router, 4.2 building an MoE model,
       5.2 normalising the router's input.
  [P3] "MoE architecture revealed: why total parameters != active
       parameters" (rkmt.cn) -- 2.3 router design, 3.3 TinyMoE.
  [P4] "GPT-4 has 1.8 trillion parameters and uses 2% of them per token"
       (wmrh.cn) -- 2.2 the meaning of 2% and dynamic routing, 5.1 MVP.
  [P5] "Training a 200B LLM from scratch 5/25: how does MoE compute with
       part of its parameters?" (shanhuang.net) -- "Who decides which
       experts to call?", "Shared experts", "200B is still there".

Readings of points the pages leave open (each also listed in the design
notes): no router bias (P1 4.2); top-k weights renormalised to sum to 1
(P1 3.3, 4.2; P3 3.3); ties broken towards the lower expert index, selection
on logits; Gumbel noise added to the logits before both selection and
weights (P3 2.3); capacity C = max(min_capacity, ceil(cf*T*k/E)), no limit
when cf <= 0 (P3 2.3); overflow decided in slot-major priority (all first
choices in token order, then all second choices); a dropped slot adds zero
and the kept weight is not renormalised; GeLU is the exact erf form;
SwiGLU is W2 (silu(W1 v) * (W3 v)); the shared expert is added with weight
1 (P5 "Shared experts"); usage statistic lambda*std_{n-1}(f)/(mean(f)+1e-8)
on pre-capacity counts f = counts/T (P1 3.1, 4.2); a token whose logits are
not all finite is routed to no expert.

Backward (training workload): the loss is L = <dY, y> + lambda*CV(I/T) with
I[e] = sum of the routing weights of the slots routed to e (P4 2.2's
"importance"), CV = std_{n-1}/(mean + 1e-8) -- the differentiable reading of
P1's balance term; its forward statistic stays the count-based one.
"""

from __future__ import annotations

import math
from fractions import Fraction
from typing import Dict, Optional

import numpy as np

# ----------------------------------------------------------------------------
# decoding of stored inputs
# ----------------------------------------------------------------------------


def decode(a) -> np.ndarray:
    """Stored tensor -> fp64 ndarray.  Accepts numpy arrays or torch tensors
    (fp32, or bf16 whose 16-bit patterns are widened exactly)."""
    if hasattr(a, "detach"):  # torch tensor, decoded without torch arithmetic
        t = a.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            bits = t.contiguous().view(dtype=__import__("torch").int16).numpy()
            u32 = (bits.astype(np.uint16).astype(np.uint32)) << 16
            return u32.view(np.float32).astype(np.float64)
        return t.numpy().astype(np.float64)
    return np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------
# routing  ([P1] 3.1, 3.3, 4.2; [P3] 2.3, 3.3)
# ----------------------------------------------------------------------------


LN_EPS = 1e-5


def layer_norm(x: np.ndarray) -> np.ndarray:
    """Row-wise (x - mean) / sqrt(var + 1e-5), var the biased (1/n) variance:
    [P2] 5.2's nn.LayerNorm in front of the router, at its initial identity
    scale and zero shift."""
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    return (x - mu) / np.sqrt(var + LN_EPS)


def layer_norm_backward(x: np.ndarray, g: np.ndarray) -> np.ndarray:
    """Gradient with respect to x of <g, layer_norm(x)> (chain rule of the
    row normalisation: r (g - mean(g) - n mean(g n)), n = layer_norm(x))."""
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    r = 1.0 / np.sqrt(var + LN_EPS)
    n = (x - mu) * r
    return r * (g - g.mean(axis=1, keepdims=True) - n * (g * n).mean(axis=1, keepdims=True))


def router_logits(x, Wr, expert_bias=None, noise=None, layernorm: bool = False) -> np.ndarray:
    """l[t,e] = sum_i x[t,i] Wr[e,i] (+ bias[e]) (+ G[t,e]).

    [P1] 3.1: "logits = h W_r"; [P3] 2.3: Gumbel noise is added to the router
    score before top-k.  The per-expert bias is an explicit input (a workload
    of skewed load).  layernorm: the router sees layer_norm(x) ([P2] 5.2);
    the experts still see x."""
    x = decode(x)
    Wr = decode(Wr)
    if layernorm:
        x = layer_norm(x)
    l = x @ Wr.T
    if expert_bias is not None:
        l = l + decode(expert_bias)[None, :]
    if noise is not None:
        l = l + decode(noise)
    return l


def top_k_route(l: np.ndarray, k: int, raw_probs: bool = False):
    """Top-k experts per token and their weights.

    Experts are ordered by (logit descending, index ascending); the first k
    are selected ([P1] 4.2 takes top-k of softmax(l); softmax is monotone, so
    ordering the logits gives the same set).  Weights (default) are the
    softmax of the selected logits, w_j = exp(l_j - l_0) / sum_j'
    exp(l_j' - l_0), which is [P1] 3.3's p_i/(p_i+p_j) and [P3] 3.3's softmax
    over the top-k logits.  raw_probs: the selected entries of the softmax
    over all E experts, not renormalised ([P2] 3.2: output = p1*e1 + p2*e2;
    [P4] 5.1 uses the top-k probabilities as they are).

    Returns idx [T,k] int64 (-1 for a token with a non-finite logit), w [T,k]
    fp64 (0 there), finite [T] bool."""
    T, E = l.shape
    idx = np.full((T, k), -1, dtype=np.int64)
    w = np.zeros((T, k), dtype=np.float64)
    finite = np.all(np.isfinite(l), axis=1)
    experts = np.arange(E)
    for t in range(T):
        if not finite[t]:
            continue
        order = np.lexsort((experts, -l[t]))  # primary: -l, secondary: index
        sel = order[:k]
        idx[t] = sel
        if raw_probs:
            z = np.exp(l[t] - l[t, sel[0]])
            w[t] = z[sel] / z.sum()
        else:
            z = np.exp(l[t, sel] - l[t, sel[0]])
            w[t] = z / z.sum()
    return idx, w, finite


def router_entropy(l: np.ndarray) -> float:
    """Mean over the tokens with finite logits of the entropy of the router's
    distribution, H_t = -sum_e p_te ln p_te with p_t = softmax(l_t) over all
    experts ([P3] 4.x monitoring: router_entropy, alert below 0.3).  NaN when
    no token has finite logits."""
    finite = np.all(np.isfinite(l), axis=1)
    if not finite.any():
        return float("nan")
    p = softmax(l[finite])
    with np.errstate(divide="ignore", invalid="ignore"):
        h = -np.where(p > 0, p * np.log(p), 0.0).sum(axis=1)
    return float(h.mean())


def softmax(l: np.ndarray) -> np.ndarray:
    """Row softmax over all experts ([P1] 3.1 p_i)."""
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------
# capacity and dispatch  ([P3] 2.3; [P1] 4.3; [P2] 4.2)
# ----------------------------------------------------------------------------


def expert_capacity(T: int, k: int, E: int, capacity_factor: float, min_capacity: int = 0) -> int:
    """C = max(min_capacity, ceil(cf * T * k / E)); no limit (C = T) if cf <= 0.

    [P3] 2.3's worked case: batch 1024, k=2, 16 experts -> (1024*2)/16 = 128.
    The ceiling is taken of the exact value of cf*T*k/E, cf being the binary
    number the caller passed (a rational), so no rounding of the product can
    move C by one."""
    if capacity_factor <= 0:
        return T
    c = math.ceil(Fraction(capacity_factor) * T * k / E)
    return max(int(min_capacity), int(c))


def usage_counts(idx: np.ndarray, E: int) -> np.ndarray:
    """counts[e] = number of (t, j) slots routed to e, before capacity."""
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.reshape(-1):
        if e >= 0:
            counts[e] += 1
    return counts


def assign_capacity(idx: np.ndarray, E: int, C: int, token_major: bool = False):
    """Queue simulation of the capacity rule.

    Slot-major priority (default): for j in 0..k-1, for t in 0..T-1; token-
    major: for t in 0..T-1, for j in 0..k-1.  The slot (t, j) gets the next
    free place of its expert if fewer than C are taken, else it is dropped
    ([P3] 2.3 / [P1] 4.3: tokens beyond capacity are dropped).
    Returns rank [T,k] (-1 dropped or unrouted) and fill[E] (kept per expert)."""
    T, k = idx.shape
    rank = np.full((T, k), -1, dtype=np.int64)
    fill = np.zeros(E, dtype=np.int64)
    order = [(t, j) for t in range(T) for j in range(k)] if token_major else \
        [(t, j) for j in range(k) for t in range(T)]
    for t, j in order:
        e = idx[t, j]
        if e < 0:
            continue
        if fill[e] < C:
            rank[t, j] = fill[e]
            fill[e] += 1
    return rank, fill


def backup_experts(l: np.ndarray, k: int) -> np.ndarray:
    """Each token's experts ranked k .. 2k-1 by (logit descending, index
    ascending): its next-best experts, which the slots that overflow can be
    rerouted to ([P3] 2.3).  -1 where fewer than 2k experts exist or the
    token's logits are not all finite.  Returns [T,k] int64."""
    T, E = l.shape
    b = np.full((T, k), -1, dtype=np.int64)
    nb = max(0, min(k, E - k))
    experts = np.arange(E)
    for t in range(T):
        if not np.all(np.isfinite(l[t])):
            continue
        order = np.lexsort((experts, -l[t]))
        b[t, :nb] = order[k:k + nb]
    return b


def reroute_overflow(idx: np.ndarray, backup: np.ndarray, rank: np.ndarray, fill: np.ndarray, C: int,
                     token_major: bool = False):
    """Second capacity pass: the slots the first pass dropped try their
    token's next-best experts ([P3] 2.3: tokens beyond capacity are dropped
    or routed to the next-best expert).

    The r-th dropped slot of token t (r counted in slot order j) tries
    backup[t, r] once.  Slots are visited in the first pass's priority order.
    A slot is kept if that expert has room left after the first pass and
    the slots rerouted to it before; it then takes that expert's next place
    after its first-pass rows.  Otherwise it stays dropped.
    Returns served [T,k] (the expert serving each slot, -1 for none), rank2
    [T,k] (place among the expert's rerouted rows, -1 if not rerouted) and
    fill2 [E] (rerouted rows per expert)."""
    T, k = idx.shape
    E = fill.shape[0]
    nth = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        r = 0
        for j in range(k):
            if idx[t, j] >= 0 and rank[t, j] < 0:
                nth[t, j] = r
                r += 1
    served = np.where(rank >= 0, idx, -1)
    rank2 = np.full((T, k), -1, dtype=np.int64)
    fill2 = np.zeros(E, dtype=np.int64)
    order = [(t, j) for t in range(T) for j in range(k)] if token_major else \
        [(t, j) for j in range(k) for t in range(T)]
    for t, j in order:
        if nth[t, j] < 0:
            continue
        b = backup[t, nth[t, j]]
        if b < 0:
            continue
        if fill[b] + fill2[b] < C:
            rank2[t, j] = fill2[b]
            fill2[b] += 1
            served[t, j] = b
    return served, rank2, fill2


def dispatch_positions(idx: np.ndarray, rank: np.ndarray, fill: np.ndarray):
    """offsets = exclusive prefix sum of the kept counts (experts in index
    order); a kept slot's row in the expert-contiguous buffer is
    offsets[e] + rank.  Returns offsets [E+1], pos [T,k] (-1 if not kept)."""
    E = fill.shape[0]
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + fill[e]
    pos = np.where(rank >= 0, offsets[np.maximum(idx, 0)] + rank, -1)
    return offsets, pos


BALANCE_VARIANTS = ("cv", "std_max", "switch")


def _std_n1(f: np.ndarray) -> float:
    """Standard deviation with the n-1 divisor (torch.std's default); 0 for
    a single value."""
    E = f.shape[0]
    if E < 2:
        return 0.0
    mean = f.sum() / E
    return math.sqrt(((f - mean) ** 2).sum() / (E - 1))


def importance(idx: np.ndarray, w: np.ndarray, E: int) -> np.ndarray:
    """I[e] = sum of the routing weights of the slots routed to e (before
    capacity): the importance of [P4] 2.2."""
    I = np.zeros(E, dtype=np.float64)
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            if idx[t, j] >= 0:
                I[idx[t, j]] += w[t, j]
    return I


def balance_stat(counts: np.ndarray, T: int, lam: float, variant: str = "cv", gamma: float = 100.0,
                 imp: np.ndarray = None) -> float:
    """The load statistic on pre-capacity usage f = counts / T.

    cv (default): lambda * std(f) / (mean(f) + 1e-8), std with n-1 --
      [P1] 3.1: L_balance = lambda * std(usage)/mean(usage); [P1] 4.2's code
      averages the one-hot selection over tokens and adds 1e-8 to the mean;
      torch.std there is the n-1 form.
    std_max: lambda * (std(f) + gamma * max(f)) -- [P2] 3.2's auxiliary loss
      on the experts' usage frequency, gamma = 100 in its DeepSeek-R1 setting.
    switch: lambda * sum_e f_e * P_e with P = imp / T, the mean routing
      weight each expert receives -- [P3] 2.3's product of two per-expert
      sums over the batch, read as usage fraction times mean weight (the
      page prints both factors alike)."""
    f = counts.astype(np.float64) / T
    E = f.shape[0]
    if variant == "cv":
        if E < 2:
            return 0.0  # one expert: nothing to balance (n-1 = 0)
        mean = f.sum() / E
        return lam * _std_n1(f) / (mean + 1e-8)
    if variant == "std_max":
        return lam * (_std_n1(f) + gamma * f.max())
    if variant == "switch":
        return lam * float((f * (np.asarray(imp, dtype=np.float64) / T)).sum())
    raise ValueError(variant)


# ----------------------------------------------------------------------------
# experts and combine  ([P2] 4.2; [P3] 3.3; [P1] 3.2; [P5])
# ----------------------------------------------------------------------------


def gelu(z):
    """Exact GeLU z * Phi(z) = z * (1 + erf(z / sqrt 2)) / 2 (nn.GELU default form)."""
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return z * 0.5 * (1.0 + erf(z / math.sqrt(2.0)))


def gelu_grad(z):
    erf = np.vectorize(math.erf, otypes=[np.float64])
    return 0.5 * (1.0 + erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def silu(z):
    """silu(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def expert_ffn(v: np.ndarray, act: str, W1, W2, W3=None, b1=None, b2=None) -> np.ndarray:
    """One expert FFN on rows v [n, d] -> [n, d].

    GeLU: W2 gelu(W1 v + b1) + b2 ([P2] 4.2, [P3] 3.3: Linear, GELU, Linear).
    SwiGLU: W2 (silu(W1 v) * (W3 v)) (gate W1, up W3, no biases)."""
    if act == "gelu":
        z = v @ W1.T
        if b1 is not None:
            z = z + b1[None, :]
        out = gelu(z) @ W2.T
        if b2 is not None:
            out = out + b2[None, :]
        return out
    if act == "swiglu":
        return (silu(v @ W1.T) * (v @ W3.T)) @ W2.T
    raise ValueError(act)


def combine(expert_out: np.ndarray, w: np.ndarray, kept: np.ndarray, shared: Optional[np.ndarray] = None):
    """y = sum over kept slots j of w_j * expert_out_j (+ shared).

    [P5] "Who decides which experts to call?": the two chosen experts'
    outputs are mixed with the routing proportions; [P5] "Shared experts":
    the shared expert's output is added.  expert_out [T,k,d], w [T,k],
    kept [T,k] bool."""
    T, k, d = expert_out.shape
    y = np.zeros((T, d), dtype=np.float64)
    for j in range(k):
        y += np.where(kept[:, j:j + 1], w[:, j:j + 1] * expert_out[:, j, :], 0.0)
    if shared is not None:
        y += shared
    return y


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------


def route_and_dispatch(cfg: dict, x, Wr, expert_bias=None, noise=None) -> Dict[str, np.ndarray]:
    """Router, top-k, capacity and dispatch of the whole batch (no experts)."""
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    l = router_logits(x, Wr, expert_bias, noise, layernorm=cfg.get("layernorm", False))
    idx, w, finite = top_k_route(l, k, raw_probs=cfg.get("raw_probs", False))
    counts = usage_counts(idx, E)
    C = expert_capacity(T, k, E, cfg.get("capacity_factor", 0.0), cfg.get("min_capacity", 0))
    rank, fill = assign_capacity(idx, E, C, token_major=cfg.get("token_major", False))
    served = np.where(rank >= 0, idx, -1)
    backup = None
    rerouted = 0
    if cfg.get("reroute"):
        backup = backup_experts(l, k)
        served, rank2, fill2 = reroute_overflow(idx, backup, rank, fill, C, cfg.get("token_major", False))
        offsets, _ = dispatch_positions(idx, rank, fill + fill2)
        # first-pass rows first, then the rerouted rows, in each expert
        pos = np.where(rank >= 0, offsets[np.maximum(idx, 0)] + rank,
                       np.where(rank2 >= 0, offsets[np.maximum(served, 0)] + fill[np.maximum(served, 0)] + rank2,
                                -1))
        fill = fill + fill2
        rerouted = int(fill2.sum())
    else:
        offsets, pos = dispatch_positions(idx, rank, fill)
    routed = int(counts.sum())
    kept_total = int(fill.sum())
    stats = dict(
        routed_slots=routed,
        kept_slots=kept_total,
        dropped_slots=T * k - kept_total,
        capacity=C,
        drop_rate=(T * k - kept_total) / (T * k),
        balance_stat=balance_stat(counts, T, cfg.get("lam", 0.01), cfg.get("balance", "cv"),
                                  cfg.get("gamma", 100.0), importance(idx, w, E)),
        numeric_error=int((~finite).sum()),
        router_entropy=router_entropy(l),
        rerouted_slots=rerouted,
    )
    return dict(logits=l, idx=idx, w=w, counts=counts, kept=fill, capacity=C,
                rank=rank, offsets=offsets, pos=pos, stats=stats, served=served, backup=backup)


def layer_forward(cfg: dict, weights: dict, x, expert_bias=None, noise=None,
                  tokens: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The whole forward pass; expert outputs computed for ``tokens`` only
    (all tokens if None).  Returns the routing results for the whole batch
    and y [len(tokens), d]."""
    r = route_and_dispatch(cfg, x, weights["Wr"], expert_bias, noise)
    X = decode(x)
    T, k, d = cfg["T"], cfg["k"], cfg["d"]
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    act = cfg["act"]
    out = np.zeros((len(toks), k, d), dtype=np.float64)
    kept = r["pos"][toks] >= 0
    idx = r["served"][toks]  # the expert serving each slot (a rerouted slot's backup)
    touched = np.zeros(len(toks), dtype=np.int64)
    for e in range(cfg["E"]):
        rows, slots = np.nonzero((idx == e) & kept)
        if rows.size == 0:
            continue
        We = expert_params(weights, e, act)
        out[rows, slots] = expert_ffn(X[toks[rows]], act, **We)
        np.add.at(touched, rows, sum(a.size for a in We.values() if a is not None))
    shared = None
    if cfg.get("has_shared"):
        Ws = shared_params(weights, act)
        shared = expert_ffn(X[toks], act, **Ws)
        touched += sum(a.size for a in Ws.values() if a is not None)
    y = combine(out, r["w"][toks], kept, shared)
    r.update(y=y, tokens=toks, expert_out=out, shared_out=shared, params_touched=touched)
    return r


def expert_params(weights: dict, e: int, act: str) -> dict:
    p = dict(W1=decode(weights["W1"][e]), W2=decode(weights["W2"][e]))
    if act == "swiglu":
        p["W3"] = decode(weights["W3"][e])
    else:
        p["b1"] = decode(weights["b1"][e]) if weights.get("b1") is not None else None
        p["b2"] = decode(weights["b2"][e]) if weights.get("b2") is not None else None
    return p


def shared_params(weights: dict, act: str) -> dict:
    p = dict(W1=decode(weights["Ws1"]), W2=decode(weights["Ws2"]))
    if act == "swiglu":
        p["W3"] = decode(weights["Ws3"])
    else:
        p["b1"] = decode(weights["bs1"]) if weights.get("bs1") is not None else None
        p["b2"] = decode(weights["bs2"]) if weights.get("bs2") is not None else None
    return p


# ----------------------------------------------------------------------------
# backward (training workload)
# ----------------------------------------------------------------------------


def expert_ffn_backward(v: np.ndarray, g_out: np.ndarray, act: str, W1, W2, W3=None, b1=None, b2=None):
    """Chain rule through one expert for rows v [n,d] with upstream g_out [n,d].

    Returns dict with dv [n,d], dW1, dW2 (and dW3 or db1/db2), plus the
    forward output of the rows (used by the routing-weight gradient)."""
    g = {}
    if act == "swiglu":
        a = v @ W1.T
        b = v @ W3.T
        hact = silu(a) * b
        out = hact @ W2.T
        dh = g_out @ W2
        da = dh * b * silu_grad(a)
        db = dh * silu(a)
        g["dW2"] = g_out.T @ hact
        g["dW1"] = da.T @ v
        g["dW3"] = db.T @ v
        g["dv"] = da @ W1 + db @ W3
    else:
        z = v @ W1.T
        if b1 is not None:
            z = z + b1[None, :]
        hact = gelu(z)
        out = hact @ W2.T
        if b2 is not None:
            out = out + b2[None, :]
        dh = g_out @ W2
        dz = dh * gelu_grad(z)
        g["dW2"] = g_out.T @ hact
        g["dW1"] = dz.T @ v
        g["db1"] = dz.sum(axis=0)
        g["db2"] = g_out.sum(axis=0)
        g["dv"] = dz @ W1
    g["out"] = out
    return g


def importance_cv_grad(idx: np.ndarray, w: np.ndarray, E: int, T: int, lam: float):
    """Value and gradient of lambda * std_{n-1}(I/T) / (mean(I/T) + 1e-8) with
    respect to each slot's weight, I[e] = sum of w over slots routed to e."""
    f = np.zeros(E, dtype=np.float64)
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            if idx[t, j] >= 0:
                f[idx[t, j]] += w[t, j]
    f /= T
    mean = f.sum() / E
    dev = f - mean
    std = math.sqrt((dev ** 2).sum() / (E - 1))
    val = lam * std / (mean + 1e-8)
    # d val / d f_e
    if std > 0:
        dstd = dev / ((E - 1) * std)
    else:
        dstd = np.zeros(E)
    dval_df = lam * (dstd / (mean + 1e-8) - std / (mean + 1e-8) ** 2 / E)
    dval_dw = np.where(idx >= 0, dval_df[np.maximum(idx, 0)] / T, 0.0)
    return val, dval_dw


def balance_term_grad(idx: np.ndarray, w: np.ndarray, E: int, T: int, lam: float, variant: str = "cv",
                      gamma: float = 100.0):
    """Value and per-slot weight gradient of the differentiable balance term
    on g = I/T (I = importance): the form of balance_stat with the counts
    replaced by the importance where the gradient flows.

    cv: lambda * CV(g) (importance_cv_grad).
    std_max: lambda * (std_{n-1}(g) + gamma * max(g)); the max's gradient goes
      to the lowest-index expert among the largest.
    switch: lambda * sum_e f_e g_e with f = counts / T, the usage fraction, a
      constant (it counts discrete choices)."""
    if variant == "cv":
        return importance_cv_grad(idx, w, E, T, lam)
    g = importance(idx, w, E) / T
    if variant == "std_max":
        sd = _std_n1(g)
        val = lam * (sd + gamma * g.max())
        dval = np.zeros(E)
        if E > 1 and sd > 0:
            dval += (g - g.sum() / E) / ((E - 1) * sd)
        dval[int(np.argmax(g))] += gamma  # argmax returns the first largest
        dval *= lam
    elif variant == "switch":
        f = usage_counts(idx, E).astype(np.float64) / T
        val = lam * float((f * g).sum())
        dval = lam * f
    else:
        raise ValueError(variant)
    return val, np.where(idx >= 0, dval[np.maximum(idx, 0)] / T, 0.0)


def layer_backward(cfg: dict, weights: dict, x, dY, expert_bias=None, noise=None) -> Dict[str, np.ndarray]:
    """Gradients of L = <dY, y> + B(I/T) for the whole (small) batch, B the
    balance term of cfg["balance"] (balance_term_grad; lambda*CV by default).

    Per slot: G[t,j] = [kept] <dY[t], FFN_e(x[t])> + dB/dw[t,j];
    logit gradient dl[t, idx_j] = w_j (G_j - sum_j' w_j' G_j') (softmax over
    the selected logits), other logits 0 -- or, with raw_probs (w_j = p_{idx_j}
    of the softmax over all E), dl[t, e] = p_e ([e selected] G_e - sum_j w_j
    G_j) for every e; dWr = dl^T x; dX = dl Wr + the experts' input
    gradients (routed rows scaled by w) + the shared expert's."""
    T, d, E, k = cfg["T"], cfg["d"], cfg["E"], cfg["k"]
    act = cfg["act"]
    lam = cfg.get("lam", 0.01)
    r = route_and_dispatch(cfg, x, weights["Wr"], expert_bias, noise)
    X = decode(x)
    DY = decode(dY)
    idx, w, pos = r["idx"], r["w"], r["pos"]
    # the expert that serves each kept slot: the router's choice, or with
    # rerouting a backup (whose output still carries the slot's weight w_j,
    # so the logit gradient stays on idx_j)
    served = r["served"]
    dX = np.zeros((T, d))
    G = np.zeros((T, k))
    grads = {}
    for name in ("W1", "W3", "W2"):
        if name in weights and weights[name] is not None:
            grads["d" + name] = np.zeros(decode(weights[name]).shape)
    if act == "gelu":
        grads["db1"] = np.zeros((E, cfg["h"]))
        grads["db2"] = np.zeros((E, d))
    y = np.zeros((T, d))
    for e in range(E):
        rows, slots = np.nonzero(served == e)
        if rows.size == 0:
            continue
        We = expert_params(weights, e, act)
        g_out = w[rows, slots][:, None] * DY[rows]
        g = expert_ffn_backward(X[rows], g_out, act, **We)
        G[rows, slots] += np.einsum("nd,nd->n", DY[rows], g["out"])
        y[rows] += w[rows, slots][:, None] * g["out"]
        np.add.at(dX, rows, g["dv"])
        for name in ("W1", "W3", "W2", "b1", "b2"):
            if "d" + name in g and "d" + name in grads:
                grads["d" + name][e] += g["d" + name]
    if cfg.get("has_shared"):
        Ws = shared_params(weights, act)
        g = expert_ffn_backward(X, DY, act, **Ws)
        dX += g["dv"]
        y += g["out"]
        grads["dWs1"] = g["dW1"]
        grads["dWs2"] = g["dW2"]
        if act == "swiglu":
            grads["dWs3"] = g["dW3"]
        else:
            grads["dbs1"] = g["db1"]
            grads["dbs2"] = g["db2"]
    val, dcv = balance_term_grad(idx, w, E, T, lam, cfg.get("balance", "cv"), cfg.get("gamma", 100.0))
    G += dcv
    dl = np.zeros((T, E))
    if cfg.get("raw_probs"):
        # w_j = p_{idx_j}, p the softmax over all E: every logit e gets
        # p_e ([e selected] G_e - sum_j w_j G_j)
        P = softmax(np.where(np.isfinite(r["logits"]), r["logits"], 0.0))
    for t in range(T):
        if idx[t, 0] < 0:
            continue
        s = (w[t] * G[t]).sum()
        if cfg.get("raw_probs"):
            dl[t] = -P[t] * s
            for j in range(k):
                dl[t, idx[t, j]] += P[t, idx[t, j]] * G[t, j]
        else:
            for j in range(k):
                dl[t, idx[t, j]] += w[t, j] * (G[t, j] - s)
    Wr = decode(weights["Wr"])
    if cfg.get("layernorm"):
        grads["dWr"] = dl.T @ layer_norm(X)
        dX += layer_norm_backward(X, dl @ Wr)
    else:
        grads["dWr"] = dl.T @ X
        dX += dl @ Wr
    grads["dX"] = dX
    grads["dlogits"] = dl
    grads["y"] = y
    grads["loss"] = float((DY * y).sum() + val)
    grads["balance_term"] = val
    grads.update(route=r)
    return grads


# ----------------------------------------------------------------------------
# sampled backward entries (for batches too large for layer_backward)
# ----------------------------------------------------------------------------


def _served(route: dict) -> np.ndarray:
    """The expert that serves each slot: the route's own map when it has one
    (with rerouting a dropped slot may be served by a backup), else the
    router's choice where the slot was kept and -1 where it was dropped."""
    if route.get("served") is not None:
        return route["served"]
    return np.where(route["pos"] >= 0, route["idx"], -1)


def _slot_dots(cfg: dict, weights: dict, X: np.ndarray, Y: np.ndarray, served: np.ndarray) -> np.ndarray:
    """G[i,j] = <Y[i], FFN_e(X[i])> for the expert e = served[i,j] of each
    kept slot (0 for a dropped slot): the upstream term of the routing
    weight's gradient."""
    act = cfg["act"]
    G = np.zeros(served.shape)
    for e in sorted(set(served[served >= 0].tolist())):
        rr, ss = np.nonzero(served == e)
        out = expert_ffn(X[rr], act, **expert_params(weights, e, act))
        G[rr, ss] = np.einsum("nd,nd->n", Y[rr], out)
    return G


def _logit_grads(cfg: dict, route: dict, toks: np.ndarray, G: np.ndarray) -> np.ndarray:
    """dl[i, e] for the listed tokens, layer_backward's rule: renormalised
    weights give w_j (G_j - sum_j' w_j' G_j') at the selected experts and 0
    elsewhere; raw softmax weights give p_e ([e selected] G_e - sum_j w_j G_j)
    at every expert (p the softmax of the route's logits)."""
    E, k = cfg["E"], cfg["k"]
    idx, w = route["idx"], route["w"]
    dl = np.zeros((len(toks), E))
    if cfg.get("raw_probs"):
        L = route["logits"][toks]
        P = softmax(np.where(np.isfinite(L), L, 0.0))
    for i, t in enumerate(toks):
        if idx[t, 0] < 0:
            continue
        s = (w[t] * G[i]).sum()
        if cfg.get("raw_probs"):
            dl[i] = -P[i] * s
            for j in range(k):
                dl[i, idx[t, j]] += P[i, idx[t, j]] * G[i, j]
        else:
            for j in range(k):
                dl[i, idx[t, j]] += w[t, j] * (G[i, j] - s)
    return dl


def _rows(a, ix) -> np.ndarray:
    """Rows ix of a stored tensor (numpy or torch, any device), decoded."""
    return decode(a[_as_index(a, ix)]) if hasattr(a, "index_select") else decode(a)[np.asarray(ix)]


def expert_grad_slices(cfg: dict, weights: dict, x, dY, route: dict, e: int, cols) -> Dict[str, np.ndarray]:
    """Weight gradients of expert e restricted to hidden units `cols`, summed
    over all of the rows the expert serves (with rerouting, a backup's rows
    include the slots moved to it): dW1[e][cols,:], dW3[e][cols,:] (or
    db1[e][cols] for GeLU) and dW2[e][:,cols].  The chain rule of
    expert_ffn_backward with the upstream gradient w[t,j] dY[t] of each
    served slot; a hidden unit's gradients depend only on that unit's row of
    W1/W3 and column of W2, so the slice is exact."""
    act = cfg["act"]
    cols = np.asarray(cols)
    rows, slots = np.nonzero(_served(route) == e)
    X = _rows(x, rows)
    Y = _rows(dY, rows)
    g_out = route["w"][rows, slots][:, None] * Y
    W1 = decode(weights["W1"][e][_as_index(weights["W1"], cols)])
    W2 = decode(weights["W2"][e][:, _as_index(weights["W2"], cols)])
    dh = g_out @ W2
    out = {}
    if act == "swiglu":
        W3 = decode(weights["W3"][e][_as_index(weights["W3"], cols)])
        a = X @ W1.T
        b = X @ W3.T
        hact = silu(a) * b
        out["dW1"] = (dh * b * silu_grad(a)).T @ X
        out["dW3"] = (dh * silu(a)).T @ X
    else:
        z = X @ W1.T
        if weights.get("b1") is not None:
            z = z + decode(weights["b1"][e])[cols][None, :]
        hact = gelu(z)
        dz = dh * gelu_grad(z)
        out["dW1"] = dz.T @ X
        out["db1"] = dz.sum(axis=0)
    out["dW2"] = g_out.T @ hact
    return out


def token_input_grads(cfg: dict, weights: dict, x, dY, route: dict, tokens) -> np.ndarray:
    """dX[t] for the listed tokens: the router term sum_e dl[t,e] Wr[e] (dl
    from layer_backward's rule, with the balance term over the whole batch;
    through the LayerNorm's backward when the router normalises), plus each
    served slot's expert input gradient for w[t,j] dY[t], plus the shared
    expert's for dY[t]."""
    T, E = cfg["T"], cfg["E"]
    act = cfg["act"]
    toks = np.asarray(tokens)
    idx, w = route["idx"], route["w"]
    served = _served(route)[toks]
    X = _rows(x, toks)
    Y = _rows(dY, toks)
    dX = np.zeros_like(X)
    G = np.zeros(served.shape)
    for e in sorted(set(served[served >= 0].tolist())):
        rr, ss = np.nonzero(served == e)
        g = _input_grad_rows(X[rr], w[toks[rr], ss][:, None] * Y[rr], act, expert_params(weights, e, act))
        np.add.at(dX, rr, g["dv"])
        G[rr, ss] = np.einsum("nd,nd->n", Y[rr], g["out"])
    if cfg.get("has_shared"):
        g = _input_grad_rows(X, Y, act, shared_params(weights, act))
        dX += g["dv"]
    _, dcv = balance_term_grad(idx, w, E, T, cfg.get("lam", 0.01), cfg.get("balance", "cv"),
                               cfg.get("gamma", 100.0))
    G += dcv[toks]
    g = _logit_grads(cfg, route, toks, G) @ decode(weights["Wr"])
    dX += layer_norm_backward(X, g) if cfg.get("layernorm") else g
    return dX


def router_grad_rows(cfg: dict, weights: dict, x, dY, route: dict, experts) -> np.ndarray:
    """Rows `experts` of the router weight gradient dWr over the whole
    batch: sum over tokens t of dl[t,e] x[t] (LayerNorm(x[t]) when the router
    normalises), dl by layer_backward's rule.  With renormalised weights
    dl[t,e] is 0 unless e is one of t's selected experts, so only the tokens
    routed to one of `experts` contribute, and only their slots' expert
    outputs are computed -- every served slot of each such token, since
    dl[t,e] involves the token's sum_j w_j G_j.  Raw softmax weights reach
    every row from every token; use layer_backward there."""
    if cfg.get("raw_probs"):
        raise ValueError("router_grad_rows: with raw softmax weights every token reaches every row")
    T, E = cfg["T"], cfg["E"]
    experts = np.asarray(experts)
    idx, w = route["idx"], route["w"]
    toks = np.nonzero(np.isin(idx, experts).any(axis=1))[0]
    X = _rows(x, toks)
    Y = _rows(dY, toks)
    G = _slot_dots(cfg, weights, X, Y, _served(route)[toks])
    _, dcv = balance_term_grad(idx, w, E, T, cfg.get("lam", 0.01), cfg.get("balance", "cv"),
                               cfg.get("gamma", 100.0))
    G += dcv[toks]
    dl = _logit_grads(cfg, route, toks, G)
    Xr = layer_norm(X) if cfg.get("layernorm") else X
    return dl[:, experts].T @ Xr


def _input_grad_rows(v, g_out, act, p):
    """Input gradient and output of one expert on rows v (no weight grads)."""
    if act == "swiglu":
        a = v @ p["W1"].T
        b = v @ p["W3"].T
        out = (silu(a) * b) @ p["W2"].T
        dh = g_out @ p["W2"]
        dv = (dh * b * silu_grad(a)) @ p["W1"] + (dh * silu(a)) @ p["W3"]
    else:
        z = v @ p["W1"].T
        if p.get("b1") is not None:
            z = z + p["b1"][None, :]
        out = gelu(z) @ p["W2"].T
        if p.get("b2") is not None:
            out = out + p["b2"][None, :]
        dv = ((g_out @ p["W2"]) * gelu_grad(z)) @ p["W1"]
    return dict(dv=dv, out=out)


def _as_index(t, ix):
    """Index array in the form `t` accepts (a torch tensor on t's device, or numpy)."""
    if hasattr(t, "index_select"):
        import torch
        return torch.as_tensor(np.asarray(ix), device=t.device)
    return np.asarray(ix)

"""Pins of the C++ fp64 oracle (oracle/moe_oracle.cpp), on the CPU.

Each step is held to what the pages or the mathematics fix, independently
of the oracle's own code: the pages' worked examples (the combine of
"Training a 200B LLM from scratch 5/25", the capacity of "MoE architecture
revealed" 2.3), brute force on tiny inputs, closed forms, torch and scipy
routines.  The whole forward is then held to the numpy oracle, itself pinned
in test_oracle_pins.py: integers bit for bit, floating point to 1e-12.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import moe_synth as S
from oracle import cpp
from oracle import moe_oracle as O


def test_capacity_rule():
    # "MoE architecture revealed" 2.3: batch 1024, top-2, 16 experts -> 128
    assert cpp.capacity(1024, 2, 16, 1.0) == 128
    # the workloads' capacities
    assert cpp.capacity(4096, 2, 16, 1.0) == 512
    assert cpp.capacity(16384, 2, 64, 1.25) == 640
    assert cpp.capacity(32768, 2, 16, 1.25) == 5120
    # no limit, and the floor
    assert cpp.capacity(300, 2, 7, 0.0) == 300
    assert cpp.capacity(300, 2, 7, -1.0) == 300
    assert cpp.capacity(100, 2, 16, 0.1, min_capacity=40) == 40
    # the exact ceiling of the fp32 factor's rational value
    rng = np.random.default_rng(3)
    for _ in range(2000):
        T, k, E = int(rng.integers(1, 1 << 20)), int(rng.integers(1, 9)), int(rng.integers(1, 1025))
        cf = np.float32(rng.uniform(0.01, 4.0))
        ref = math.ceil(Fraction(float(cf)) * T * k / E)
        assert cpp.capacity(T, k, E, float(cf)) == ref, (T, k, E, float(cf))
    # a factor whose product lands exactly on an integer, and the extremes
    assert cpp.capacity(1000, 2, 8, 1.25) == 313  # 312.5 -> 313
    assert cpp.capacity(640, 2, 5, 1.0) == 256
    assert cpp.capacity(64, 2, 4, 1e-30) == 1
    assert cpp.capacity(64, 2, 4, 1e30) == 2 ** 31 - 1


def test_combine_worked_example():
    """0.75 * [0.8, 0.2, -0.4] + 0.25 * [0.4, 0.6, 0.8] = [0.7, 0.3, -0.1]."""
    out = np.array([[[0.8, 0.2, -0.4], [0.4, 0.6, 0.8]]])
    y = cpp.combine(out, np.array([[0.75, 0.25]]), np.array([[True, True]]))
    np.testing.assert_allclose(y, [[0.7, 0.3, -0.1]], rtol=0, atol=1e-15)
    # a dropped slot adds nothing; the shared expert adds with weight 1
    y = cpp.combine(out, np.array([[0.75, 0.25]]), np.array([[True, False]]), shared=np.array([[1.0, 2.0, 3.0]]))
    np.testing.assert_allclose(y, [[1.6, 2.15, 2.7]], rtol=0, atol=1e-15)


def _beats(l, a, b):
    """Expert a precedes b: larger logit, or equal logit and lower index."""
    return l[a] > l[b] or (l[a] == l[b] and a < b)


def test_top_k_brute_force():
    rng = np.random.default_rng(5)
    for E, k in ((5, 2), (6, 3), (4, 1), (4, 4)):
        l = rng.normal(size=(300, E))
        l[::7, 1] = l[::7, 3]  # exact ties
        idx, w, nf = cpp.top_k(l, k)
        assert nf == 0
        for t in range(l.shape[0]):
            sel = list(idx[t])
            # brute force over all k-subsets: the chosen one is the only set
            # whose every member precedes every other expert
            ok = [s for s in itertools.combinations(range(E), k)
                  if all(_beats(l[t], a, b) for a in s for b in range(E) if b not in s)]
            assert ok == [tuple(sorted(sel))]
            assert all(_beats(l[t], sel[j], sel[j + 1]) for j in range(k - 1))
            ref = [math.exp(l[t, e]) for e in sel]
            np.testing.assert_allclose(w[t], np.array(ref) / sum(ref), rtol=1e-13, atol=0)
            assert abs(w[t].sum() - 1.0) < 1e-14


def test_top_k_ties_and_nonfinite():
    l = np.array([[1.0, 1.0, 1.0, 1.0], [1.0, 3.0, 3.0, 2.0], [0.0, np.nan, 1.0, 2.0], [np.inf, 0.0, 0.0, 0.0]])
    idx, w, nf = cpp.top_k(l, 2)
    assert idx[0].tolist() == [0, 1] and idx[1].tolist() == [1, 2]
    np.testing.assert_allclose(w[0], [0.5, 0.5], rtol=0, atol=1e-15)
    assert idx[2].tolist() == [-1, -1] and idx[3].tolist() == [-1, -1] and nf == 2
    assert not w[2].any() and not w[3].any()


def test_router_logits_definition():
    rng = np.random.default_rng(7)
    x = torch.tensor(rng.normal(size=(9, 24)), dtype=torch.bfloat16)
    Wr = torch.tensor(rng.normal(size=(5, 24)), dtype=torch.bfloat16)
    bias = rng.normal(size=5).astype(np.float32)
    noise = rng.gumbel(size=(9, 5)).astype(np.float32)
    l = cpp.router_logits(x, Wr, bias, noise)
    ref = x.double().numpy() @ Wr.double().numpy().T + bias.astype(np.float64) + noise.astype(np.float64)
    np.testing.assert_allclose(l, ref, rtol=1e-13, atol=1e-13)


def test_capacity_queue_and_positions():
    """Slot-major queue against a direct simulation: all first choices in
    token order, then all second choices; each expert takes up to C."""
    rng = np.random.default_rng(11)
    T, k, E, C = 500, 3, 7, 160
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    idx[rng.random(T) < 0.05] = -1  # unrouted tokens
    counts = cpp.usage_counts(idx, E)
    np.testing.assert_array_equal(counts, np.bincount(idx[idx >= 0], minlength=E))
    rank, fill = cpp.assign_capacity(idx, E, C)
    queue = {e: [] for e in range(E)}
    for j in range(k):
        for t in range(T):
            if idx[t, j] >= 0:
                queue[idx[t, j]].append((t, j))
    for e in range(E):
        assert fill[e] == min(len(queue[e]), C)
        for r, (t, j) in enumerate(queue[e]):
            assert rank[t, j] == (r if r < C else -1)
    assert (rank[idx < 0] == -1).all()
    offsets, pos = cpp.dispatch_positions(idx, rank, fill)
    assert offsets[0] == 0 and (np.diff(offsets) == fill).all()
    kept = pos >= 0
    # every kept slot has one row of its expert's block, and rows follow the queue
    assert sorted(pos[kept].tolist()) == list(range(int(fill.sum())))
    for e in range(E):
        rows = [pos[t, j] for t, j in queue[e][:C]]
        assert rows == list(range(offsets[e], offsets[e + 1]))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_expert_ffn_against_torch(act):
    """One expert as torch's fp64 dense FFN (exact-erf GeLU with biases, or
    SwiGLU), on rows and weights stored in bf16."""
    g = torch.Generator().manual_seed(13)
    n, d, h = 11, 40, 56
    v = torch.randn(n, d, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(h, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    W3 = (torch.randn(h, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn(d, h, generator=g) / h ** 0.5).to(torch.bfloat16)
    b1 = (torch.randn(h, generator=g) * 0.3).to(torch.bfloat16)
    b2 = (torch.randn(d, generator=g) * 0.3).to(torch.bfloat16)
    vd, W1d, W3d, W2d, b1d, b2d = (a.double() for a in (v, W1, W3, W2, b1, b2))
    if act == "gelu":
        got = cpp.expert_ffn(v, "gelu", W1, W2, b1=b1, b2=b2)
        ref = torch.nn.functional.gelu(vd @ W1d.T + b1d) @ W2d.T + b2d
    else:
        got = cpp.expert_ffn(v, "swiglu", W1, W2, W3=W3)
        ref = (torch.nn.functional.silu(vd @ W1d.T) * (vd @ W3d.T)) @ W2d.T
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_balance_statistic_and_entropy():
    from scipy.stats import entropy
    counts = np.array([30, 10, 0, 24, 16], dtype=np.int64)
    T, lam = 40, 0.01
    f = torch.tensor(counts / T, dtype=torch.float64)
    ref = lam * float(f.std(unbiased=True)) / (float(f.mean()) + 1e-8)
    assert abs(cpp.balance_stat(counts, T, lam) - ref) <= 1e-15
    assert cpp.balance_stat(np.array([7], dtype=np.int64), T, lam) == 0.0
    assert cpp.balance_stat(np.full(4, 9, dtype=np.int64), T, lam) == 0.0
    rng = np.random.default_rng(17)
    l = rng.normal(size=(50, 6)) * 2
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    assert abs(cpp.router_entropy(l) - float(np.mean([entropy(r) for r in p]))) <= 1e-13
    assert abs(cpp.router_entropy(np.zeros((3, 6))) - math.log(6)) <= 1e-14
    l[0, 2] = np.nan  # a non-finite token is left out of the mean
    assert abs(cpp.router_entropy(l) - float(np.mean([entropy(r) for r in p[1:]]))) <= 1e-13
    assert math.isnan(cpp.router_entropy(np.full((2, 3), np.nan)))


LAYERS = [
    # GeLU in fp32 with biases, no capacity limit
    S.WORKLOADS["tiny_fp32"].replace(T=40, seed=21),
    # SwiGLU in bf16 with the shared expert, Gumbel noise and a binding capacity
    S.WORKLOADS["training"].replace(T=160, d=48, h=64, E=6, capacity_factor=0.7, seed=23),
    # a skewed router bias and k = 3
    S.WORKLOADS["small_prefill"].replace(T=150, d=32, h=40, E=5, k=3, capacity_factor=0.9, zipf_s=1.1, seed=29),
]


@pytest.mark.parametrize("wl", LAYERS, ids=lambda w: w.name)
def test_layer_forward_matches_numpy_oracle(wl):
    t = S.make_inputs(wl, "cpu")
    cfg = dict(T=wl.T, d=wl.d, h=wl.h, E=wl.E, k=wl.k, act=wl.act, capacity_factor=float(np.float32(wl.capacity_factor)),
               min_capacity=wl.min_capacity, lam=0.01, has_shared=wl.has_shared)
    c = cpp.layer_forward(cfg, t, t["x"], t.get("expert_bias"), t.get("noise"))
    n = O.layer_forward(cfg, t, t["x"], t.get("expert_bias"), t.get("noise"))
    for key in ("idx", "counts", "kept", "offsets", "pos"):
        np.testing.assert_array_equal(c[key], n[key], err_msg=key)
    np.testing.assert_allclose(c["w"], n["w"], rtol=0, atol=1e-14)
    scale = max(1.0, float(np.abs(n["y"]).max()))
    np.testing.assert_allclose(c["y"], n["y"], rtol=0, atol=1e-12 * scale)
    for key in ("routed_slots", "kept_slots", "dropped_slots", "capacity", "numeric_error"):
        assert c["stats"][key] == n["stats"][key], key
    for key in ("drop_rate", "balance_stat", "router_entropy"):
        assert abs(c["stats"][key] - n["stats"][key]) <= 1e-12 * max(1.0, abs(n["stats"][key])), key
    if wl.capacity_factor > 0:
        assert c["stats"]["dropped_slots"] > 0  # capacity binds


# ----------------------------------------------------------------------------
# the backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_expert_ffn_backward_against_autograd(act):
    """One expert's input, weight and bias gradients for an upstream g_out
    equal torch autograd's of <g_out, FFN(v)> in fp64, on rows and weights
    stored in bf16; the forward output comes back too."""
    g = torch.Generator().manual_seed(31)
    n, d, h = 9, 24, 40
    st = dict(v=torch.randn(n, d, generator=g), W1=torch.randn(h, d, generator=g) / d ** 0.5,
              W3=torch.randn(h, d, generator=g) / d ** 0.5, W2=torch.randn(d, h, generator=g) / h ** 0.5,
              b1=torch.randn(h, generator=g) * 0.3, b2=torch.randn(d, generator=g) * 0.3)
    st = {k_: v_.to(torch.bfloat16) for k_, v_ in st.items()}
    leaf = {k_: v_.double().requires_grad_(True) for k_, v_ in st.items()}
    go = torch.randn(n, d, generator=g, dtype=torch.float64)
    if act == "gelu":
        out = torch.nn.functional.gelu(leaf["v"] @ leaf["W1"].T + leaf["b1"]) @ leaf["W2"].T + leaf["b2"]
        got = cpp.expert_ffn_backward(st["v"], go.numpy(), "gelu", st["W1"], st["W2"], b1=st["b1"], b2=st["b2"])
        names = ("v", "W1", "W2", "b1", "b2")
    else:
        out = (torch.nn.functional.silu(leaf["v"] @ leaf["W1"].T) * (leaf["v"] @ leaf["W3"].T)) @ leaf["W2"].T
        got = cpp.expert_ffn_backward(st["v"], go.numpy(), "swiglu", st["W1"], st["W2"], W3=st["W3"])
        names = ("v", "W1", "W2", "W3")
    (out * go).sum().backward()
    np.testing.assert_allclose(got["out"], out.detach().numpy(), rtol=1e-12, atol=1e-12)
    for nm in names:
        key = "dv" if nm == "v" else "d" + nm
        ref = leaf[nm].grad.numpy()
        np.testing.assert_allclose(got[key], ref, rtol=0, atol=1e-12 * max(1.0, float(np.abs(ref).max())),
                                   err_msg=key)


@pytest.mark.parametrize("variant", ["cv", "std_max", "switch"])
def test_balance_term_grad_against_autograd(variant):
    """The balance term on the importance g = I/T and its per-slot weight
    gradient, against torch autograd in fp64 (an unrouted slot, -1, has
    none): cv lambda * std(g) / (mean(g) + 1e-8); std_max lambda * (std(g)
    + gamma * max(g)) with a unique largest g; switch lambda * sum f g with
    the usage f = counts / T held constant.  Equal importances give a zero
    CV term."""
    rng = np.random.default_rng(41)
    T, k, E, lam, gamma = 30, 2, 5, 0.01, 100.0
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[4] = -1
    w = rng.uniform(0.1, 0.9, size=(T, k))
    wt = torch.tensor(w, requires_grad=True)
    onehot = torch.zeros(T, k, E, dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            if idx[t, j] >= 0:
                onehot[t, j, idx[t, j]] = 1.0
    gI = (wt[:, :, None] * onehot).sum(dim=(0, 1)) / T
    if variant == "cv":
        B = lam * gI.std(unbiased=True) / (gI.mean() + 1e-8)
    elif variant == "std_max":
        assert int((gI == gI.max()).sum()) == 1
        B = lam * (gI.std(unbiased=True) + gamma * gI.max())
    else:
        f = onehot.sum(dim=(0, 1)) / T
        B = lam * (f * gI).sum()
    B.backward()
    val, dw = cpp.balance_term_grad(idx, w, E, T, lam, variant, gamma)
    assert abs(val - float(B.detach())) <= 1e-13 * max(1.0, abs(float(B.detach())))
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=0, atol=1e-13)
    assert (dw[4] == 0).all()
    if variant == "cv":
        val, dw = cpp.balance_term_grad(np.array([[0], [1]], dtype=np.int32), np.array([[0.5], [0.5]]), 2, 2, lam)
        assert val == 0.0 and np.all(np.abs(dw) <= 1e-6)


def test_balance_std_max_tie_goes_to_lower_index():
    """With two experts tied for the largest importance, the max's
    (sub)gradient goes to the lower expert index, as in the numpy oracle:
    slots of expert 1 carry lambda*gamma/T more than slots of expert 3."""
    T, lam, gamma = 4, 0.01, 100.0
    idx = np.array([[1, 3], [3, 1], [0, 2], [2, 0]], dtype=np.int32)
    w = np.array([[0.6, 0.4], [0.6, 0.4], [0.3, 0.2], [0.1, 0.2]])
    _, dw = cpp.balance_term_grad(idx, w, 4, T, lam, "std_max", gamma)
    # I = [0.5, 1.0, 0.3, 1.0]: experts 1 and 3 tie at the top, with the same std part
    assert abs((dw[0, 0] - dw[0, 1]) - lam * gamma / T) <= 1e-15
    _, dn = O.balance_term_grad(idx, w, 4, T, lam, "std_max", gamma)
    np.testing.assert_allclose(dw, dn, rtol=0, atol=1e-15)


BACKWARD_LAYERS = [
    # GeLU in fp32 with biases, no capacity limit
    (S.WORKLOADS["tiny_fp32"].replace(T=24, d=16, h=24, seed=43, training=True), "cv"),
    # SwiGLU in bf16 with the shared expert, Gumbel noise and a binding capacity
    (S.WORKLOADS["training"].replace(T=64, d=24, h=32, E=6, capacity_factor=0.7, seed=47), "cv"),
    # the other balance terms, with a lambda large enough to show
    (S.WORKLOADS["training"].replace(T=48, d=16, h=24, E=5, capacity_factor=0.8, lam=0.3, seed=61), "std_max"),
    (S.WORKLOADS["tiny_fp32"].replace(T=24, d=16, h=24, lam=0.3, seed=67, training=True), "switch"),
]


def _bwd_cfg(wl, balance="cv"):
    return dict(T=wl.T, d=wl.d, h=wl.h, E=wl.E, k=wl.k, act=wl.act,
                capacity_factor=float(np.float32(wl.capacity_factor)), min_capacity=wl.min_capacity,
                lam=float(np.float32(wl.lam)), has_shared=wl.has_shared, balance=balance, gamma=100.0)


@pytest.mark.parametrize("wl,balance", BACKWARD_LAYERS, ids=lambda p: p.name if hasattr(p, "name") else p)
def test_layer_backward_matches_numpy_oracle(wl, balance):
    """Every gradient, the logit gradient, y and the loss of the C++
    backward equal the numpy oracle's (itself pinned by finite differences)
    to 1e-11 of each tensor's largest entry, for each balance term; the
    forward's load statistic in that form to 1e-12."""
    t = S.make_inputs(wl, "cpu")
    cfg = _bwd_cfg(wl, balance)
    c = cpp.layer_backward(cfg, t, t["x"], t["dY"], t.get("expert_bias"), t.get("noise"))
    n = O.layer_backward(cfg, t, t["x"], t["dY"], t.get("expert_bias"), t.get("noise"))
    keys = [k_ for k_ in c if k_ not in ("loss", "balance_term")]
    assert set(keys) <= set(n), set(keys) - set(n)
    for key in keys:
        scale = max(1e-3, float(np.abs(n[key]).max()))
        np.testing.assert_allclose(c[key], n[key], rtol=0, atol=1e-11 * scale, err_msg=key)
    assert abs(c["loss"] - n["loss"]) <= 1e-11 * max(1.0, abs(n["loss"]))
    assert abs(c["balance_term"] - n["balance_term"]) <= 1e-14 * max(1.0, abs(n["balance_term"]))
    if wl.capacity_factor > 0:
        assert (n["route"]["pos"] < 0).any()  # a dropped slot takes part
    # the forward's load statistic in the same form
    cf = cpp.layer_forward(cfg, t, t["x"], t.get("expert_bias"), t.get("noise"))
    ref = n["route"]["stats"]["balance_stat"]
    assert abs(cf["stats"]["balance_stat"] - ref) <= 1e-12 * max(1.0, abs(ref)), balance


def test_layer_backward_finite_differences():
    """Central differences of the C++ oracle's own loss, on a GeLU layer
    stored in fp32 with a shared expert, match its gradients: entries of x,
    Wr, W1, b1, W2, b2 and the shared expert's weights.  The perturbation is 2^-9,
    exact in fp32 for these magnitudes.  An entry of x or Wr whose
    perturbation changes the routing (the loss is not differentiable
    there) is passed over for another; each tensor gets three checks."""
    wl = S.WORKLOADS["tiny_fp32"].replace(T=12, d=8, h=12, E=4, has_shared=True, capacity_factor=0.8, seed=53,
                                          training=True)
    t = S.make_inputs(wl, "cpu")
    cfg = _bwd_cfg(wl)
    base = cpp.layer_backward(cfg, t, t["x"], t["dY"], t.get("expert_bias"), t.get("noise"))
    fwd0 = cpp.layer_forward(cfg, t, t["x"], t.get("expert_bias"), t.get("noise"))
    assert (fwd0["pos"] < 0).any()  # the capacity drops a slot
    hstep = 2.0 ** -9
    rng = np.random.default_rng(59)
    checks = [("x", "dX"), ("Wr", "dWr"), ("W1", "dW1"), ("b1", "db1"), ("W2", "dW2"), ("b2", "db2"),
              ("Ws1", "dWs1"), ("Ws2", "dWs2")]
    for name, gname in checks:
        done = 0
        for _ in range(40):
            flat = int(rng.integers(t[name].numel()))
            vals, same = [], True
            for sgn in (1, -1):
                tt = dict(t)
                a = t[name].clone().reshape(-1)
                a[flat] += sgn * hstep
                tt[name] = a.reshape(t[name].shape)
                f = cpp.layer_forward(cfg, tt, tt["x"], tt.get("expert_bias"), tt.get("noise"))
                same = same and np.array_equal(f["pos"], fwd0["pos"]) and np.array_equal(f["idx"], fwd0["idx"])
                r = cpp.layer_backward(cfg, tt, tt["x"], tt["dY"], tt.get("expert_bias"), tt.get("noise"))
                vals.append(r["loss"])
            if not same:
                assert name in ("x", "Wr")  # only the router's inputs move the routing
                continue
            fd = (vals[0] - vals[1]) / (2 * hstep)
            an = float(base[gname].reshape(-1)[flat])
            assert abs(fd - an) <= 1e-5 * max(1.0, abs(an)), (name, flat, fd, an)
            done += 1
            if done == 3:
                break
        assert done == 3, name


# ----------------------------------------------------------------------------
# routing variants: raw probabilities, token-major priority, a LayerNorm in
# front of the router
# ----------------------------------------------------------------------------

def test_layer_norm_against_torch():
    """The router's LayerNorm (no affine, eps 1e-5, biased variance) and its
    input gradient against torch's layer_norm and autograd in fp64, on rows
    with their own offsets and scales stored in bf16."""
    g = torch.Generator().manual_seed(71)
    x = (torch.randn(7, 33, generator=g) * torch.rand(7, 1, generator=g) * 3 + torch.randn(7, 1, generator=g))
    x = x.to(torch.bfloat16)
    xd = x.double().requires_grad_(True)
    ref = torch.nn.functional.layer_norm(xd, (33,), eps=1e-5)
    np.testing.assert_allclose(cpp.layer_norm(x), ref.detach().numpy(), rtol=0, atol=1e-13)
    gout = torch.randn(7, 33, generator=g, dtype=torch.float64)
    (ref * gout).sum().backward()
    np.testing.assert_allclose(cpp.layer_norm_backward(x, gout.numpy()), xd.grad.numpy(), rtol=0, atol=1e-12)


def test_top_k_raw_probabilities():
    """With raw probabilities the weights are the selected entries of the
    softmax over all E experts (torch.softmax), the same experts as the
    default selection, and sum to at most 1."""
    rng = np.random.default_rng(73)
    l = rng.normal(size=(40, 9)) * 2
    idx0, w0, _ = cpp.top_k(l, 3)
    idx, w, nf = cpp.top_k_probs(l, 3, raw=True)
    np.testing.assert_array_equal(idx, idx0)
    p = torch.softmax(torch.tensor(l), dim=1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(p, idx.astype(np.int64), axis=1), rtol=0, atol=1e-15)
    assert nf == 0 and (w.sum(axis=1) <= 1 + 1e-15).all() and (w.sum(axis=1) < w0.sum(axis=1)).all()


def test_token_major_capacity_queue():
    """Token-major priority: a direct queue over (t, j) in token order; each
    expert keeps its first C slots in that order."""
    rng = np.random.default_rng(79)
    T, k, E, C = 50, 3, 6, 17
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[5] = -1
    rank, fill = cpp.assign_capacity_token_major(idx, E, C)
    seen = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            want = -1 if e < 0 or seen[e] >= C else seen[e]
            assert rank[t, j] == want, (t, j)
            if want >= 0:
                seen[e] += 1
    np.testing.assert_array_equal(fill, seen)
    assert (fill == C).any()


def test_backup_experts_and_reroute_queue():
    """Backups are each token's experts ranked k .. 2k-1 by (logit
    descending, index ascending), against a sort; the second capacity pass
    against a direct queue in either priority: the r-th dropped slot of a
    token tries its r-th backup once, kept if the expert has room after
    its first-pass rows and the slots rerouted to it before."""
    rng = np.random.default_rng(101)
    T, k, E = 60, 2, 7
    l = np.round(rng.normal(size=(T, E)), 1)  # rounding makes ties
    l[3, 2] = np.inf
    b = cpp.backup_experts(l, k)
    for t in range(T):
        if not np.all(np.isfinite(l[t])):
            assert (b[t] == -1).all()
            continue
        order = sorted(range(E), key=lambda e: (-l[t, e], e))
        np.testing.assert_array_equal(b[t], order[k:2 * k])
    idx, _, _ = cpp.top_k(l, k)
    C = 15
    for tm in (False, True):
        rank, fill = cpp.assign_capacity_token_major(idx, E, C) if tm else cpp.assign_capacity(idx, E, C)
        served, rank2, fill2 = cpp.reroute_overflow(idx, b, rank, fill, C, tm)
        nth = -np.ones((T, k), dtype=np.int64)
        for t in range(T):
            r = 0
            for j in range(k):
                if idx[t, j] >= 0 and rank[t, j] < 0:
                    nth[t, j] = r
                    r += 1
        used = fill.astype(np.int64).copy()
        extra = np.zeros(E, dtype=np.int64)
        order = [(t, j) for t in range(T) for j in range(k)] if tm else [(t, j) for j in range(k) for t in range(T)]
        for t, j in order:
            want_served = idx[t, j] if rank[t, j] >= 0 else -1
            want_rank2 = -1
            if nth[t, j] >= 0 and b[t, nth[t, j]] >= 0 and used[b[t, nth[t, j]]] < C:
                e = b[t, nth[t, j]]
                want_served, want_rank2 = e, extra[e]
                extra[e] += 1
                used[e] += 1
            assert served[t, j] == want_served and rank2[t, j] == want_rank2, (tm, t, j)
        np.testing.assert_array_equal(fill2, extra)
        assert extra.sum() > 0


VARIANT_ROUTES = [dict(raw_probs=True), dict(token_major=True), dict(layernorm=True),
                  dict(raw_probs=True, token_major=True, layernorm=True), dict(reroute=True),
                  dict(reroute=True, token_major=True, raw_probs=True)]


@pytest.mark.parametrize("route", VARIANT_ROUTES, ids=lambda r: "+".join(r))
def test_routing_variants_match_numpy_oracle(route):
    """Forward and backward of a SwiGLU bf16 layer with the shared expert, a
    binding capacity and Gumbel noise, under each routing variant (and
    rerouting, which moves some dropped slots to backups): routing and the
    slot counts bit for bit, every output and gradient to 1e-11 of the
    numpy oracle's."""
    wl = S.WORKLOADS["training"].replace(T=64, d=24, h=32, E=6, capacity_factor=0.7, seed=83)
    t = S.make_inputs(wl, "cpu")
    cfg = dict(_bwd_cfg(wl), **route)
    c = cpp.layer_forward(dict(cfg), t, t["x"], t.get("expert_bias"), t.get("noise"))
    n = O.layer_forward(cfg, t, t["x"], t.get("expert_bias"), t.get("noise"))
    for key in ("idx", "counts", "kept", "offsets", "pos"):
        np.testing.assert_array_equal(c[key], n[key], err_msg=key)
    np.testing.assert_allclose(c["w"], n["w"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(c["y"], n["y"], rtol=0, atol=1e-12 * max(1.0, float(np.abs(n["y"]).max())))
    assert (c["pos"] < 0).any()
    for key in ("kept_slots", "dropped_slots", "rerouted_slots"):
        assert c["stats"][key] == n["stats"][key], key
    assert (c["stats"]["rerouted_slots"] > 0) == bool(route.get("reroute"))
    cb = cpp.layer_backward(cfg, t, t["x"], t["dY"], t.get("expert_bias"), t.get("noise"))
    nb = O.layer_backward(cfg, t, t["x"], t["dY"], t.get("expert_bias"), t.get("noise"))
    for key in [k_ for k_ in cb if k_ not in ("loss", "balance_term")]:
        scale = max(1e-3, float(np.abs(nb[key]).max()))
        np.testing.assert_allclose(cb[key], nb[key], rtol=0, atol=1e-11 * scale, err_msg=key)
    assert abs(cb["loss"] - nb["loss"]) <= 1e-11 * max(1.0, abs(nb["loss"]))


def test_routing_variants_finite_differences():
    """Central differences of the C++ oracle's loss with raw probabilities
    and a LayerNorm in front of the router (fp32 storage, 2^-9 steps, the
    routing checked unchanged) match its x and Wr gradients."""
    wl = S.WORKLOADS["tiny_fp32"].replace(T=12, d=8, h=12, E=4, has_shared=True, capacity_factor=0.8, seed=89,
                                          training=True)
    t = S.make_inputs(wl, "cpu")
    cfg = dict(_bwd_cfg(wl), raw_probs=True, layernorm=True)
    base = cpp.layer_backward(cfg, t, t["x"], t["dY"], t.get("expert_bias"), t.get("noise"))
    fwd0 = cpp.layer_forward(cfg, t, t["x"], t.get("expert_bias"), t.get("noise"))
    hstep = 2.0 ** -9
    rng = np.random.default_rng(97)
    for name, gname in (("x", "dX"), ("Wr", "dWr")):
        done = 0
        for _ in range(60):
            flat = int(rng.integers(t[name].numel()))
            vals, same = [], True
            for sgn in (1, -1):
                tt = dict(t)
                a = t[name].clone().reshape(-1)
                a[flat] += sgn * hstep
                tt[name] = a.reshape(t[name].shape)
                f = cpp.layer_forward(cfg, tt, tt["x"], tt.get("expert_bias"), tt.get("noise"))
                same = same and np.array_equal(f["pos"], fwd0["pos"]) and np.array_equal(f["idx"], fwd0["idx"])
                vals.append(cpp.layer_backward(cfg, tt, tt["x"], tt["dY"], tt.get("expert_bias"),
                                               tt.get("noise"))["loss"])
            if not same:
                continue
            fd = (vals[0] - vals[1]) / (2 * hstep)
            an = float(base[gname].reshape(-1)[flat])
            assert abs(fd - an) <= 1e-5 * max(1.0, abs(an)), (name, flat, fd, an)
            done += 1
            if done == 4:
                break
        assert done == 4, name

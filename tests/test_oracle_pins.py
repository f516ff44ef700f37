"""Pins of the fp64 oracle to facts other than itself: the pages' printed
examples (tests/golden), closed forms, invariants, brute force on tiny inputs,
library routines for special cases, and finite differences for the backward.
Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand) fails at least one of them."""

import itertools
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import moe_oracle as O


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# printed examples
# ---------------------------------------------------------------------------


def test_combine_worked_example():
    g = read_golden("combine_worked_example.txt")
    out = np.array([[g["expert_out_0"], g["expert_out_1"]]])  # [T=1, k=2, d=3]
    w = np.array([g["weights"]])
    y = O.combine(out, w, np.ones((1, 2), bool))
    np.testing.assert_allclose(y[0], g["expected"], atol=1e-15, rtol=0)
    # first cell spelled out on the page: 0.75*0.8 + 0.25*0.4 = 0.7
    assert abs(y[0, 0] - 0.7) < 1e-15


def test_combine_dropped_slot_adds_zero_and_shared_adds_one():
    g = read_golden("combine_worked_example.txt")
    out = np.array([[g["expert_out_0"], g["expert_out_1"]]])
    w = np.array([g["weights"]])
    y = O.combine(out, w, np.array([[True, False]]))
    np.testing.assert_allclose(y[0], 0.75 * np.array(g["expert_out_0"]), atol=1e-15)
    sh = np.array([[1.0, -2.0, 3.0]])
    y2 = O.combine(out, w, np.ones((1, 2), bool), sh)
    np.testing.assert_allclose(y2[0], np.array(g["expected"]) + sh[0], atol=1e-15)


def test_top2_gate_sample():
    g = read_golden("top2_gate_sample.txt")
    p = np.array(g["probs"])
    l = np.log(p)[None, :]
    idx, w, finite = O.top_k_route(l, 2)
    assert finite.all()
    assert idx[0].tolist() == [int(v) for v in g["top2"]]
    sel = np.array(g["top2_probs"])
    np.testing.assert_allclose(w[0], sel / sel.sum(), rtol=1e-14)
    np.testing.assert_allclose(w[0], [0.85 / 0.93, 0.08 / 0.93], rtol=1e-14)
    # the full softmax of ln p gives p back (P1 3.1's p_i)
    np.testing.assert_allclose(O.softmax(l)[0], p / p.sum(), rtol=1e-14)


def test_capacity_examples():
    g = read_golden("capacity_examples.txt")
    for T, k, E, cf, C in g["_rows"]:
        assert O.expert_capacity(int(T), int(k), int(E), cf) == int(C)
    # workloads: 4096*2/16*1.0 = 512, 16384*2/64*1.25 = 640, 32768*2/16*1.25 = 5120
    assert O.expert_capacity(4096, 2, 16, 1.0) == 512
    assert O.expert_capacity(16384, 2, 64, 1.25) == 640
    assert O.expert_capacity(32768, 2, 16, 1.25) == 5120
    assert O.expert_capacity(64, 2, 4, 0.0) == 64          # no limit
    assert O.expert_capacity(10, 2, 16, 1.0) == 2          # ceil(1.25)
    assert O.expert_capacity(10, 2, 16, 1.0, min_capacity=4) == 4


def test_call_counting():
    g = read_golden("call_counting.txt")
    T, E = int(g["tokens"][0]), int(g["experts"][0])
    # every token through every expert
    assert T * E == g["calls_all"][0]
    # top-2, balanced: token t prefers experts (t mod 4) and (t+1 mod 4) --
    # a construction where each expert is first choice 25 times and second
    # choice 25 times
    l = np.zeros((T, E))
    for t in range(T):
        l[t, t % E] = 2.0
        l[t, (t + 1) % E] = 1.0
    idx, w, _ = O.top_k_route(l, 2)
    counts = O.usage_counts(idx, E)
    assert counts.sum() == g["calls_top2"][0]
    assert counts.tolist() == [g["per_expert_balanced"][0]] * E
    assert O.balance_stat(counts, T, 0.01) == 0.0
    # any routing: sum of counts is T*k
    rl = _rng(3).normal(size=(T, E))
    idx2, _, _ = O.top_k_route(rl, 2)
    assert O.usage_counts(idx2, E).sum() == T * 2


def test_parameter_accounting():
    """A scaled layer: 16 routed SwiGLU experts of 60 parameters each (d=2,
    h=10: 3*2*10) -> routed total 960 = 160 units of 6; shared expert of 240
    parameters (d=2, h=40) = 40 units.  The oracle must touch 2*60 + 240 =
    360 = 60 units per token, 30% of 1200 = 200 units."""
    g = read_golden("parameter_accounting.txt")
    assert g["routed_total"][0] * g["k"][0] / g["experts"][0] == g["routed_active"][0]
    assert g["common"][0] + g["routed_active"][0] == g["active"][0]
    assert abs(g["active"][0] / g["total"][0] - g["active_fraction"][0]) < 1e-12
    rng = _rng(5)
    T, d, h, hs, E = 8, 2, 10, 40, 16
    unit = 6
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)),
             W3=rng.normal(size=(E, h, d)), W2=rng.normal(size=(E, d, h)),
             Ws1=rng.normal(size=(hs, d)), Ws3=rng.normal(size=(hs, d)),
             Ws2=rng.normal(size=(d, hs)))
    cfg = dict(T=T, d=d, h=h, E=E, k=2, act="swiglu", capacity_factor=0.0, has_shared=True)
    x = rng.normal(size=(T, d))
    r = O.layer_forward(cfg, w, x)
    routed_total = sum(w[n].size for n in ("W1", "W3", "W2"))
    common = sum(w[n].size for n in ("Ws1", "Ws3", "Ws2"))
    assert routed_total == g["routed_total"][0] * unit
    assert common == g["common"][0] * unit
    assert (r["params_touched"] == g["active"][0] * unit).all()
    assert np.allclose(r["params_touched"] / (routed_total + common), g["active_fraction"][0])


def test_pair_count_and_bruteforce_top2():
    g = read_golden("pair_count.txt")
    E = int(g["experts"][0])
    pairs = list(itertools.combinations(range(E), 2))
    assert len(pairs) == g["pairs"][0]
    rng = _rng(7)
    l = rng.normal(size=(40, E))
    l[0, 5] = l[0, 9] = 10.0  # an exact tie at the top: lower index first
    idx, w, _ = O.top_k_route(l, 2)
    p = O.softmax(l)
    for t in range(l.shape[0]):
        # the pair maximising p_i + p_j; among equal sums the lexicographically
        # smallest pair
        best = max(pairs, key=lambda ij: (p[t, ij[0]] + p[t, ij[1]], -ij[0], -ij[1]))
        assert sorted(idx[t].tolist()) == list(best)
        # order within the pair: larger logit first, equal -> lower index first
        a, b = idx[t]
        assert (l[t, a] > l[t, b]) or (l[t, a] == l[t, b] and a < b)
    assert idx[0].tolist() == [5, 9]


def test_topk_against_sort_for_larger_k():
    rng = _rng(11)
    E = 32
    l = np.round(rng.normal(size=(50, E)), 1)  # many exact ties
    for k in (1, 3, 6, 8):
        idx, w, _ = O.top_k_route(l, k)
        for t in range(l.shape[0]):
            ref = sorted(range(E), key=lambda e: (-l[t, e], e))[:k]
            assert idx[t].tolist() == ref
            np.testing.assert_allclose(w[t].sum(), 1.0, atol=1e-15)
            ex = np.exp(l[t, ref])
            np.testing.assert_allclose(w[t], ex / ex.sum(), rtol=1e-13)


def test_weights_sum_to_one_and_tie():
    l = np.zeros((3, 8))
    idx, w, _ = O.top_k_route(l, 2)
    assert (idx == np.array([[0, 1]] * 3)).all()
    np.testing.assert_array_equal(w, 0.5)
    rng = _rng(2)
    l = rng.normal(size=(100, 16)) * 3
    idx, w, _ = O.top_k_route(l, 2)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-15)
    # w = p_i / (p_i + p_j) with the full softmax p ([P1] 3.3)
    p = O.softmax(l)
    pi = np.take_along_axis(p, idx, 1)
    np.testing.assert_allclose(w, pi / pi.sum(1, keepdims=True), rtol=1e-12)


def test_nonfinite_logit_routes_nowhere():
    l = np.array([[1.0, np.nan, 0.0, 2.0], [1.0, 0.5, 0.0, 2.0], [np.inf, 0, 0, 0]])
    idx, w, finite = O.top_k_route(l, 2)
    assert finite.tolist() == [False, True, False]
    assert idx[0].tolist() == [-1, -1] and idx[2].tolist() == [-1, -1]
    assert idx[1].tolist() == [3, 0]
    assert (w[0] == 0).all()


def test_balance_stat_closed_forms():
    T, E = 10, 4
    counts = np.array([T, T, 0, 0])
    # f = (1,1,0,0): mean 1/2, std_{n-1} = sqrt(1/3); ratio 2/sqrt(3) up to
    # the 1e-8 guard on the mean
    assert abs(O.balance_stat(counts, T, 0.01) - 0.01 * math.sqrt(1 / 3) / (0.5 + 1e-8)) < 1e-15
    assert abs(O.balance_stat(counts, T, 0.01) - 0.01 * 2 / math.sqrt(3)) < 1e-9
    assert O.balance_stat(np.array([5, 5, 5, 5]), T, 0.01) == 0.0
    # torch.std (n-1 default, as in [P1] 4.2's code) as an independent routine
    c = np.array([3, 9, 1, 7, 0, 12])
    f = torch.tensor(c / 20.0, dtype=torch.float64)
    ref = 0.01 * (torch.std(f) / (torch.mean(f) + 1e-8)).item()
    assert abs(O.balance_stat(c, 20, 0.01) - ref) < 1e-15


# ---------------------------------------------------------------------------
# capacity and dispatch
# ---------------------------------------------------------------------------


def _dispatch_by_sorting(idx, E, C):
    """Independent formulation: for each expert the kept slots are its first
    C slots in (choice j, token t) order; positions follow expert order."""
    T, k = idx.shape
    slots = [(j, t) for j in range(k) for t in range(T)]
    pos = -np.ones((T, k), dtype=np.int64)
    base = 0
    for e in range(E):
        mine = [(j, t) for (j, t) in slots if idx[t, j] == e][:C]
        for r, (j, t) in enumerate(mine):
            pos[t, j] = base + r
        base += len(mine)
    return pos


@pytest.mark.parametrize("T,E,k,cf", [(37, 5, 2, 1.0), (64, 4, 2, 0.5), (50, 8, 3, 1.25), (20, 3, 1, 0.4)])
def test_dispatch_against_sorting_and_invariants(T, E, k, cf):
    rng = _rng(T * 31 + E)
    # skewed logits so that capacity binds
    l = rng.normal(size=(T, E)) + np.linspace(2, 0, E)[None, :]
    idx, w, _ = O.top_k_route(l, k)
    C = O.expert_capacity(T, k, E, cf)
    rank, fill = O.assign_capacity(idx, E, C)
    offsets, pos = O.dispatch_positions(idx, rank, fill)
    np.testing.assert_array_equal(pos, _dispatch_by_sorting(idx, E, C))
    counts = O.usage_counts(idx, E)
    np.testing.assert_array_equal(fill, np.minimum(counts, C))
    kept_pos = np.sort(pos[pos >= 0])
    np.testing.assert_array_equal(kept_pos, np.arange(fill.sum()))  # each row served once
    assert offsets[0] == 0 and offsets[-1] == fill.sum()
    assert fill.sum() + (pos < 0).sum() == T * k
    # a token's first choice is never dropped in favour of another's second
    for e in range(E):
        firsts_dropped = np.any((idx[:, 0] == e) & (pos[:, 0] < 0))
        seconds_kept = np.any((idx[:, 1:] == e) & (pos[:, 1:] >= 0)) if k > 1 else False
        assert not (firsts_dropped and seconds_kept)


def test_route_and_dispatch_stats():
    rng = _rng(9)
    T, E, d = 64, 4, 8
    x = rng.normal(size=(T, d))
    Wr = rng.normal(size=(E, d))
    Wr[0] *= 3  # skew
    cfg = dict(T=T, d=d, E=E, k=2, capacity_factor=1.0, lam=0.01)
    r = O.route_and_dispatch(cfg, x, Wr)
    s = r["stats"]
    assert s["capacity"] == 32
    assert s["routed_slots"] == T * 2
    assert s["kept_slots"] == r["kept"].sum()
    assert s["dropped_slots"] == T * 2 - s["kept_slots"]
    assert abs(s["drop_rate"] - s["dropped_slots"] / (T * 2)) < 1e-15


# ---------------------------------------------------------------------------
# experts
# ---------------------------------------------------------------------------


def test_single_expert_layer_is_dense_ffn_gelu():
    """E=1, k=1, no capacity limit: the layer is a dense GeLU FFN; checked
    against torch's float64 Linear/GELU (exact erf form) as a library routine."""
    rng = _rng(13)
    T, d, h = 16, 6, 10
    w = dict(Wr=rng.normal(size=(1, d)), W1=rng.normal(size=(1, h, d)),
             W2=rng.normal(size=(1, d, h)), b1=rng.normal(size=(1, h)), b2=rng.normal(size=(1, d)))
    x = rng.normal(size=(T, d))
    cfg = dict(T=T, d=d, h=h, E=1, k=1, act="gelu", capacity_factor=0.0)
    r = O.layer_forward(cfg, w, x)
    xt = torch.tensor(x)
    ref = torch.nn.functional.linear(
        torch.nn.functional.gelu(torch.nn.functional.linear(xt, torch.tensor(w["W1"][0]), torch.tensor(w["b1"][0]))),
        torch.tensor(w["W2"][0]), torch.tensor(w["b2"][0]))
    np.testing.assert_allclose(r["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_expert_layer_is_dense_ffn_swiglu():
    rng = _rng(17)
    T, d, h = 16, 6, 10
    w = dict(Wr=rng.normal(size=(1, d)), W1=rng.normal(size=(1, h, d)),
             W3=rng.normal(size=(1, h, d)), W2=rng.normal(size=(1, d, h)))
    x = rng.normal(size=(T, d))
    cfg = dict(T=T, d=d, h=h, E=1, k=1, act="swiglu", capacity_factor=0.0)
    r = O.layer_forward(cfg, w, x)
    F = torch.nn.functional
    xt = torch.tensor(x)
    ref = F.linear(F.silu(F.linear(xt, torch.tensor(w["W1"][0]))) * F.linear(xt, torch.tensor(w["W3"][0])),
                   torch.tensor(w["W2"][0]))
    np.testing.assert_allclose(r["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_activation_special_values():
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([0.0]))[0] == 0.0
    z = np.linspace(-6, 6, 101)
    F = torch.nn.functional
    np.testing.assert_allclose(O.gelu(z), F.gelu(torch.tensor(z)).numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.silu(z), F.silu(torch.tensor(z)).numpy(), rtol=1e-14, atol=1e-15)
    # derivatives against central differences
    e = 1e-6
    np.testing.assert_allclose(O.gelu_grad(z), (O.gelu(z + e) - O.gelu(z - e)) / (2 * e), atol=1e-8)
    np.testing.assert_allclose(O.silu_grad(z), (O.silu(z + e) - O.silu(z - e)) / (2 * e), atol=1e-8)


def test_zero_up_projection_gives_zero_output():
    rng = _rng(19)
    T, d, h, E = 12, 4, 6, 3
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)),
             W3=np.zeros((E, h, d)), W2=rng.normal(size=(E, d, h)))
    cfg = dict(T=T, d=d, h=h, E=E, k=2, act="swiglu", capacity_factor=0.0)
    r = O.layer_forward(cfg, w, rng.normal(size=(T, d)))
    assert (r["y"] == 0).all()


def test_layer_equals_per_token_definition():
    """Each token: y = sum over its kept slots of w * FFN_e(x) -- computed
    token by token, expert by expert, with no batching."""
    rng = _rng(23)
    T, d, h, E = 24, 5, 7, 4
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)),
             W3=rng.normal(size=(E, h, d)), W2=rng.normal(size=(E, d, h)),
             Ws1=rng.normal(size=(h, d)), Ws3=rng.normal(size=(h, d)), Ws2=rng.normal(size=(d, h)))
    x = rng.normal(size=(T, d))
    cfg = dict(T=T, d=d, h=h, E=E, k=2, act="swiglu", capacity_factor=0.5, has_shared=True)
    r = O.layer_forward(cfg, w, x)

    def ffn(v, A, B, C):
        g = A @ v
        u = B @ v
        return C @ (g / (1 + np.exp(-g)) * u)

    for t in range(T):
        ref = ffn(x[t], w["Ws1"], w["Ws3"], w["Ws2"])
        for j in range(2):
            if r["pos"][t, j] >= 0:
                e = r["idx"][t, j]
                ref = ref + r["w"][t, j] * ffn(x[t], w["W1"][e], w["W3"][e], w["W2"][e])
        np.testing.assert_allclose(r["y"][t], ref, rtol=1e-12, atol=1e-12)


def test_gumbel_noise_special_cases():
    rng = _rng(29)
    T, d, E = 30, 6, 8
    x = rng.normal(size=(T, d))
    Wr = rng.normal(size=(E, d))
    cfg = dict(T=T, d=d, E=E, k=2, capacity_factor=0.0)
    clean = O.route_and_dispatch(cfg, x, Wr)
    zero = O.route_and_dispatch(cfg, x, Wr, noise=np.zeros((T, E)))
    np.testing.assert_array_equal(clean["idx"], zero["idx"])
    np.testing.assert_array_equal(clean["w"], zero["w"])
    big = np.zeros((T, E))
    big[:, 6] = 1e3
    forced = O.route_and_dispatch(cfg, x, Wr, noise=big)
    assert (forced["idx"][:, 0] == 6).all()
    # weights use the noisy logits: the forced expert takes all the weight
    np.testing.assert_allclose(forced["w"][:, 0], 1.0)


def test_bf16_decode_is_exact():
    v = torch.tensor([1.0, -2.5, 3.140625, 1e-3, 65280.0], dtype=torch.bfloat16)
    np.testing.assert_array_equal(O.decode(v), v.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# backward: central finite differences of L in fp64
# ---------------------------------------------------------------------------


def _loss(cfg, w, x, dY, bias=None, noise=None):
    r = O.layer_forward(cfg, w, x, bias, noise)
    val, _ = O.importance_cv_grad(r["idx"], r["w"], cfg["E"], cfg["T"], cfg["lam"])
    return float((dY * r["y"]).sum()) + val, r


@pytest.mark.parametrize("act,shared,cf,lam", [("swiglu", True, 0.75, 0.01), ("gelu", False, 0.0, 0.01),
                                             ("swiglu", False, 0.0, 0.0)])
def test_backward_finite_differences(act, shared, cf, lam):
    rng = _rng(31 + int(shared) + int(cf * 4))
    T, d, h, E = 10, 4, 5, 4
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) * 0.7,
             W2=rng.normal(size=(E, d, h)) * 0.7)
    if act == "swiglu":
        w["W3"] = rng.normal(size=(E, h, d)) * 0.7
    else:
        w["b1"] = rng.normal(size=(E, h)) * 0.3
        w["b2"] = rng.normal(size=(E, d)) * 0.3
    if shared:
        w.update(Ws1=rng.normal(size=(h, d)), Ws3=rng.normal(size=(h, d)), Ws2=rng.normal(size=(d, h)))
    x = rng.normal(size=(T, d))
    dY = rng.normal(size=(T, d))
    noise = rng.gumbel(size=(T, E))
    cfg = dict(T=T, d=d, h=h, E=E, k=2, act=act, capacity_factor=cf, has_shared=shared, lam=lam)
    g = O.layer_backward(cfg, w, x, dY, noise=noise)
    L0, r0 = _loss(cfg, w, x, dY, noise=noise)
    assert abs(g["loss"] - L0) < 1e-10
    if cf > 0:
        assert (r0["pos"] < 0).any(), "the case must exercise dropped slots"
    eps = 1e-6
    targets = [("x", None)] + [(n, n) for n in w]
    for name, key in targets:
        base = x if key is None else w[key]
        grad = g["dX"] if key is None else g[{"Wr": "dWr", "W1": "dW1", "W2": "dW2", "W3": "dW3",
                                              "b1": "db1", "b2": "db2", "Ws1": "dWs1", "Ws2": "dWs2",
                                              "Ws3": "dWs3"}[key]]
        flat = base.reshape(-1)
        picks = rng.choice(flat.size, size=min(flat.size, 12), replace=False)
        for i in picks:
            old = flat[i]
            flat[i] = old + eps
            Lp, rp = _loss(cfg, w, x, dY, noise=noise)
            flat[i] = old - eps
            Lm, rm = _loss(cfg, w, x, dY, noise=noise)
            flat[i] = old
            assert (rp["idx"] == r0["idx"]).all() and (rm["idx"] == r0["idx"]).all()
            fd = (Lp - Lm) / (2 * eps)
            an = grad.reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, i, fd, an)


def test_backward_balance_term_isolated():
    """lambda=0 vs lambda=0.01: only the router and input gradients change,
    by the gradient of the importance term alone."""
    rng = _rng(37)
    T, d, h, E = 12, 4, 5, 4
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)),
             W3=rng.normal(size=(E, h, d)), W2=rng.normal(size=(E, d, h)))
    x = rng.normal(size=(T, d))
    dY = rng.normal(size=(T, d))
    base = dict(T=T, d=d, h=h, E=E, k=2, act="swiglu", capacity_factor=0.0)
    g0 = O.layer_backward(dict(base, lam=0.0), w, x, dY)
    g1 = O.layer_backward(dict(base, lam=0.01), w, x, dY)
    for n in ("dW1", "dW2", "dW3"):
        np.testing.assert_array_equal(g0[n], g1[n])
    assert np.abs(g1["dWr"] - g0["dWr"]).max() > 0
    # a dZero upstream leaves only the balance term
    gz = O.layer_backward(dict(base, lam=0.01), w, x, np.zeros_like(dY))
    np.testing.assert_allclose(gz["dWr"], g1["dWr"] - g0["dWr"], atol=1e-12)


SAMPLED_VARIANTS = [("swiglu", True, {}), ("gelu", False, {}), ("swiglu", True, {"reroute": True}),
                    ("swiglu", False, {"raw_probs": True}), ("swiglu", True, {"layernorm": True}),
                    ("gelu", True, {"balance": "std_max"}), ("swiglu", False, {"balance": "switch", "raw_probs": True})]


@pytest.mark.parametrize("act,shared,route", SAMPLED_VARIANTS)
def test_sampled_backward_entries_match_full_backward(act, shared, route):
    """The sampled-entry functions used at full size (expert_grad_slices,
    token_input_grads, router_grad_rows) agree with the
    finite-difference-pinned layer_backward on a tiny batch, under the
    routing and balance variants: rerouted slots are served by their backup,
    raw softmax weights give every logit a gradient, the LayerNorm router
    carries its backward."""
    rng = _rng(71)
    T, d, h, E, k = 30, 6, 10, 4, 2
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) / 2, W2=rng.normal(size=(E, d, h)) / 3)
    if act == "swiglu":
        w["W3"] = rng.normal(size=(E, h, d)) / 2
    else:
        w["b1"] = rng.normal(size=(E, h)) * 0.1
        w["b2"] = rng.normal(size=(E, d)) * 0.1
    if shared:
        w.update(Ws1=rng.normal(size=(h, d)) / 2, Ws3=rng.normal(size=(h, d)) / 2, Ws2=rng.normal(size=(d, h)) / 3)
        if act == "gelu":
            w.update(bs1=rng.normal(size=h) * 0.1, bs2=rng.normal(size=d) * 0.1)
    cfg = dict(T=T, d=d, h=h, E=E, k=k, act=act, capacity_factor=0.75, has_shared=shared, lam=0.05, **route)
    x = rng.normal(size=(T, d)) * 1.5 + 0.3
    dY = rng.normal(size=(T, d))
    bias = np.array([1.0, 0.5, 0.0, -0.5])
    full = O.layer_backward(cfg, w, x, dY, bias)
    r = full["route"]
    assert (r["pos"] < 0).any() or route.get("reroute")
    if route.get("reroute"):
        assert ((r["served"] >= 0) & (r["served"] != r["idx"])).any()
    for e in range(E):
        cols = [1, 4, 7]
        sl = O.expert_grad_slices(cfg, w, x, dY, r, e, cols)
        np.testing.assert_allclose(sl["dW1"], full["dW1"][e][cols], atol=1e-12)
        np.testing.assert_allclose(sl["dW2"], full["dW2"][e][:, cols], atol=1e-12)
        if act == "swiglu":
            np.testing.assert_allclose(sl["dW3"], full["dW3"][e][cols], atol=1e-12)
        else:
            np.testing.assert_allclose(sl["db1"], full["db1"][e][cols], atol=1e-12)
    toks = [0, 3, 11, 29]
    np.testing.assert_allclose(O.token_input_grads(cfg, w, x, dY, r, toks), full["dX"][toks], atol=1e-12)
    if route.get("raw_probs"):
        with pytest.raises(ValueError):
            O.router_grad_rows(cfg, w, x, dY, r, [1])
    else:
        for ex in ([1], [0, 3], [2, 1]):
            np.testing.assert_allclose(O.router_grad_rows(cfg, w, x, dY, r, ex), full["dWr"][ex], atol=1e-12)


# ---------------------------------------------------------------------------
# routing variants
# ---------------------------------------------------------------------------


def test_raw_probability_weights_on_gate_sample():
    """[P4] 5.1 prints the top-2 probabilities (0.85, 0.08) as the weights it
    uses; raw_probs returns exactly those, not renormalised."""
    g = read_golden("top2_gate_sample.txt")
    p = np.array(g["probs"])
    idx, w, _ = O.top_k_route(np.log(p)[None, :], 2, raw_probs=True)
    assert idx[0].tolist() == [1, 2]
    np.testing.assert_allclose(w[0], g["top2_probs"], rtol=1e-14)
    # raw weights are the softmax entries: they sum to p1 + p2 < 1
    rl = _rng(31).normal(size=(50, 9))
    idx, w, _ = O.top_k_route(rl, 3, raw_probs=True)
    sm = O.softmax(rl)
    np.testing.assert_allclose(w, np.take_along_axis(sm, idx, axis=1), rtol=1e-13)


def test_router_entropy_closed_forms_and_library():
    from scipy.stats import entropy
    E = 16
    assert abs(O.router_entropy(np.zeros((5, E))) - math.log(E)) < 1e-14
    one_hot = np.full((3, E), -1e4)
    one_hot[:, 2] = 0.0
    assert O.router_entropy(one_hot) < 1e-12
    l = _rng(33).normal(size=(40, E)) * 2
    ref = np.mean([entropy(O.softmax(l[t:t + 1])[0]) for t in range(40)])
    assert abs(O.router_entropy(l) - ref) < 1e-13
    # tokens with a non-finite logit are left out
    l2 = l.copy()
    l2[3, 0] = np.nan
    ref2 = np.mean([entropy(O.softmax(l[t:t + 1])[0]) for t in range(40) if t != 3])
    assert abs(O.router_entropy(l2) - ref2) < 1e-13


def _dispatch_token_major_by_sorting(idx, E, C):
    """Independent formulation: each expert keeps its first C slots in
    (token t, choice j) order."""
    T, k = idx.shape
    pos = -np.ones((T, k), dtype=np.int64)
    base = 0
    for e in range(E):
        mine = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e][:C]
        for r, (t, j) in enumerate(mine):
            pos[t, j] = base + r
        base += len(mine)
    return pos


@pytest.mark.parametrize("T,E,k,cf", [(37, 5, 2, 1.0), (50, 8, 3, 0.6)])
def test_token_major_capacity(T, E, k, cf):
    rng = _rng(T + 7 * E)
    l = rng.normal(size=(T, E)) + np.linspace(2, 0, E)[None, :]
    idx, _, _ = O.top_k_route(l, k)
    C = O.expert_capacity(T, k, E, cf)
    rank, fill = O.assign_capacity(idx, E, C, token_major=True)
    _, pos = O.dispatch_positions(idx, rank, fill)
    np.testing.assert_array_equal(pos, _dispatch_token_major_by_sorting(idx, E, C))
    # a kept slot of an expert never follows, in token order, a dropped one
    for e in range(E):
        slots = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        kept = [pos[t, j] >= 0 for t, j in slots]
        assert kept == sorted(kept, reverse=True)
    # the two priority orders differ once capacity binds on second choices
    rank_s, _ = O.assign_capacity(idx, E, C)
    assert (rank_s != rank).any()


def test_layer_norm_against_torch_and_backward_by_finite_differences():
    """[P2] 5.2's LayerNorm before the router: layer_norm equals torch's
    F.layer_norm (no affine, eps 1e-5); layer_norm_backward equals central
    differences of <g, layer_norm(x)>."""
    rng = _rng(81)
    x = rng.normal(size=(6, 11)) * 3 + 5.5
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (11,), eps=1e-5).numpy()
    np.testing.assert_allclose(O.layer_norm(x), ref, rtol=1e-12, atol=1e-12)
    g = rng.normal(size=x.shape)
    an = O.layer_norm_backward(x, g)
    h = 1e-6
    num = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num[i, j] = ((g * O.layer_norm(xp)).sum() - (g * O.layer_norm(xm)).sum()) / (2 * h)
    np.testing.assert_allclose(an, num, rtol=1e-6, atol=1e-8)


def test_backward_with_router_layernorm_finite_differences():
    """The layer's gradients with the router's LayerNorm against central
    differences of L (routing fixed, away from ties)."""
    rng = _rng(83)
    T, d, h, E, k = 12, 5, 6, 4, 2
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) / 2, W3=rng.normal(size=(E, h, d)) / 2,
             W2=rng.normal(size=(E, d, h)) / 3)
    cfg = dict(T=T, d=d, h=h, E=E, k=k, act="swiglu", capacity_factor=0.0, lam=0.05, layernorm=True)
    x = rng.normal(size=(T, d)) + 2.0
    dY = rng.normal(size=(T, d))
    g = O.layer_backward(cfg, w, x, dY)

    def loss(xx, ww):
        return O.layer_backward(cfg, ww, xx, dY)["loss"]

    hh = 1e-6
    for (t, i) in [(0, 0), (3, 2), (11, 4)]:
        xp, xm = x.copy(), x.copy()
        xp[t, i] += hh
        xm[t, i] -= hh
        num = (loss(xp, w) - loss(xm, w)) / (2 * hh)
        assert abs(num - g["dX"][t, i]) <= 1e-6 * max(1.0, abs(num)), (t, i, num, g["dX"][t, i])
    for (e, i) in [(0, 1), (2, 3), (3, 0)]:
        wp = dict(w, Wr=w["Wr"].copy())
        wm = dict(w, Wr=w["Wr"].copy())
        wp["Wr"][e, i] += hh
        wm["Wr"][e, i] -= hh
        num = (loss(x, wp) - loss(x, wm)) / (2 * hh)
        assert abs(num - g["dWr"][e, i]) <= 1e-6 * max(1.0, abs(num)), (e, i, num, g["dWr"][e, i])


def test_layernorm_router_ignores_row_offset_and_scale():
    """With the LayerNorm in front of the router ([P2] 5.2) the logits of a
    row do not change when the row is shifted and scaled (up to the 1e-5 in
    the variance), while the plain router's do."""
    rng = _rng(85)
    x = rng.normal(size=(5, 64))
    Wr = rng.normal(size=(8, 64)) / 8
    a = np.array([0.5, 1.0, 2.0, 3.0, 7.0])[:, None]
    b = np.array([-2.0, 0.0, 1.5, 4.0, -9.0])[:, None]
    l0 = O.router_logits(x, Wr, layernorm=True)
    l1 = O.router_logits(a * x + b, Wr, layernorm=True)
    # the eps moves a row's scale by a relative eps/2 * |1/var - 1/(a^2 var)| < 3e-5 here
    np.testing.assert_allclose(l1, l0, rtol=3e-5, atol=1e-9)
    assert np.abs(O.router_logits(a * x + b, Wr) - O.router_logits(x, Wr)).max() > 0.5


def test_balance_variants_closed_forms():
    """[P2] 3.2's lambda*(std + gamma*max) and [P3] 2.3's product form, on
    hand-worked cases and against torch.std (the n-1 form)."""
    counts = np.array([3, 1, 0, 0])
    f = counts / 2.0
    ref = 0.01 * (torch.tensor(f).std().item() + 100 * 1.5)
    assert abs(O.balance_stat(counts, 2, 0.01, "std_max", 100.0) - ref) < 1e-12
    assert abs(O.balance_stat(counts, 2, 0.01, "std_max", 100.0) - 0.01 * (math.sqrt(0.5) + 150)) < 1e-12
    # one expert: the n-1 std is 0, the max term remains
    assert O.balance_stat(np.array([7]), 7, 0.5, "std_max", 3.0) == 0.5 * 3.0
    # product form: token 0 -> experts 0, 1 (0.75, 0.25); token 1 -> 0, 2 (0.6, 0.4)
    idx = np.array([[0, 1], [0, 2]])
    w = np.array([[0.75, 0.25], [0.6, 0.4]])
    imp = O.importance(idx, w, 4)
    np.testing.assert_allclose(imp, [1.35, 0.25, 0.4, 0.0], rtol=0, atol=1e-15)
    v = O.balance_stat(O.usage_counts(idx, 4), 2, 0.01, "switch", imp=imp)
    assert abs(v - 0.01 * (1.0 * 0.675 + 0.5 * 0.125 + 0.5 * 0.2)) < 1e-15
    # perfectly uniform routing: f = k/E, mean weight 1/E -> lambda*k/E
    E, k, T = 8, 2, 64
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    w = np.full((T, k), 0.5)
    v = O.balance_stat(O.usage_counts(idx, E), T, 0.01, "switch", imp=O.importance(idx, w, E))
    assert abs(v - 0.01 * k / E) < 1e-15
    assert O.balance_stat(O.usage_counts(idx, E), T, 0.01, "std_max", 100.0) == pytest.approx(0.01 * 100 * k / E)


@pytest.mark.parametrize("variant", ["std_max", "switch"])
def test_balance_variant_gradients_finite_differences(variant):
    """Each slot's gradient of the balance term against central differences
    in that slot's weight (routing fixed, a unique largest importance)."""
    rng = _rng(87)
    T, E, k = 40, 6, 2
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    idx[3, :] = -1  # a token routed nowhere
    w = rng.uniform(0.1, 0.9, size=(T, k))
    val, g = O.balance_term_grad(idx, w, E, T, 0.05, variant, 7.0)
    imp = O.importance(idx, w, E)
    assert np.sort(imp)[-1] - np.sort(imp)[-2] > 1e-3
    h = 1e-6
    for (t, j) in [(0, 0), (5, 1), (17, 0), (39, 1), (3, 0)]:
        wp, wm = w.copy(), w.copy()
        wp[t, j] += h
        wm[t, j] -= h
        num = (O.balance_term_grad(idx, wp, E, T, 0.05, variant, 7.0)[0]
               - O.balance_term_grad(idx, wm, E, T, 0.05, variant, 7.0)[0]) / (2 * h)
        assert abs(num - g[t, j]) <= 1e-7 * max(1.0, abs(num)), (t, j, num, g[t, j])


@pytest.mark.parametrize("variant", ["cv", "std_max", "switch"])
def test_layer_backward_balance_variants_finite_differences(variant):
    """The whole layer's dX and dWr under each balance term against central
    differences of L = <dY, y> + B (routing fixed, away from ties)."""
    rng = _rng(89)
    T, d, h, E, k = 14, 5, 6, 4, 2
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) / 2, W3=rng.normal(size=(E, h, d)) / 2,
             W2=rng.normal(size=(E, d, h)) / 3)
    cfg = dict(T=T, d=d, h=h, E=E, k=k, act="swiglu", capacity_factor=1.0, lam=0.3, balance=variant,
               gamma=2.0)
    x = rng.normal(size=(T, d))
    dY = rng.normal(size=(T, d))
    g = O.layer_backward(cfg, w, x, dY)
    if variant != "cv":
        cv = O.layer_backward(dict(cfg, balance="cv"), w, x, dY)
        assert np.abs(cv["dWr"] - g["dWr"]).max() > 1e-3  # the term reaches the router

    def loss(xx, ww):
        return O.layer_backward(cfg, ww, xx, dY)["loss"]

    hh = 1e-6
    for (t, i) in [(0, 0), (6, 2), (13, 4)]:
        xp, xm = x.copy(), x.copy()
        xp[t, i] += hh
        xm[t, i] -= hh
        num = (loss(xp, w) - loss(xm, w)) / (2 * hh)
        assert abs(num - g["dX"][t, i]) <= 1e-6 * max(1.0, abs(num)), (t, i, num, g["dX"][t, i])
    for (e, i) in [(0, 1), (2, 3), (3, 0)]:
        wp = dict(w, Wr=w["Wr"].copy())
        wm = dict(w, Wr=w["Wr"].copy())
        wp["Wr"][e, i] += hh
        wm["Wr"][e, i] -= hh
        num = (loss(x, wp) - loss(x, wm)) / (2 * hh)
        assert abs(num - g["dWr"][e, i]) <= 1e-6 * max(1.0, abs(num)), (e, i, num, g["dWr"][e, i])


def test_reroute_overflow_worked_example():
    """[P3] 2.3's alternative to dropping: route the overflow to the next-best
    expert.  T=4, E=3, top-1, C=1: tokens 0-2 all prefer expert 0 (backups
    1, 1, 2), token 3 prefers expert 1.  Token 0 keeps expert 0; token 1's
    backup (expert 1) is taken by token 3 in the first pass, so it stays
    dropped; token 2 moves to expert 2."""
    l = np.array([[3.0, 2.0, 1.0], [3.0, 2.0, 1.0], [3.0, 1.0, 2.0], [0.0, 3.0, 1.0]])
    idx, w, _ = O.top_k_route(l, 1)
    np.testing.assert_array_equal(O.backup_experts(l, 1), [[1], [1], [2], [2]])
    C = O.expert_capacity(4, 1, 3, 0.75, 0)
    assert C == 1
    rank, fill = O.assign_capacity(idx, 3, C)
    served, rank2, fill2 = O.reroute_overflow(idx, O.backup_experts(l, 1), rank, fill, C)
    np.testing.assert_array_equal(served[:, 0], [0, -1, 2, 1])
    np.testing.assert_array_equal(fill2, [0, 0, 1])
    cfg = dict(T=4, E=3, k=1, capacity_factor=0.75, reroute=True)
    r = O.route_and_dispatch(cfg, l, np.eye(3))
    np.testing.assert_array_equal(r["pos"][:, 0], [0, -1, 2, 1])
    np.testing.assert_array_equal(r["kept"], [1, 1, 1])
    assert r["stats"]["rerouted_slots"] == 1 and r["stats"]["kept_slots"] == 3
    # without the flag token 2 is dropped too
    r0 = O.route_and_dispatch(dict(cfg, reroute=False), l, np.eye(3))
    np.testing.assert_array_equal(r0["pos"][:, 0], [0, -1, -1, 1])


@pytest.mark.parametrize("T,E,k,cf,tm", [(300, 8, 2, 0.8, False), (200, 6, 3, 0.6, True), (150, 5, 2, 1.0, False),
                                         (64, 3, 2, 0.5, False)])
def test_reroute_properties(T, E, k, cf, tm):
    """On random skewed logits: the first pass is untouched (every slot kept
    without rerouting keeps its expert and place order); no expert exceeds
    C; a rerouted slot is served by the token's backup of its drop order,
    never by an expert the token already uses; for each expert the rerouted
    slots are exactly the first (C - first-pass rows) candidates aimed at it
    in priority order (greedy); rerouting never lowers the kept count."""
    rng = _rng(91 + T)
    l = rng.normal(size=(T, E)) + np.linspace(2.0, 0.0, E)[None, :]
    cfg = dict(T=T, E=E, k=k, capacity_factor=cf, token_major=tm)
    r0 = O.route_and_dispatch(cfg, l, np.eye(E))
    r1 = O.route_and_dispatch(dict(cfg, reroute=True), l, np.eye(E))
    C = r0["capacity"]
    idx, b = r1["idx"], r1["backup"]
    assert (r1["kept"] <= C).all() and r1["kept"].sum() >= r0["kept"].sum()
    assert r1["stats"]["rerouted_slots"] == r1["kept"].sum() - r0["kept"].sum()
    first = r0["pos"] >= 0
    np.testing.assert_array_equal(r1["served"][first], idx[first])
    # each expert's rows: first-pass rows in their order, then rerouted rows
    for e in range(E):
        o0, o1 = r1["offsets"][e], r1["offsets"][e + 1]
        mine = np.nonzero((r1["served"] == e) & (r1["pos"] >= 0))
        got = np.sort(r1["pos"][mine])
        np.testing.assert_array_equal(got, np.arange(o0, o1))
    order = [(t, j) for t in range(T) for j in range(k)] if tm else [(t, j) for j in range(k) for t in range(T)]
    cand = {e: [] for e in range(E)}
    for t in range(T):
        r = 0
        for j in range(k):
            if not first[t, j]:
                if b[t, r] >= 0:
                    assert b[t, r] not in idx[t]
                    cand[b[t, r]].append((t, j))
                if r1["pos"][t, j] >= 0:
                    assert r1["served"][t, j] == b[t, r]
                r += 1
    for e in range(E):
        room = C - int(first[idx == e].sum())
        ranked = sorted(cand[e], key=order.index)
        taken = {(t, j) for (t, j) in ranked[:max(room, 0)]}
        got = {(t, j) for t, j in zip(*np.nonzero((r1["served"] == e) & ~first))}
        assert got == taken, e
    assert r1["stats"]["rerouted_slots"] > 0


def test_backward_with_reroute_finite_differences():
    """With rerouting ([P3] 2.3), a moved slot's output comes from its backup
    expert but keeps the weight of the router's choice: dX, dWr and the
    backup expert's weights match central differences of L (routing fixed,
    away from ties), and the run does reroute."""
    rng = _rng(93)
    T, d, h, E, k = 16, 5, 6, 4, 2
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) / 2, W3=rng.normal(size=(E, h, d)) / 2,
             W2=rng.normal(size=(E, d, h)) / 3)
    bias = np.array([1.5, 1.0, 0.0, -0.5])
    cfg = dict(T=T, d=d, h=h, E=E, k=k, act="swiglu", capacity_factor=0.5, lam=0.2, reroute=True)
    x = rng.normal(size=(T, d))
    dY = rng.normal(size=(T, d))
    g = O.layer_backward(cfg, w, x, dY, bias)
    r = g["route"] if "route" in g else O.route_and_dispatch(cfg, x, w["Wr"], bias)
    moved = (r["served"] >= 0) & (r["served"] != r["idx"])
    assert moved.any()
    b = int(r["served"][moved][0])

    def loss(xx, ww):
        return O.layer_backward(cfg, ww, xx, dY, bias)["loss"]

    hh = 1e-6
    for (t, i) in [(0, 0), (7, 3), (15, 4)]:
        xp, xm = x.copy(), x.copy()
        xp[t, i] += hh
        xm[t, i] -= hh
        num = (loss(xp, w) - loss(xm, w)) / (2 * hh)
        assert abs(num - g["dX"][t, i]) <= 1e-6 * max(1.0, abs(num)), (t, i, num, g["dX"][t, i])
    for name, ix in [("Wr", (0, 1)), ("Wr", (3, 2)), ("W1", (b, 2, 1)), ("W2", (b, 3, 4))]:
        wp = dict(w, **{name: w[name].copy()})
        wm = dict(w, **{name: w[name].copy()})
        wp[name][ix] += hh
        wm[name][ix] -= hh
        num = (loss(x, wp) - loss(x, wm)) / (2 * hh)
        got = g["d" + name][ix]
        assert abs(num - got) <= 1e-6 * max(1.0, abs(num)), (name, ix, num, got)


@pytest.mark.parametrize("balance", ["cv", "switch"])
def test_backward_raw_probs_finite_differences(balance):
    """With raw softmax weights ([P2] 3.2: output = p1*e1 + p2*e2) every
    logit reaches the loss through the softmax's denominator, so dWr gets
    rows for unselected experts too: dX and dWr against central
    differences of L (routing fixed, away from ties)."""
    rng = _rng(95)
    T, d, h, E, k = 12, 5, 6, 5, 2
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) / 2, W3=rng.normal(size=(E, h, d)) / 2,
             W2=rng.normal(size=(E, d, h)) / 3)
    cfg = dict(T=T, d=d, h=h, E=E, k=k, act="swiglu", capacity_factor=1.0, lam=0.3, raw_probs=True,
               balance=balance)
    x = rng.normal(size=(T, d))
    dY = rng.normal(size=(T, d))
    g = O.layer_backward(cfg, w, x, dY)
    # an expert no token selects still gets a router gradient
    sel = np.zeros(E, bool)
    sel[np.unique(g["route"]["idx"])] = True
    assert (np.abs(g["dlogits"]) > 0).sum() > T * k

    def loss(xx, ww):
        return O.layer_backward(cfg, ww, xx, dY)["loss"]

    hh = 1e-6
    for (t, i) in [(0, 0), (5, 2), (11, 4)]:
        xp, xm = x.copy(), x.copy()
        xp[t, i] += hh
        xm[t, i] -= hh
        num = (loss(xp, w) - loss(xm, w)) / (2 * hh)
        assert abs(num - g["dX"][t, i]) <= 1e-6 * max(1.0, abs(num)), (t, i, num, g["dX"][t, i])
    for (e, i) in [(0, 1), (2, 3), (4, 0)]:
        wp = dict(w, Wr=w["Wr"].copy())
        wm = dict(w, Wr=w["Wr"].copy())
        wp["Wr"][e, i] += hh
        wm["Wr"][e, i] -= hh
        num = (loss(x, wp) - loss(x, wm)) / (2 * hh)
        assert abs(num - g["dWr"][e, i]) <= 1e-6 * max(1.0, abs(num)), (e, i, num, g["dWr"][e, i])

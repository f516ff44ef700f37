"""Shared helpers of the parity tests: seeded inputs with the top-k margin
guard, comparison metrics."""

from __future__ import annotations

import numpy as np
import torch

import moe_synth as S
from oracle import moe_oracle as O

MARGIN = 1e-3


def oracle_cfg(wl, **route) -> dict:
    # the C ABI carries lambda, gamma and the capacity factor as fp32 values;
    # the oracle gets those same values; route: raw_probs, token_major,
    # layernorm, balance, balance_gamma (the oracle's gamma)
    route = dict(route)
    if "balance_gamma" in route:
        route["gamma"] = float(np.float32(route.pop("balance_gamma")))
    return dict(T=wl.T, d=wl.d, h=wl.h, E=wl.E, k=wl.k, act=wl.act,
                capacity_factor=float(np.float32(wl.capacity_factor)),
                min_capacity=wl.min_capacity, lam=float(np.float32(wl.lam)), has_shared=wl.has_shared,
                **route)


def small_gaps(l: np.ndarray, k: int, margin: float = MARGIN) -> np.ndarray:
    """Tokens whose adjacent gaps among the top-(k+1) sorted logits fall below
    `margin` -- where an fp32 and an fp64 router could order differently."""
    kk = min(k + 1, l.shape[1])
    top = -np.sort(-l, axis=1)[:, :kk]
    gaps = top[:, :-1] - top[:, 1:]
    return np.nonzero((gaps < margin).any(axis=1))[0]


def guard(wl, t: dict, max_attempts=50, layernorm=False) -> dict:
    """Redraw (in place) every row of t['x'] whose top-k margins are below
    1e-3, from counter attempt a = 1, 2, ..., until none is left (margins of
    the router that sees LayerNorm(x) when layernorm)."""
    for a in range(1, max_attempts + 1):
        l = O.router_logits(t["x"], t["Wr"], t.get("expert_bias"), t.get("noise"), layernorm=layernorm)
        bad = small_gaps(l, wl.k)
        if bad.size == 0:
            return t
        S.redraw_rows(wl, t["x"], torch.as_tensor(bad), a)
    raise RuntimeError("margin guard did not converge")


def guarded_inputs(wl, device="cpu", parts=None, layernorm=False):
    """Inputs of workload `wl` with every token's top-k margin >= 1e-3."""
    return guard(wl, S.make_inputs(wl, device, parts), layernorm=layernorm)


def to_np(t: torch.Tensor) -> np.ndarray:
    return O.decode(t)


def rel_frob(a: np.ndarray, b: np.ndarray) -> float:
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def max_abs(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.abs(a - b).max()) if a.size else 0.0


def assert_close_bf16(got: np.ndarray, ref: np.ndarray, what: str, rel=1e-2, mabs=2e-2):
    rf, ma = rel_frob(got, ref), max_abs(got, ref)
    assert rf <= rel and ma <= mabs, f"{what}: rel-Frobenius {rf:.3e} (<= {rel}), max-abs {ma:.3e} (<= {mabs})"


def assert_close_bf16_scaled(got: np.ndarray, ref: np.ndarray, what: str, rel=1e-2, frac=3e-2):
    """assert_close_bf16 for rows of any scale: relative-Frobenius <= rel and
    |err| <= frac * max(1, RMS of the element's reference row, |ref|).  The
    bf16 stores of a row (its hidden units, expert outputs and the output
    itself) err by a fixed fraction of the row's scale (sums of products)
    and of the element (the final rounding: half an ulp, up to 2^-8 of
    |ref|).  A fp64 model of those stores on rows with offsets up to +-2 and
    scales up to 3 reaches 1.3e-2 of that scale, so 3e-2 leaves over 2x."""
    rf = rel_frob(got, ref)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    scale = np.maximum(np.maximum(1.0, rms), np.abs(ref))
    worst = float((np.abs(got - ref) / scale).max()) if ref.size else 0.0
    assert rf <= rel and worst <= frac, f"{what}: rel-Frobenius {rf:.3e} (<= {rel}), max |err|/scale {worst:.3e} (<= {frac})"


def round_bf16(a: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round to nearest even) -> fp64."""
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def bf16_storage_model_expert_grads(t: dict, route: dict, dY, e: int) -> dict:
    """Expert e's SwiGLU weight gradients computed in fp64 but with the
    values rounded wherever the layer stores them between kernels: the
    pre-activations g, u in fp32; dA and dB (the tensor-core operands of the
    W1/W3 gradients) in bf16; the weighted hidden rows w*silu(g)*u (the
    operand of the W2 gradient) as a bf16 value plus its bf16 residual.  The
    upstream rows dY enter as stored and the routing weight w (fp32) scales
    the W2 product in fp32.  A model of the storage arithmetic (not the
    oracle): it explains the layer's deviation from the fp64 oracle, so the
    GPU must match it much more tightly."""
    rows, slots = np.nonzero((route["idx"] == e) & (route["pos"] >= 0))
    v = O.decode(t["x"])[rows]
    W1, W3, W2 = (O.decode(t[n][e]) for n in ("W1", "W3", "W2"))
    f32 = lambda a: np.asarray(a, dtype=np.float32).astype(np.float64)
    g, u = f32(v @ W1.T), f32(v @ W3.T)
    w32 = f32(route["w"][rows, slots])[:, None]
    dy = O.decode(dY)[rows]
    dH = w32 * (dy @ W2)
    dA = round_bf16(dH * u * O.silu_grad(g))
    dB = round_bf16(dH * O.silu(g))
    Hw = w32 * O.silu(g) * u
    hi = round_bf16(Hw)
    return dict(dW1=dA.T @ v, dW3=dB.T @ v, dW2=dy.T @ (hi + round_bf16(Hw - hi)))

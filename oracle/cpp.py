"""ctypes binding of the C++ fp64 oracle (``oracle/moe_oracle.cpp``).

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: the tests, the smoke check
and the benchmark's CPU-baseline leg call it; the CUDA library never does.

The library is built with g++ into ``oracle/_build`` (plain -O2, no fused
multiply-adds, so every product is rounded before it is added, as written).
Stored inputs are passed as they are -- bf16 or fp32 CPU tensors, or fp32
numpy arrays -- and the C++ side decodes each element to fp64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmoe_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-Wextra"]

F32, BF16 = 0, 1
ACT = {"gelu": 0, "swiglu": 1}


def build(force: bool = False) -> str:
    """Compile the C++ oracle (only when the source is newer than the library)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(SRC) > os.path.getmtime(LIB):
        os.makedirs(BUILD, exist_ok=True)
        tmp = LIB + f".{os.getpid()}.tmp"
        r = subprocess.run(["g++", *FLAGS, SRC, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("g++ failed on the C++ oracle:\n" + r.stderr)
        os.replace(tmp, LIB)
    return LIB


class _Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("h", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("act", ctypes.c_int), ("dtype", ctypes.c_int),
                ("min_capacity", ctypes.c_int), ("has_shared", ctypes.c_int),
                ("capacity_factor", ctypes.c_float), ("lam", ctypes.c_double), ("balance", ctypes.c_int),
                ("gamma", ctypes.c_double), ("route", ctypes.c_int)]


BALANCE = {"cv": 0, "std_max": 1, "switch": 2}
ROUTE_BITS = {"raw_probs": 1, "token_major": 2, "layernorm": 4, "reroute": 8}


def _route(cfg: dict) -> int:
    """mo_config.route of an oracle cfg."""
    return sum(bit for name, bit in ROUTE_BITS.items() if cfg.get(name))


class _Inputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "Wr", "W1", "W3", "b1", "W2", "b2", "Ws1", "Ws3", "bs1",
                                               "Ws2", "bs2", "bias", "noise")]


class _Outputs(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("kept", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("stats", ctypes.c_void_p)]


class _Grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dX", "dWr", "dW1", "dW3", "dW2", "db1", "db2", "dWs1", "dWs3",
                                               "dWs2", "dbs1", "dbs2", "dl", "y")] + \
               [("loss", ctypes.c_double), ("balance", ctypes.c_double)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i, f, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
        sig = {
            "mo_router_logits": ([i, i, i, i, vp, vp, vp, vp, vp], None),
            "mo_top_k": ([i, i, i, vp, vp, vp], i),
            "mo_router_entropy": ([i, i, vp], d),
            "mo_capacity": ([i, i, i, f, i], i),
            "mo_usage_counts": ([i, i, i, vp, vp], None),
            "mo_assign_capacity": ([i, i, i, i, vp, vp, vp], None),
            "mo_dispatch_positions": ([i, i, i, vp, vp, vp, vp, vp], None),
            "mo_expert_ffn": ([i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp], None),
            "mo_combine": ([i, i, i, vp, vp, vp, vp, vp], None),
            "mo_balance_stat": ([i, i, vp, d], d),
            "mo_layer_forward": ([ctypes.POINTER(_Config), ctypes.POINTER(_Inputs), ctypes.POINTER(_Outputs)], i),
            "mo_expert_ffn_backward": ([i, i, i, i, i] + [vp] * 14, None),
            "mo_balance_term_grad": ([i, i, i, vp, vp, d, i, d, vp], d),
            "mo_layer_norm": ([i, i, i, vp, vp], None),
            "mo_layer_norm_backward": ([i, i, i, vp, vp, vp], None),
            "mo_top_k_probs": ([i, i, i, vp, i, vp, vp], i),
            "mo_assign_capacity_token_major": ([i, i, i, i, vp, vp, vp], None),
            "mo_backup_experts": ([i, i, i, vp, vp], None),
            "mo_reroute_overflow": ([i, i, i, i, vp, vp, vp, vp, i, vp, vp, vp], None),
            "mo_layer_backward": ([ctypes.POINTER(_Config), ctypes.POINTER(_Inputs), vp, ctypes.POINTER(_Grads)],
                                  i),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes, fn.restype = args, res
        _lib = L
    return _lib


# ----------------------------------------------------------------------------
# arguments
# ----------------------------------------------------------------------------

def _stored(a):
    """(pointer, dtype code, keep-alive) of a stored tensor: a bf16 or fp32
    CPU torch tensor, or an fp32 numpy array; None -> null."""
    if a is None:
        return None, None, None
    if isinstance(a, np.ndarray):
        a = np.ascontiguousarray(a, dtype=np.float32)
        return a.ctypes.data, F32, a
    import torch
    a = a.detach().to("cpu").contiguous()
    if a.dtype == torch.bfloat16:
        return a.data_ptr(), BF16, a
    if a.dtype == torch.float32:
        return a.data_ptr(), F32, a
    raise TypeError(f"stored inputs are bf16 or fp32, not {a.dtype}")


def _f32(a):
    """fp32 side input (expert bias, noise) as a contiguous numpy array."""
    if a is None:
        return None
    if not isinstance(a, np.ndarray):
        a = a.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _p(a):
    return None if a is None else a.ctypes.data


# ----------------------------------------------------------------------------
# the oracle's steps
# ----------------------------------------------------------------------------

def capacity(T: int, k: int, E: int, capacity_factor: float, min_capacity: int = 0) -> int:
    return lib().mo_capacity(T, k, E, float(np.float32(capacity_factor)), min_capacity)


def router_logits(x, Wr, expert_bias=None, noise=None) -> np.ndarray:
    px, dt, kx = _stored(x)
    pw, dw, kw = _stored(Wr)
    assert dt == dw
    T, d = kx.shape
    E = kw.shape[0]
    b, n = _f32(expert_bias), _f32(noise)
    l = np.empty((T, E), dtype=np.float64)
    lib().mo_router_logits(T, d, E, dt, px, pw, _p(b), _p(n), l.ctypes.data)
    return l


def top_k(l: np.ndarray, k: int):
    """(idx [T,k] int32, w [T,k] fp64, tokens with a non-finite logit)."""
    l = np.ascontiguousarray(l, dtype=np.float64)
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    nf = lib().mo_top_k(T, E, k, l.ctypes.data, idx.ctypes.data, w.ctypes.data)
    return idx, w, nf


def router_entropy(l: np.ndarray) -> float:
    l = np.ascontiguousarray(l, dtype=np.float64)
    return lib().mo_router_entropy(l.shape[0], l.shape[1], l.ctypes.data)


def usage_counts(idx: np.ndarray, E: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    c = np.empty(E, dtype=np.int64)
    lib().mo_usage_counts(idx.shape[0], idx.shape[1], E, idx.ctypes.data, c.ctypes.data)
    return c


def assign_capacity(idx: np.ndarray, E: int, C: int):
    """(rank [T,k] int32, fill [E] int64), slot-major priority."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    rank = np.empty((T, k), dtype=np.int32)
    fill = np.empty(E, dtype=np.int64)
    lib().mo_assign_capacity(T, k, E, C, idx.ctypes.data, rank.ctypes.data, fill.ctypes.data)
    return rank, fill


def dispatch_positions(idx: np.ndarray, rank: np.ndarray, fill: np.ndarray):
    """(offsets [E+1], pos [T,k]) int64."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    rank = np.ascontiguousarray(rank, dtype=np.int32)
    fill = np.ascontiguousarray(fill, dtype=np.int64)
    T, k = idx.shape
    E = fill.shape[0]
    offsets = np.empty(E + 1, dtype=np.int64)
    pos = np.empty((T, k), dtype=np.int64)
    lib().mo_dispatch_positions(T, k, E, idx.ctypes.data, rank.ctypes.data, fill.ctypes.data,
                                offsets.ctypes.data, pos.ctypes.data)
    return offsets, pos


def expert_ffn(v, act: str, W1, W2, W3=None, b1=None, b2=None) -> np.ndarray:
    """One expert on the stored rows v [n,d] -> fp64 [n,d]."""
    pv, dt, kv = _stored(v)
    n, d = kv.shape
    args = [_stored(a) for a in (W1, W3, b1, W2, b2)]
    h = args[0][2].shape[0]
    for p_, dta, _ in args:
        assert p_ is None or dta == dt, "the weights share the rows' storage type"
    out = np.empty((n, d), dtype=np.float64)
    lib().mo_expert_ffn(n, d, h, ACT[act], dt, pv, *[a[0] for a in args], out.ctypes.data)
    return out


def combine(expert_out: np.ndarray, w: np.ndarray, kept: np.ndarray, shared=None) -> np.ndarray:
    """y = sum over the kept slots of w * expert_out (+ shared); expert_out
    [T,k,d], w [T,k], kept [T,k] bool, shared [T,d] or None."""
    o = np.ascontiguousarray(expert_out, dtype=np.float64)
    T, k, d = o.shape
    w = np.ascontiguousarray(w, dtype=np.float64)
    kp = np.ascontiguousarray(kept, dtype=np.int32)
    s = None if shared is None else np.ascontiguousarray(shared, dtype=np.float64)
    y = np.empty((T, d), dtype=np.float64)
    lib().mo_combine(T, k, d, o.ctypes.data, w.ctypes.data, kp.ctypes.data, _p(s), y.ctypes.data)
    return y


def balance_stat(counts: np.ndarray, T: int, lam: float) -> float:
    c = np.ascontiguousarray(counts, dtype=np.int64)
    return lib().mo_balance_stat(c.shape[0], T, c.ctypes.data, float(lam))


STATS = ("routed_slots", "kept_slots", "dropped_slots", "capacity", "drop_rate", "balance_stat",
         "numeric_error", "router_entropy", "rerouted_slots")


def layer_forward(cfg: dict, weights: dict, x, expert_bias=None, noise=None) -> dict:
    """The whole forward pass.  cfg: T, d, h, E, k, act, capacity_factor,
    min_capacity, lam, balance, gamma, has_shared and the routing flags
    raw_probs, token_major, layernorm, reroute (as for
    moe_oracle.layer_forward);
    weights: Wr, W1, W3, b1, W2, b2, Ws1, Ws3, bs1, Ws2, bs2 (stored
    tensors, absent or None where the layer has none)."""
    T, d, E, k = cfg["T"], cfg["d"], cfg["E"], cfg["k"]
    px, dt, kx = _stored(x)
    keep = [kx]
    inp = _Inputs()
    inp.x = px
    for n in ("Wr", "W1", "W3", "b1", "W2", "b2", "Ws1", "Ws3", "bs1", "Ws2", "bs2"):
        p_, dta, ka = _stored(weights.get(n))
        assert p_ is None or dta == dt, f"{n} shares x's storage type"
        setattr(inp, n, p_)
        keep.append(ka)
    b, nz = _f32(expert_bias), _f32(noise)
    inp.bias, inp.noise = _p(b), _p(nz)
    c = _Config(T=T, d=d, h=cfg["h"], E=E, k=k, act=ACT[cfg["act"]], dtype=dt,
                min_capacity=int(cfg.get("min_capacity", 0)), has_shared=int(bool(cfg.get("has_shared"))),
                capacity_factor=float(np.float32(cfg.get("capacity_factor", 0.0))),
                lam=float(cfg.get("lam", 0.01)), balance=BALANCE[cfg.get("balance", "cv")],
                gamma=float(cfg.get("gamma", 100.0)), route=_route(cfg))
    r = dict(y=np.empty((T, d)), idx=np.empty((T, k), dtype=np.int32), w=np.empty((T, k)),
             counts=np.empty(E, dtype=np.int64), kept=np.empty(E, dtype=np.int64),
             offsets=np.empty(E + 1, dtype=np.int64), pos=np.empty((T, k), dtype=np.int64),
             stats=np.empty(len(STATS)))
    out = _Outputs(**{n: r[n].ctypes.data for n in ("y", "idx", "w", "counts", "kept", "offsets", "pos", "stats")})
    if lib().mo_layer_forward(ctypes.byref(c), ctypes.byref(inp), ctypes.byref(out)) != 0:
        raise ValueError("invalid configuration for the C++ oracle")
    st = dict(zip(STATS, r.pop("stats").tolist()))
    for n in ("routed_slots", "kept_slots", "dropped_slots", "capacity", "numeric_error", "rerouted_slots"):
        st[n] = int(st[n])
    r["stats"] = st
    return r


def expert_ffn_backward(v, g_out: np.ndarray, act: str, W1, W2, W3=None, b1=None, b2=None) -> dict:
    """Chain rule through one expert for the stored rows v [n,d] with the
    fp64 upstream gradient g_out [n,d]: dv, the forward output out, dW1,
    dW2 and dW3 (SwiGLU) or db1, db2 (GeLU), all fp64."""
    pv, dt, kv = _stored(v)
    n, d = kv.shape
    args = [_stored(a) for a in (W1, W3, b1, W2, b2)]
    h = args[0][2].shape[0]
    for p_, dta, _ in args:
        assert p_ is None or dta == dt, "the weights share the rows' storage type"
    go = np.ascontiguousarray(g_out, dtype=np.float64)
    assert go.shape == (n, d)
    r = dict(dv=np.empty((n, d)), out=np.empty((n, d)), dW1=np.zeros((h, d)), dW2=np.zeros((d, h)))
    if act == "swiglu":
        r["dW3"] = np.zeros((h, d))
    else:
        r["db1"], r["db2"] = np.zeros(h), np.zeros(d)
    lib().mo_expert_ffn_backward(n, d, h, ACT[act], dt, pv, go.ctypes.data, *[a[0] for a in args],
                                 r["dv"].ctypes.data, r["out"].ctypes.data, r["dW1"].ctypes.data,
                                 _p(r.get("dW3")), r["dW2"].ctypes.data, _p(r.get("db1")), _p(r.get("db2")))
    return r


def balance_term_grad(idx: np.ndarray, w: np.ndarray, E: int, T: int, lam: float, variant: str = "cv",
                      gamma: float = 100.0):
    """(B, dB/dw [T,k]) of the balance term on the importance I/T in the
    form `variant` (cv, std_max, switch) gives."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    dw = np.empty(idx.shape, dtype=np.float64)
    val = lib().mo_balance_term_grad(T, idx.shape[1], E, idx.ctypes.data, w.ctypes.data, float(lam),
                                     BALANCE[variant], float(gamma), dw.ctypes.data)
    return val, dw


def layer_backward(cfg: dict, weights: dict, x, dY, expert_bias=None, noise=None) -> dict:
    """Gradients of L = <dY, y> + B(I/T) with the routing of cfg (raw_probs,
    token_major, layernorm, reroute) and the balance term of
    cfg["balance"] (cv, std_max or switch, with cfg["gamma"]; cfg and
    weights as for layer_forward; dY [T,d] stored like x).  Keys as moe_oracle.layer_backward's: dX, dWr, dW1, dW2, dW3 or
    db1/db2, the shared expert's dWs1, dWs2, dWs3 or dbs1/dbs2, dlogits, y,
    loss, balance_term."""
    T, d, h, E, k = cfg["T"], cfg["d"], cfg["h"], cfg["E"], cfg["k"]
    act = cfg["act"]
    px, dt, kx = _stored(x)
    pd, dtd, kd = _stored(dY)
    assert dtd == dt, "dY shares x's storage type"
    keep = [kx, kd]
    inp = _Inputs()
    inp.x = px
    for n in ("Wr", "W1", "W3", "b1", "W2", "b2", "Ws1", "Ws3", "bs1", "Ws2", "bs2"):
        p_, dta, ka = _stored(weights.get(n))
        assert p_ is None or dta == dt, f"{n} shares x's storage type"
        setattr(inp, n, p_)
        keep.append(ka)
    b, nz = _f32(expert_bias), _f32(noise)
    inp.bias, inp.noise = _p(b), _p(nz)
    c = _Config(T=T, d=d, h=h, E=E, k=k, act=ACT[act], dtype=dt,
                min_capacity=int(cfg.get("min_capacity", 0)), has_shared=int(bool(cfg.get("has_shared"))),
                capacity_factor=float(np.float32(cfg.get("capacity_factor", 0.0))),
                lam=float(cfg.get("lam", 0.01)), balance=BALANCE[cfg.get("balance", "cv")],
                gamma=float(cfg.get("gamma", 100.0)), route=_route(cfg))
    r = dict(dX=np.empty((T, d)), dWr=np.empty((E, d)), dW1=np.empty((E, h, d)), dW2=np.empty((E, d, h)),
             dlogits=np.empty((T, E)), y=np.empty((T, d)))
    if act == "swiglu":
        r["dW3"] = np.empty((E, h, d))
    else:
        r["db1"], r["db2"] = np.empty((E, h)), np.empty((E, d))
    if cfg.get("has_shared"):
        r["dWs1"], r["dWs2"] = np.empty((h, d)), np.empty((d, h))
        if act == "swiglu":
            r["dWs3"] = np.empty((h, d))
        else:
            r["dbs1"], r["dbs2"] = np.empty(h), np.empty(d)
    g = _Grads(dX=_p(r["dX"]), dWr=_p(r["dWr"]), dW1=_p(r["dW1"]), dW3=_p(r.get("dW3")), dW2=_p(r["dW2"]),
               db1=_p(r.get("db1")), db2=_p(r.get("db2")), dWs1=_p(r.get("dWs1")), dWs3=_p(r.get("dWs3")),
               dWs2=_p(r.get("dWs2")), dbs1=_p(r.get("dbs1")), dbs2=_p(r.get("dbs2")), dl=_p(r["dlogits"]),
               y=_p(r["y"]))
    if lib().mo_layer_backward(ctypes.byref(c), ctypes.byref(inp), pd, ctypes.byref(g)) != 0:
        raise ValueError("invalid configuration for the C++ oracle")
    r["loss"], r["balance_term"] = g.loss, g.balance
    return r


def layer_norm(x) -> np.ndarray:
    """Row-wise layer norm of the stored x [T,d] in fp64 (eps 1e-5)."""
    px, dt, kx = _stored(x)
    T, d = kx.shape
    n = np.empty((T, d))
    lib().mo_layer_norm(T, d, dt, px, n.ctypes.data)
    return n


def layer_norm_backward(x, g: np.ndarray) -> np.ndarray:
    """d<g, layer_norm(x)>/dx for the stored x [T,d]."""
    px, dt, kx = _stored(x)
    T, d = kx.shape
    g = np.ascontiguousarray(g, dtype=np.float64)
    dx = np.zeros((T, d))
    lib().mo_layer_norm_backward(T, d, dt, px, g.ctypes.data, dx.ctypes.data)
    return dx


def top_k_probs(l: np.ndarray, k: int, raw: bool):
    """top_k with raw probabilities (the softmax over all E, not renormalised) when raw."""
    l = np.ascontiguousarray(l, dtype=np.float64)
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    nf = lib().mo_top_k_probs(T, E, k, l.ctypes.data, int(bool(raw)), idx.ctypes.data, w.ctypes.data)
    return idx, w, nf


def assign_capacity_token_major(idx: np.ndarray, E: int, C: int):
    """(rank [T,k] int32, fill [E] int64), token-major priority."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    rank = np.empty((T, k), dtype=np.int32)
    fill = np.empty(E, dtype=np.int64)
    lib().mo_assign_capacity_token_major(T, k, E, C, idx.ctypes.data, rank.ctypes.data, fill.ctypes.data)
    return rank, fill


def backup_experts(l: np.ndarray, k: int) -> np.ndarray:
    """Each token's experts ranked k .. 2k-1 [T,k] int32, -1 where none."""
    l = np.ascontiguousarray(l, dtype=np.float64)
    T, E = l.shape
    b = np.empty((T, k), dtype=np.int32)
    lib().mo_backup_experts(T, E, k, l.ctypes.data, b.ctypes.data)
    return b


def reroute_overflow(idx, backup, rank, fill, C: int, token_major: bool = False):
    """(served [T,k], rank2 [T,k], fill2 [E]) of the second capacity pass."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    backup = np.ascontiguousarray(backup, dtype=np.int32)
    rank = np.ascontiguousarray(rank, dtype=np.int32)
    fill = np.ascontiguousarray(fill, dtype=np.int64)
    T, k = idx.shape
    E = fill.shape[0]
    served = np.empty((T, k), dtype=np.int32)
    rank2 = np.empty((T, k), dtype=np.int32)
    fill2 = np.empty(E, dtype=np.int64)
    lib().mo_reroute_overflow(T, k, E, C, idx.ctypes.data, backup.ctypes.data, rank.ctypes.data, fill.ctypes.data,
                              int(bool(token_major)), served.ctypes.data, rank2.ctypes.data, fill2.ctypes.data)
    return served, rank2, fill2

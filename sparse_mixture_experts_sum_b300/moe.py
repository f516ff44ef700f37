"""ctypes binding of the sparse-MoE layer's C ABI (include/moe.h).

Argument marshalling only: every function forwards torch tensors' device
pointers and the current CUDA stream to the entry point of the same name in
libmoe_b300.so.  No arithmetic of the layer happens here, and there is no
fallback: if the library is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE, MOE_ERR_TIMEOUT = range(6)
ACT = {"gelu": 0, "swiglu": 1}
DTYPE = {"f32": 0, "bf16": 1}
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("h", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("act", ctypes.c_int), ("dtype", ctypes.c_int),
                ("capacity_factor", ctypes.c_float), ("min_capacity", ctypes.c_int),
                ("lambda_balance", ctypes.c_float), ("has_shared", ctypes.c_int), ("route_flags", ctypes.c_int),
                ("balance", ctypes.c_int), ("balance_gamma", ctypes.c_float), ("gemm_flags", ctypes.c_int)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("Wr", "W1", "W3", "W2", "b1", "b2", "Ws1", "Ws3", "Ws2", "bs1", "bs2", "expert_bias")]


class MoeSaved(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("idx", "w", "counts", "kept", "offsets", "pos", "Xp", "H", "Yp", "Sx", "Z", "Hs", "Zs", "logits")]


class MoeGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("dX", "dWr", "dW1", "dW3", "dW2", "db1", "db2", "dWs1", "dWs3", "dWs2", "dbs1", "dbs2")]


class MoeStats(ctypes.Structure):
    _fields_ = [("routed_slots", ctypes.c_longlong), ("kept_slots", ctypes.c_longlong),
                ("dropped_slots", ctypes.c_longlong), ("capacity", ctypes.c_int),
                ("numeric_error", ctypes.c_int), ("drop_rate", ctypes.c_double),
                ("balance_stat", ctypes.c_double), ("router_entropy", ctypes.c_double),
                ("rerouted_slots", ctypes.c_longlong)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


EXPORTS = ("moe_capacity", "moe_workspace_size", "moe_route", "moe_dispatch", "moe_dispatch_static",
           "moe_slot_counts", "moe_dispatch_ep", "moe_permute_rows",
           "moe_expert_ffn", "moe_expert_ffn_shared",
           "moe_combine", "moe_layer_fwd", "moe_layer_bwd", "moe_check_error", "moe_status_string",
           "moe_selftest_wait_timeout")

_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_b300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python __graft_entry__.py` "
                               "or sparse_mixture_experts_sum_b300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        cfgp = ctypes.POINTER(MoeConfig)
        sig = {
            "moe_capacity": [cfgp, ctypes.POINTER(i)],
            "moe_workspace_size": [cfgp, i, ctypes.POINTER(sz)],
            "moe_route": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "moe_dispatch": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "moe_dispatch_static": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp],
            "moe_slot_counts": [cfgp, vp, vp, vp],
            "moe_dispatch_ep": [cfgp, vp, vp, vp, vp, i, vp, vp, vp, vp],
            "moe_permute_rows": [vp, vp, ctypes.c_longlong, ctypes.c_longlong, i, vp, vp],
            "moe_expert_ffn": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "moe_expert_ffn_shared": [cfgp, vp, vp, ctypes.POINTER(MoeWeights), vp, vp, vp, vp, vp, vp, vp],
            "moe_combine": [cfgp, vp, vp, vp, vp, vp, vp],
            "moe_layer_fwd": [cfgp, ctypes.POINTER(MoeWeights), vp, vp, vp, ctypes.POINTER(MoeSaved), vp, vp,
                              sz, vp],
            "moe_layer_bwd": [cfgp, ctypes.POINTER(MoeWeights), vp, ctypes.POINTER(MoeSaved), vp,
                              ctypes.POINTER(MoeGrads), vp, sz, vp],
            "moe_check_error": [vp, ctypes.POINTER(i), vp],
            "moe_status_string": [i],
            "moe_selftest_wait_timeout": [vp, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name == "moe_status_string" else ctypes.c_int
        _lib = L
    return _lib


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {lib().moe_status_string(status).decode()} (status {status})")


def _check(fn, status):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


ROUTE_RAW_PROBS, ROUTE_TOKEN_MAJOR, ROUTE_LAYERNORM, ROUTE_REROUTE = 1, 2, 4, 8
GEMM_CTA_PAIRS, GEMM_SINGLE_CTA = 1, 2
BALANCE = {"cv": 0, "std_max": 1, "switch": 2}


def make_config(T, d, h, E, k, act="swiglu", dtype="bf16", capacity_factor=0.0, min_capacity=0,
                lambda_balance=0.01, has_shared=False, raw_probs=False, token_major=False,
                layernorm=False, balance="cv", balance_gamma=100.0, reroute=False,
                cta_pairs: Optional[bool] = None) -> MoeConfig:
    """cta_pairs: None = the library's choice per launch, True = CTA pair
    tiles, False = single-CTA tiles (moe_config.gemm_flags)."""
    flags = ((ROUTE_RAW_PROBS if raw_probs else 0) | (ROUTE_TOKEN_MAJOR if token_major else 0)
             | (ROUTE_LAYERNORM if layernorm else 0) | (ROUTE_REROUTE if reroute else 0))
    return MoeConfig(T, d, h, E, k, ACT[act], DTYPE[dtype], capacity_factor, min_capacity,
                     lambda_balance, int(bool(has_shared)), flags, BALANCE[balance], balance_gamma,
                     0 if cta_pairs is None else (GEMM_CTA_PAIRS if cta_pairs else GEMM_SINGLE_CTA))


def config_of(wl, **route) -> MoeConfig:
    """MoeConfig of a moe_synth.Workload (route: raw_probs, token_major,
    layernorm, balance, balance_gamma, reroute)."""
    return make_config(wl.T, wl.d, wl.h, wl.E, wl.k, wl.act, wl.dtype, wl.capacity_factor,
                       wl.min_capacity, wl.lam, wl.has_shared, **route)


def moe_capacity(cfg: MoeConfig) -> int:
    c = ctypes.c_int()
    _check("moe_capacity", lib().moe_capacity(ctypes.byref(cfg), ctypes.byref(c)))
    return c.value


def moe_workspace_size(cfg: MoeConfig, training: int = 0) -> int:
    """training: 0 inference forward, 1 training forward, 2 backward."""
    n = ctypes.c_size_t()
    _check("moe_workspace_size", lib().moe_workspace_size(ctypes.byref(cfg), int(training), ctypes.byref(n)))
    return n.value


def workspace(cfg: MoeConfig, training=0, device="cuda") -> torch.Tensor:
    return torch.empty(moe_workspace_size(cfg, int(training)), dtype=torch.uint8, device=device)


def stats_buffer(device="cuda") -> torch.Tensor:
    return torch.zeros(ctypes.sizeof(MoeStats), dtype=torch.uint8, device=device)


def read_stats(buf: torch.Tensor) -> dict:
    raw = bytes(buf.cpu().numpy().tobytes())
    return MoeStats.from_buffer_copy(raw).as_dict()


def moe_route(cfg, x, Wr, expert_bias, noise, idx, w, counts, ws=None, stream=None, entropy=None):
    _check("moe_route", lib().moe_route(ctypes.byref(cfg), _p(x), _p(Wr), _p(expert_bias), _p(noise),
                                        _p(idx), _p(w), _p(counts), _p(entropy), _p(ws), _stream(stream)))


def moe_dispatch(cfg, idx, x, kept, offsets, pos, Xp, stats, ws, stream=None):
    _check("moe_dispatch", lib().moe_dispatch(ctypes.byref(cfg), _p(idx), _p(x), _p(kept), _p(offsets),
                                              _p(pos), _p(Xp), _p(stats), _p(ws), _stream(stream)))


def moe_dispatch_static(cfg, idx, x, kept, offsets, pos, Xp, stats, stream=None):
    """moe_dispatch with the library's own fixed scratch (no workspace)."""
    _check("moe_dispatch_static", lib().moe_dispatch_static(ctypes.byref(cfg), _p(idx), _p(x), _p(kept),
                                                            _p(offsets), _p(pos), _p(Xp), _p(stats),
                                                            _stream(stream)))


def moe_slot_counts(cfg, idx, counts, stream=None):
    _check("moe_slot_counts", lib().moe_slot_counts(ctypes.byref(cfg), _p(idx), _p(counts), _stream(stream)))


def moe_dispatch_ep(cfg, idx, x, rank_adjust, send_adjust, capacity, pos, Xsend, ws, stream=None):
    _check("moe_dispatch_ep", lib().moe_dispatch_ep(ctypes.byref(cfg), _p(idx), _p(x), _p(rank_adjust),
                                                    _p(send_adjust), int(capacity), _p(pos), _p(Xsend), _p(ws),
                                                    _stream(stream)))


def moe_permute_rows(src, index, n, scatter, dst, stream=None):
    """Rows of src/dst (2-D tensors with the same row size): scatter
    dst[index[i]] = src[i], or gather dst[i] = src[index[i]], i < n."""
    row_bytes = src.stride(0) * src.element_size()
    _check("moe_permute_rows", lib().moe_permute_rows(_p(src), _p(index), int(n), int(row_bytes),
                                                      1 if scatter else 0, _p(dst), _stream(stream)))


def moe_expert_ffn(cfg, Xp, offsets, W1, W3, b1, W2, b2, H, Yp, ws, stream=None):
    _check("moe_expert_ffn", lib().moe_expert_ffn(ctypes.byref(cfg), _p(Xp), _p(offsets), _p(W1), _p(W3),
                                                  _p(b1), _p(W2), _p(b2), _p(H), _p(Yp), _p(ws),
                                                  _stream(stream)))


def moe_expert_ffn_shared(cfg, Xp, offsets, weights: dict, H, Yp, x, Hs, Sx, ws, stream=None):
    W = weights_struct(weights)
    _check("moe_expert_ffn_shared", lib().moe_expert_ffn_shared(ctypes.byref(cfg), _p(Xp), _p(offsets), ctypes.byref(W),
                                                                _p(H), _p(Yp), _p(x), _p(Hs), _p(Sx), _p(ws),
                                                                _stream(stream)))


def moe_combine(cfg, Yp, pos, w, Sx, y, stream=None):
    _check("moe_combine", lib().moe_combine(ctypes.byref(cfg), _p(Yp), _p(pos), _p(w), _p(Sx), _p(y),
                                            _stream(stream)))


def weights_struct(t: dict) -> MoeWeights:
    return MoeWeights(*[(t[n].data_ptr() if t.get(n) is not None else None) for n, _ in MoeWeights._fields_])


def saved_struct(t: dict) -> MoeSaved:
    return MoeSaved(*[(t[n].data_ptr() if t.get(n) is not None else None) for n, _ in MoeSaved._fields_])


def moe_layer_fwd(cfg, weights: dict, x, noise, y, saved: Optional[dict], stats, ws, stream=None):
    W = weights_struct(weights)
    S = saved_struct(saved) if saved is not None else None
    _check("moe_layer_fwd", lib().moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(W), _p(x), _p(noise), _p(y),
                                                ctypes.byref(S) if S is not None else None, _p(stats), _p(ws),
                                                ws.numel(), _stream(stream)))


def grads_struct(t: dict) -> MoeGrads:
    return MoeGrads(*[(t[n].data_ptr() if t.get(n) is not None else None) for n, _ in MoeGrads._fields_])


def moe_layer_bwd(cfg, weights: dict, x, saved: dict, dY, grads: dict, ws, stream=None):
    W = weights_struct(weights)
    S = saved_struct(saved)
    G = grads_struct(grads)
    _check("moe_layer_bwd", lib().moe_layer_bwd(ctypes.byref(cfg), ctypes.byref(W), _p(x), ctypes.byref(S), _p(dY),
                                                ctypes.byref(G), _p(ws), ws.numel(), _stream(stream)))


def alloc_grads(cfg: MoeConfig, device="cuda") -> dict:
    """Caller-owned fp32 gradient buffers of one backward (the moe_grads set)."""
    T, E, d, h = cfg.T, cfg.E, cfg.d, cfg.h
    f = dict(dtype=torch.float32, device=device)
    swiglu = cfg.act == ACT["swiglu"]
    out = dict(dX=torch.empty(T, d, **f), dWr=torch.empty(E, d, **f), dW1=torch.empty(E, h, d, **f),
               dW2=torch.empty(E, d, h, **f))
    if swiglu:
        out["dW3"] = torch.empty(E, h, d, **f)
    else:
        out["db1"] = torch.empty(E, h, **f)
        out["db2"] = torch.empty(E, d, **f)
    if cfg.has_shared:
        out["dWs1"] = torch.empty(h, d, **f)
        out["dWs2"] = torch.empty(d, h, **f)
        if swiglu:
            out["dWs3"] = torch.empty(h, d, **f)
        else:
            out["dbs1"] = torch.empty(h, **f)
            out["dbs2"] = torch.empty(d, **f)
    return out


def moe_check_error(ws, stream=None) -> int:
    code = ctypes.c_int()
    st = lib().moe_check_error(_p(ws), ctypes.byref(code), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_TIMEOUT):
        raise MoeError("moe_check_error", st)
    return code.value


def moe_selftest_wait_timeout(ws, stream=None):
    """Enqueue the failure-detection self-test: a kernel whose bounded wait
    runs out (~1 s) and records its code in ws's error word."""
    _check("moe_selftest_wait_timeout", lib().moe_selftest_wait_timeout(_p(ws), _stream(stream)))


def alloc_saved(cfg: MoeConfig, device="cuda", backward=False) -> dict:
    """Caller-owned buffers of one forward (the moe_saved set); with
    backward=True also the pre-activations and shared hidden rows that
    moe_layer_bwd reads (and, with raw softmax weights, the logits)."""
    T, k, E, d, h = cfg.T, cfg.k, cfg.E, cfg.d, cfg.h
    dt = torch.bfloat16 if cfg.dtype == DTYPE["bf16"] else torch.float32
    out = dict(idx=torch.empty(T, k, dtype=torch.int32, device=device),
               w=torch.empty(T, k, dtype=torch.float32, device=device),
               counts=torch.empty(E, dtype=torch.int32, device=device),
               kept=torch.empty(E, dtype=torch.int32, device=device),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=device),
               pos=torch.empty(T, k, dtype=torch.int32, device=device),
               Xp=torch.empty(T * k, d, dtype=dt, device=device),
               H=torch.empty(T * k, h, dtype=dt, device=device),
               Yp=torch.empty(T * k, d, dtype=dt, device=device))
    if cfg.has_shared:
        out["Sx"] = torch.empty(T, d, dtype=dt, device=device)
    if backward:
        hz = 2 * h if cfg.act == ACT["swiglu"] else h
        # pre-activations are fp32 (the backward's activation derivative reads them)
        out["Z"] = torch.empty(T * k, hz, dtype=torch.float32, device=device)
        if cfg.has_shared:
            out["Hs"] = torch.empty(T, h, dtype=dt, device=device)
            out["Zs"] = torch.empty(T, hz, dtype=torch.float32, device=device)
        if cfg.route_flags & ROUTE_RAW_PROBS:
            out["logits"] = torch.empty(T, E, dtype=torch.float32, device=device)
    return out

"""Seeded synthetic inputs for the sparse-MoE layer.

This module is shared by the tests, the benchmark and the callers of the
oracle. It holds none of the layer's arithmetic: only a counter-based random
stream, the transforms that turn it into uniform / normal / Gumbel draws,
the rounding of those draws to the storage type, and the shape recipe of each
workload.

Random stream
-------------
splitmix64 (S. Vigna, "Further scramblings of Marsaglia's xorshift
generators", 2014; public-domain reference definition), written from that
definition:

    state += 0x9E3779B97F4A7C15
    z = state
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    return z ^ (z >> 31)

used counter-style: tensor ``tid`` of workload seed ``seed`` has the key
``K = mix(((seed mod 2^32) << 32) | (tid mod 2^32))`` and its element ``i``
is the ``(i+1)``-th output of splitmix64 started from state ``K``, i.e.
``r_i = mix(K + (i+1)*0x9E3779B97F4A7C15 mod 2^64)``.  Any slice of a tensor
can therefore be produced on its own, on any device, with identical bits.

Transforms (all in fp64)
------------------------
* uniform  ``u_i = ((r_i >> 11) + 0.5) * 2^-53``, strictly inside (0, 1);
* normal   ``z_i = sqrt(-2 ln u_{2i}) * cos(2 pi u_{2i+1})`` (Box-Muller,
  cosine branch only);
* Gumbel   ``g_i = -ln(-ln u_i)``.

Storage rounding: fp64 -> fp32 (round to nearest even), then for bf16 the
fp32 value -> bf16 (round to nearest even).  Integer steps are exact on every
device; the fp64 ``log``/``cos`` of two libraries can differ in the last
place, so a test that feeds the same inputs to both sides generates them once
and copies them, never regenerates them on the other device.

Tensor ids: x=1, Wr=2, W1=3, W3=4, W2=5, Ws1=6, Ws3=7, Ws2=8, b1=9, b2=10,
noise=11, dY=12, x_scale=13, x_shift=14.  A row of x that is redrawn (see
``redraw_rows``) on attempt ``a`` comes from tensor id ``1 + 256*a`` at the
same element counters.

Rows of varying offset and scale (``Workload.x_affine``): row t of x is
``a_t * z + b_t`` before the storage rounding, z the row's normal draws,
``a_t = 0.5 + 2.5 u`` (u the t-th uniform of tensor id 13) and
``b_t = 4 (u' - 0.5)`` (u' the t-th uniform of tensor id 14): activations
whose rows differ in mean and spread, the input a LayerNorm in front of the
router normalises.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterable, Optional

import torch

_MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

TID = dict(x=1, Wr=2, W1=3, W3=4, W2=5, Ws1=6, Ws3=7, Ws2=8, b1=9, b2=10,
           noise=11, dY=12, x_scale=13, x_shift=14)

_CHUNK = 1 << 25  # elements generated per torch pass (bounds temporaries)


def _signed(v: int) -> int:
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def mix64_int(z: int) -> int:
    """The splitmix64 output function on a Python int (exact, slow)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * MIX1) & _MASK64
    z = ((z ^ (z >> 27)) * MIX2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int) -> int:
    return mix64_int(((seed & 0xFFFFFFFF) << 32) | (tid & 0xFFFFFFFF))


def raw_int(seed: int, tid: int, i: int) -> int:
    """Element ``i`` of stream (seed, tid) as an unsigned Python int."""
    return mix64_int(stream_key(seed, tid) + (i + 1) * GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    # logical right shift of int64 bit patterns
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _signed(MIX1)
    z = (z ^ _lsr(z, 27)) * _signed(MIX2)
    return z ^ _lsr(z, 31)


def raw(seed: int, tid: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """int64 bit patterns of elements start..start+n-1 of stream (seed, tid)."""
    key = _signed(stream_key(seed, tid))
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    return _mix64(i * _signed(GAMMA) + key)


def uniform(seed, tid, start, n, device="cpu") -> torch.Tensor:
    r = raw(seed, tid, start, n, device)
    return (_lsr(r, 11).to(torch.float64) + 0.5) * (2.0 ** -53)


def normal(seed, tid, start, n, device="cpu") -> torch.Tensor:
    u = uniform(seed, tid, 2 * start, 2 * n, device).view(n, 2)
    return torch.sqrt(-2.0 * torch.log(u[:, 0])) * torch.cos((2.0 * math.pi) * u[:, 1])


def gumbel(seed, tid, start, n, device="cpu") -> torch.Tensor:
    u = uniform(seed, tid, start, n, device)
    return -torch.log(-torch.log(u))


def store(v64: torch.Tensor, dtype: str) -> torch.Tensor:
    """Round fp64 draws to the storage type: fp32 (RNE), or fp32 then bf16 (RNE)."""
    f32 = v64.to(torch.float32)
    if dtype == "f32":
        return f32
    if dtype == "bf16":
        return f32.to(torch.bfloat16)
    raise ValueError(dtype)


def tensor(kind: str, seed: int, tid: int, shape, dtype: str, scale: float = 1.0,
           device="cpu", start: int = 0) -> torch.Tensor:
    """A tensor of ``kind`` in {'normal','gumbel','uniform'} draws times ``scale``,
    rounded to ``dtype`` ('f32' | 'bf16'), generated chunk by chunk."""
    n = 1
    for s in shape:
        n *= int(s)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    out = torch.empty(n, dtype=tdt, device=device)
    fn = dict(normal=normal, gumbel=gumbel, uniform=uniform)[kind]
    for c0 in range(0, n, _CHUNK):
        c = min(_CHUNK, n - c0)
        v = fn(seed, tid, start + c0, c, device)
        if scale != 1.0:
            v = v * scale
        out[c0:c0 + c] = store(v, dtype)
    return out.view(*shape)


def zipf_pmf(E: int, s: float) -> torch.Tensor:
    """pmf of Zipf(s) on ranks 1..E, fp64: (e+1)^-s / sum_i i^-s."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    p = r ** (-s)
    return p / p.sum()


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape, dtype and input recipe of one workload of the layer."""
    name: str
    T: int
    d: int
    h: int
    E: int
    k: int
    act: str                 # 'gelu' | 'swiglu'
    dtype: str               # 'f32' | 'bf16'
    capacity_factor: float   # <= 0: no capacity limit
    min_capacity: int
    lam: float
    has_shared: bool
    seed: int
    weight_std: Optional[float]  # None: 1/sqrt(fan_in)
    zipf_s: Optional[float]      # per-expert Zipf(s) logit bias
    gumbel: bool                 # Gumbel(0,1) noise on the router logits
    training: bool
    x_affine: bool = False       # rows of x with their own offset and scale
    zipf_log: bool = False       # the Zipf bias as ln(pmf) instead of the pmf itself

    def std(self, fan_in: int) -> float:
        return self.weight_std if self.weight_std is not None else 1.0 / math.sqrt(fan_in)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    # T=64, d=64, E=4, top-2, GeLU d->128->d, fp32, no capacity limit, no shared
    "tiny_fp32": Workload("tiny_fp32", 64, 64, 128, 4, 2, "gelu", "f32", 0.0, 0, 0.01,
                          False, 0, 0.02, None, False, False),
    # T=4096, d=1024, E=16, SwiGLU h=2816, cf=1.0 (C=512)
    "small_prefill": Workload("small_prefill", 4096, 1024, 2816, 16, 2, "swiglu", "bf16",
                              1.0, 0, 0.01, False, 1, None, None, False, False),
    # T=16384, d=4096, E=64, SwiGLU h=14336, cf=1.25 (C=640), Zipf(1.1) logit bias
    "large_prefill": Workload("large_prefill", 16384, 4096, 14336, 64, 2, "swiglu", "bf16",
                              1.25, 0, 0.01, False, 2, None, 1.1, False, False),
    # stress variant of the large prefill: the Zipf(1.1) bias taken as ln(pmf)
    # (a logit spread of 4.6 between the first and last expert), so that the
    # popular experts overflow their capacity (~75% of slots dropped) and
    # most experts receive fewer than one 128-row tile
    "large_prefill_3z": Workload("large_prefill_3z", 16384, 4096, 14336, 64, 2, "swiglu", "bf16",
                                 1.25, 0, 0.01, False, 2, None, 1.1, False, False, zipf_log=True),
    # four experts of the large prefill layer at its rows per expert (~512):
    # the same GEMM tile shapes at 1/16 of the device memory (profiling case)
    "large_prefill_slice": Workload("large_prefill_slice", 1024, 4096, 14336, 4, 2, "swiglu", "bf16",
                                    1.25, 0, 0.01, False, 2, None, 1.1, False, False),
    # fine-grained routing: E=384 routed experts, top-6, plus 1 shared expert;
    # T=8192, d=4096, SwiGLU h=1024 (the widths are this workload's choice),
    # cf=1.25 (C=160)
    "fine_grained": Workload("fine_grained", 8192, 4096, 1024, 384, 6, "swiglu", "bf16", 1.25, 0,
                             0.01, True, 5, None, None, False, False),
    # 96 experts of the fine-grained layer at its rows per expert (~128) plus
    # the shared expert: the same GEMM tile shapes at a quarter of the
    # weights (profiling case)
    "fine_grained_slice": Workload("fine_grained_slice", 2048, 4096, 1024, 96, 6, "swiglu", "bf16", 1.25, 0,
                                   0.01, True, 5, None, None, False, False),
    # T=64, d=4096, E=128 routed + 1 shared, SwiGLU h=8192, no capacity limit
    "decode": Workload("decode", 64, 4096, 8192, 128, 2, "swiglu", "bf16", 0.0, 0, 0.01,
                       True, 3, None, None, False, False),
    # T=32768, d=4096, E=16 + 1 shared, SwiGLU h=14336, Gumbel noise, cf=1.25 (C=5120)
    "training": Workload("training", 32768, 4096, 14336, 16, 2, "swiglu", "bf16", 1.25, 0,
                         0.01, True, 4, None, None, True, True),
}


def make_inputs(wl: Workload, device="cpu", parts: Optional[Iterable[str]] = None) -> dict:
    """Every input tensor of workload ``wl`` (or only ``parts``), on ``device``.

    Weights are [E, out, in] row-major (in = contraction dim, contiguous).
    """
    want = set(parts) if parts is not None else None

    def need(name):
        return want is None or name in want

    T, d, h, E = wl.T, wl.d, wl.h, wl.E
    s, dt = wl.seed, wl.dtype
    out = {}
    if need("x"):
        if wl.x_affine:
            a, b = _row_affine(wl, 0, T, device)
            z = normal(s, TID["x"], 0, T * d, device).reshape(T, d)
            out["x"] = store(z * a[:, None] + b[:, None], dt)
        else:
            out["x"] = tensor("normal", s, TID["x"], (T, d), dt, 1.0, device)
    if need("Wr"):
        out["Wr"] = tensor("normal", s, TID["Wr"], (E, d), dt, wl.std(d), device)
    if need("W1"):
        out["W1"] = tensor("normal", s, TID["W1"], (E, h, d), dt, wl.std(d), device)
    if need("W3") and wl.act == "swiglu":
        out["W3"] = tensor("normal", s, TID["W3"], (E, h, d), dt, wl.std(d), device)
    if need("W2"):
        out["W2"] = tensor("normal", s, TID["W2"], (E, d, h), dt, wl.std(h), device)
    if wl.act == "gelu":
        # the workloads that use GeLU have zero biases
        tdt = torch.float32 if dt == "f32" else torch.bfloat16
        if need("b1"):
            out["b1"] = torch.zeros(E, h, dtype=tdt, device=device)
        if need("b2"):
            out["b2"] = torch.zeros(E, d, dtype=tdt, device=device)
    if wl.has_shared:
        if need("Ws1"):
            out["Ws1"] = tensor("normal", s, TID["Ws1"], (h, d), dt, wl.std(d), device)
        if need("Ws3") and wl.act == "swiglu":
            out["Ws3"] = tensor("normal", s, TID["Ws3"], (h, d), dt, wl.std(d), device)
        if need("Ws2"):
            out["Ws2"] = tensor("normal", s, TID["Ws2"], (d, h), dt, wl.std(h), device)
    if wl.zipf_s is not None and need("expert_bias"):
        pmf = zipf_pmf(E, wl.zipf_s)
        out["expert_bias"] = (torch.log(pmf) if wl.zipf_log else pmf).to(torch.float32).to(device)
    if wl.gumbel and need("noise"):
        out["noise"] = tensor("gumbel", s, TID["noise"], (T, E), "f32", 1.0, device)
    if wl.training and need("dY"):
        out["dY"] = tensor("normal", s, TID["dY"], (T, d), dt, 1.0, device)
    return out


def _row_affine(wl: Workload, t0: int, n: int, device):
    """Scale a_t and offset b_t (fp64) of rows t0 .. t0+n-1 (x_affine)."""
    a = 0.5 + 2.5 * uniform(wl.seed, TID["x_scale"], t0, n, device)
    b = 4.0 * (uniform(wl.seed, TID["x_shift"], t0, n, device) - 0.5)
    return a, b


def redraw_rows(wl: Workload, x: torch.Tensor, rows: torch.Tensor, attempt: int) -> None:
    """Replace rows ``rows`` of x (in place) by their draw of attempt ``attempt``:
    the same element counters of tensor id ``1 + 256*attempt`` (a row keeps
    its offset and scale under x_affine)."""
    d = wl.d
    tid = TID["x"] + 256 * attempt
    for t in rows.tolist():
        v = normal(wl.seed, tid, t * d, d, x.device)
        if wl.x_affine:
            a, b = _row_affine(wl, t, 1, x.device)
            v = v * a[0] + b[0]
        x[t] = store(v, wl.dtype)

"""The C-ABI library loads without a GPU, exports every entry point that
include/moe.h declares, agrees with the header on struct layouts, and
rejects bad arguments before launching anything."""

import ctypes
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

from conftest import ROOT
from oracle import moe_oracle as O

HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def M():
    import sparse_mixture_experts_sum_b300 as pkg
    from sparse_mixture_experts_sum_b300 import build
    build.build()
    pkg.moe.lib()
    return pkg


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(M):
    names = declared_functions()
    assert "moe_layer_fwd" in names and "moe_route" in names
    lib = ctypes.CDLL(M.moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(M.moe.EXPORTS) <= set(names)


def test_struct_layouts_match_header(M):
    """Compile a C program against the header (gcc, no CUDA) that prints
    sizeof/offsetof of the public structs; compare with the ctypes mirror."""
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "moe.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(moe_config), sizeof(moe_weights), sizeof(moe_saved), sizeof(moe_stats));
  printf("%zu %zu %zu %zu\n", offsetof(moe_config, has_shared), offsetof(moe_stats, drop_rate),
         offsetof(moe_stats, balance_stat), offsetof(moe_weights, expert_bias));
  printf("%zu %zu %zu %zu\n", offsetof(moe_config, route_flags), offsetof(moe_stats, router_entropy),
         offsetof(moe_saved, Zs), sizeof(moe_grads));
  printf("%zu\n", offsetof(moe_config, gemm_flags));
  printf("%zu %zu %zu\n", offsetof(moe_config, balance), offsetof(moe_config, balance_gamma),
         offsetof(moe_stats, rerouted_slots));
  return 0;
}'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(prog)
        subprocess.check_call(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), c, "-o", exe])
        out = subprocess.check_output([exe], text=True).split()
    m = M.moe
    got = [ctypes.sizeof(m.MoeConfig), ctypes.sizeof(m.MoeWeights), ctypes.sizeof(m.MoeSaved),
           ctypes.sizeof(m.MoeStats), m.MoeConfig.has_shared.offset, m.MoeStats.drop_rate.offset,
           m.MoeStats.balance_stat.offset, m.MoeWeights.expert_bias.offset,
           m.MoeConfig.route_flags.offset, m.MoeStats.router_entropy.offset, m.MoeSaved.Zs.offset,
           ctypes.sizeof(m.MoeGrads), m.MoeConfig.gemm_flags.offset,
           m.MoeConfig.balance.offset, m.MoeConfig.balance_gamma.offset,
           m.MoeStats.rerouted_slots.offset]
    assert [int(v) for v in out] == got


@pytest.mark.parametrize("T,k,E,cf,minc", [(1024, 2, 16, 1.0, 0), (4096, 2, 16, 1.0, 0), (16384, 2, 64, 1.25, 0),
                                           (32768, 2, 16, 1.25, 0), (64, 2, 4, 0.0, 0), (10, 2, 16, 1.0, 4),
                                           (1000, 3, 7, 1.1, 0), (333, 6, 384, 1.0, 0),
                                           # fp32 cf a hair above the decimal: the exact product sits
                                           # just above an integer, and the ceiling takes the next one
                                           (1000, 2, 16, 0.8, 0), (5, 1, 2, 0.4, 0), (700, 2, 16, 0.8, 0),
                                           # exact integer products, large and tiny factors
                                           (1 << 20, 8, 1024, 0.5, 0), (64, 2, 4, 3e7, 0), (3, 1, 3, 1e-30, 0)])
def test_capacity_matches_oracle(M, T, k, E, cf, minc):
    cfg = M.make_config(T, 64, 64, E, k, capacity_factor=cf, min_capacity=minc)
    assert M.moe_capacity(cfg) == O.expert_capacity(T, k, E, float(np.float32(cf)), minc)


@pytest.mark.parametrize("kw,status", [
    (dict(k=5, E=4), 1), (dict(k=9, E=16), 1), (dict(E=1025), 1), (dict(T=0), 1),
    (dict(d=100), 2), (dict(h=36), 2), (dict(act=7), 1), (dict(route_flags=16), 1), (dict(balance=3), 1),
    (dict(route_flags=8, k=5, E=16), 2),
    (dict(balance_gamma=float("nan")), 1), (dict(gemm_flags=3), 1), (dict(gemm_flags=4), 1)])
def test_bad_configs_rejected(M, kw, status):
    base = dict(T=64, d=64, h=64, E=8, k=2)
    base.update({k: v for k, v in kw.items() if k in base})
    cfg = M.make_config(**base)
    if "act" in kw:
        cfg.act = kw["act"]
    for name in ("route_flags", "balance", "balance_gamma", "gemm_flags"):
        if name in kw:
            setattr(cfg, name, kw[name])
    with pytest.raises(M.moe.MoeError) as ei:
        M.moe_workspace_size(cfg)
    assert ei.value.status == status


def test_tile_choice_flags(M):
    """cta_pairs None leaves the choice to the library (0); True and False
    set MOE_GEMM_CTA_PAIRS and MOE_GEMM_SINGLE_CTA, which validate alone."""
    for arg, flags in ((None, 0), (True, M.moe.GEMM_CTA_PAIRS), (False, M.moe.GEMM_SINGLE_CTA)):
        cfg = M.make_config(64, 64, 64, 8, 2, cta_pairs=arg)
        assert cfg.gemm_flags == flags
        assert M.moe_workspace_size(cfg) > 0


def test_null_pointers_rejected_before_launch(M):
    cfg = M.make_config(64, 64, 64, 8, 2)
    lib = M.moe.lib()
    st = lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None)
    assert st == M.moe.MOE_ERR_INVALID_ARG
    st = lib.moe_layer_fwd(ctypes.byref(cfg), None, None, None, None, None, None, None, 0, None)
    assert st == M.moe.MOE_ERR_INVALID_ARG
    st = lib.moe_expert_ffn(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None, None)
    assert st == M.moe.MOE_ERR_INVALID_ARG


def test_workspace_too_small_rejected(M):
    cfg = M.make_config(64, 64, 64, 8, 2)
    lib = M.moe.lib()
    W = M.moe.MoeWeights(*([16] * 12))
    st = lib.moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(W), ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                           None, None, ctypes.c_void_p(256), 10, None)
    assert st == M.moe.MOE_ERR_WORKSPACE


def test_workspace_sizes(M):
    cfg = M.make_config(16384, 4096, 14336, 64, 2, capacity_factor=1.25)
    inf = M.moe_workspace_size(cfg, False)
    tr = M.moe_workspace_size(cfg, True)
    # inference keeps Xp, H, Yp in the workspace: at least T*k*(2d + h) bf16
    assert inf >= 16384 * 2 * (2 * 4096 + 14336) * 2
    assert tr < inf


def test_workspace_grows_with_the_variants_that_need_scratch(M):
    """The host-side workspace layout makes room for each variant's
    scratch: LayerNorm's weight-row sums (forward) and per-token terms
    (backward), the reroute backups and second-pass ranks, and the product
    balance term's importance words."""
    T, d, h, E, k = 4096, 1024, 2816, 12, 2
    base = M.make_config(T, d, h, E, k, capacity_factor=1.0)
    ln = M.make_config(T, d, h, E, k, capacity_factor=1.0, layernorm=True)
    rr = M.make_config(T, d, h, E, k, capacity_factor=1.0, reroute=True)
    sw = M.make_config(T, d, h, E, k, capacity_factor=1.0, balance="switch")
    for training in (0, 1):
        b = M.moe_workspace_size(base, training)
        assert M.moe_workspace_size(ln, training) >= b + 16 * 4  # E rounded up to 16 sums
        assert M.moe_workspace_size(rr, training) >= b + T * k * 4 * 2  # backups + first-pass ranks
        assert M.moe_workspace_size(sw, training) >= b + E * 8
    assert M.moe_workspace_size(ln, 2) >= M.moe_workspace_size(base, 2) + 3 * T * 4
    # the router scratch pads the logit rows to the 8-column GEMM granule
    e5 = M.make_config(T, d, h, 5, k, capacity_factor=1.0)
    e8 = M.make_config(T, d, h, 8, k, capacity_factor=1.0)
    assert M.moe_workspace_size(e5, 1) >= T * 8 * 4
    assert M.moe_workspace_size(e5, 1) <= M.moe_workspace_size(e8, 1)

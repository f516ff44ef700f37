"""Failure detection on the GPU without a fault: a kernel's bounded wait
runs out on a barrier that nothing completes, records its code in the
workspace error word and returns.  The host reads the status, and the
context stays usable for the next call on the same workspace."""

import ctypes

import numpy as np
import pytest
import torch

import moe_synth as S
import sparse_mixture_experts_sum_b300 as M
from moe_testlib import guarded_inputs
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_gives_up_reports_and_the_context_stays_usable():
    wl = S.WORKLOADS["small_prefill"].replace(T=256, d=256, E=16, seed=43)
    cfg = M.config_of(wl)
    ws = M.moe.workspace(cfg, 1)
    M.moe.moe_selftest_wait_timeout(ws)
    code = ctypes.c_int()
    st = M.moe.lib().moe_check_error(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(code),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == M.moe.MOE_ERR_TIMEOUT and code.value == 0x1FF
    # the same workspace serves the next call, which clears the word
    t = guarded_inputs(wl, "cpu", parts=["x", "Wr"])
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k, device=DEV)
    counts = torch.empty(wl.E, dtype=torch.int32, device=DEV)
    M.moe_route(cfg, t["x"].to(DEV), t["Wr"].to(DEV), None, None, idx, w, counts, ws)
    assert M.moe_check_error(ws) == 0
    ridx, _, _ = O.top_k_route(O.router_logits(t["x"], t["Wr"]), wl.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)

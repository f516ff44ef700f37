"""Expert parallelism's kernels on one GPU: R ranks emulated one after the
other (no collective; the all-to-all is the test's tensor slicing).

Each emulated rank routes its own slice of the batch (moe_route), counts its
slots (moe_slot_counts), and places them with moe_dispatch_ep from the plan
that sparse_mixture_experts_sum_b300.ep derives from all ranks' counts; each
owner scatters its received rows into expert-contiguous order
(moe_permute_rows), runs its experts (moe_expert_ffn) and gathers the
outputs back; each rank combines (moe_combine).  Every row is the same
arithmetic as on one GPU, so the results must be the same bits as
moe_layer_fwd on the whole batch: routing, each owner's rows (the one-GPU Xp
slice of its experts) and y."""

import numpy as np
import pytest
import torch

import moe_synth as S
import sparse_mixture_experts_sum_b300 as M
from sparse_mixture_experts_sum_b300 import ep
from moe_testlib import guarded_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("R", [2, 3])
def test_expert_parallel_kernels_match_one_gpu_layer(R):
    # 12 experts over R ranks; capacity binds (cf 0.8); the groups average
    # under 256 rows both in the whole layer and in each owner's block
    wl = S.WORKLOADS["small_prefill"].replace(T=1200, d=256, h=384, E=12, capacity_factor=0.8, seed=37)
    t = guarded_inputs(wl, DEV)
    cfg = M.config_of(wl)
    T, d, h, E, k = wl.T, wl.d, wl.h, wl.E, wl.k
    C = M.moe_capacity(cfg)
    # the one-GPU layer
    sv = M.moe.alloc_saved(cfg)
    y_ref = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    M.moe_layer_fwd(cfg, {n: t.get(n) for n in ("Wr", "W1", "W3", "W2")}, t["x"], None, y_ref, sv, None,
                    M.moe.workspace(cfg, 1))
    assert (sv["pos"] < 0).any()
    # R ranks of uneven size
    cut = np.linspace(0, T, R + 1).astype(int)
    cut[1] -= 37
    first = ep.expert_blocks(E, R)
    ranks = []
    for r in range(R):
        cr = M.make_config(int(cut[r + 1] - cut[r]), d, h, E, k, "swiglu", "bf16", capacity_factor=0.0)
        x = t["x"][cut[r]:cut[r + 1]].contiguous()
        idx = torch.empty(cr.T, k, dtype=torch.int32, device=DEV)
        w = torch.empty(cr.T, k, dtype=torch.float32, device=DEV)
        routed = torch.empty(E, dtype=torch.int32, device=DEV)
        ws = M.moe.workspace(cr, 1)
        M.moe_route(cr, x, t["Wr"], None, None, idx, w, routed, ws)
        counts = torch.empty(k, E, dtype=torch.int32, device=DEV)
        M.moe.moe_slot_counts(cr, idx, counts)
        ranks.append(dict(cfg=cr, x=x, idx=idx, w=w, ws=ws, counts=counts))
    counts_all = np.stack([rk["counts"].cpu().numpy() for rk in ranks])
    for r, rk in enumerate(ranks):
        # the counts are the per-slot histogram of the routing
        idx = rk["idx"].cpu().numpy()
        for j in range(k):
            np.testing.assert_array_equal(counts_all[r, j], np.bincount(idx[:, j], minlength=E))
        np.testing.assert_array_equal(idx, sv["idx"][cut[r]:cut[r + 1]].cpu().numpy())
        plan = ep.make_plan(counts_all, C, r)
        n_send = int(plan.send_splits.sum())
        pos = torch.empty(rk["cfg"].T, k, dtype=torch.int32, device=DEV)
        Xsend = torch.empty(max(1, n_send), d, dtype=torch.bfloat16, device=DEV)
        M.moe.moe_dispatch_ep(rk["cfg"], rk["idx"], rk["x"], torch.as_tensor(plan.rank_adjust, dtype=torch.int32,
                                                                            device=DEV),
                              torch.as_tensor(plan.send_adjust, dtype=torch.int32, device=DEV), C, pos, Xsend,
                              rk["ws"])
        p = pos.cpu().numpy()
        # kept exactly where the one-GPU layer keeps; each send row once
        np.testing.assert_array_equal(p >= 0, sv["pos"][cut[r]:cut[r + 1]].cpu().numpy() >= 0)
        assert (np.sort(p[p >= 0]) == np.arange(n_send)).all()
        rk.update(plan=plan, pos=pos, Xsend=Xsend[:n_send], splits=np.concatenate([[0], np.cumsum(plan.send_splits)]))
    # owners: receive, place, run their experts, return
    Yret = []
    for o in range(R):
        plan = ranks[o]["plan"]
        Xrecv = torch.cat([rk["Xsend"][rk["splits"][o]:rk["splits"][o + 1]] for rk in ranks])
        f, l = int(first[o]), int(first[o + 1])
        n_loc = plan.local_rows
        lcfg = M.make_config(-(-n_loc // k), d, h, l - f, k, "swiglu", "bf16")
        rows = lcfg.T * k
        rpos = torch.as_tensor(plan.recv_pos, dtype=torch.int32, device=DEV)
        Xl = torch.empty(rows, d, dtype=torch.bfloat16, device=DEV)
        M.moe.moe_permute_rows(Xrecv, rpos, Xrecv.shape[0], True, Xl)
        a, b = int(sv["offsets"][f]), int(sv["offsets"][l])
        assert b - a == n_loc
        assert torch.equal(Xl[:n_loc], sv["Xp"][a:b])  # the one-GPU rows of this owner's experts
        H = torch.empty(rows, h, dtype=torch.bfloat16, device=DEV)
        Yl = torch.empty(rows, d, dtype=torch.bfloat16, device=DEV)
        M.moe_expert_ffn(lcfg, Xl, torch.as_tensor(plan.local_offsets, dtype=torch.int32, device=DEV),
                         t["W1"][f:l], t["W3"][f:l], None, t["W2"][f:l], None, H, Yl, M.moe.workspace(lcfg, 1))
        assert torch.equal(Yl[:n_loc], sv["Yp"][a:b])
        Y = torch.empty(Xrecv.shape[0], d, dtype=torch.bfloat16, device=DEV)
        M.moe.moe_permute_rows(Yl, rpos, Xrecv.shape[0], False, Y)
        Yret.append((Y, np.concatenate([[0], np.cumsum(plan.recv_splits)])))
    for r, rk in enumerate(ranks):
        Yback = torch.cat([Y[rs[r]:rs[r + 1]] for Y, rs in Yret])
        y = torch.empty(rk["cfg"].T, d, dtype=torch.bfloat16, device=DEV)
        M.moe_combine(rk["cfg"], Yback, rk["pos"], rk["w"], None, y)
        assert torch.equal(y, y_ref[cut[r]:cut[r + 1]]), r


def test_permute_rows_scatter_and_gather():
    """dst[map[i]] = src[i] and dst[i] = src[map[i]], rows of 48 bytes, a
    negative map entry skipped."""
    src = torch.arange(5 * 24, dtype=torch.int16, device=DEV).view(5, 24)
    m = torch.tensor([3, 0, -1, 4, 1], dtype=torch.int32, device=DEV)
    dst = torch.full((5, 24), -1, dtype=torch.int16, device=DEV)
    M.moe.moe_permute_rows(src, m, 5, True, dst)
    ref = torch.full((5, 24), -1, dtype=torch.int16)
    for i, v in enumerate(m.tolist()):
        if v >= 0:
            ref[v] = src[i].cpu()
    assert torch.equal(dst.cpu(), ref)
    back = torch.full((5, 24), -1, dtype=torch.int16, device=DEV)
    M.moe.moe_permute_rows(dst, m, 5, False, back)
    for i, v in enumerate(m.tolist()):
        assert torch.equal(back[i].cpu(), src[i].cpu() if v >= 0 else torch.full((24,), -1, dtype=torch.int16))


def test_expert_parallel_layer_forward_on_one_rank():
    """ep.layer_forward with its collectives (NCCL, one rank owning every
    expert): the same bits as moe_layer_fwd."""
    import socket
    import torch.distributed as dist
    wl = S.WORKLOADS["small_prefill"].replace(T=700, d=256, h=384, E=8, capacity_factor=0.9, seed=39)
    t = guarded_inputs(wl, DEV)
    cfg = M.config_of(wl)
    weights = {n: t.get(n) for n in ("Wr", "W1", "W3", "W2")}
    y_ref = torch.empty(wl.T, wl.d, dtype=torch.bfloat16, device=DEV)
    M.moe_layer_fwd(cfg, weights, t["x"], None, y_ref, None, None, M.moe.workspace(cfg, 0))
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device(DEV, torch.cuda.current_device()))
    try:
        y = torch.empty_like(y_ref)
        plan = ep.layer_forward(cfg, {n: t[n] for n in ("W1", "W3", "W2")}, t["Wr"], t["x"], y,
                                M.moe.workspace(cfg, 1), M.moe_capacity(cfg))
    finally:
        dist.destroy_process_group()
    assert plan.stats["kept_slots"] < wl.T * wl.k  # capacity binds
    assert torch.equal(y, y_ref)

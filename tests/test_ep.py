"""Expert parallelism on CPU ranks (gloo): the plan and the exchange of
sparse_mixture_experts_sum_b300.ep give, on every rank, what the fp64 oracle's
one-batch layer gives for the ranks' batches concatenated in rank order.

Each rank routes its own tokens (the oracle's router on its slice), counts
its slots per (slot, expert), and the ranks exchange the counts and build the
plan; the per-slot steps the library's kernels do on a GPU (placing slots,
permuting rows, the experts, the combine) are done here in numpy from the
plan's tables, and the rows travel with gloo's all-to-all.  Checked against
the oracle on the whole batch: kept slots and expert offsets exactly, each
owner's expert-contiguous rows bit for bit, and y to 1e-12."""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(world):
    """The whole batch (seeded) and each rank's token range (uneven)."""
    rng = np.random.default_rng(100 + world)
    T, d, h, E, k = 96, 12, 16, 5 if world == 3 else 6, 2
    x = rng.normal(size=(T, d))
    w = dict(Wr=rng.normal(size=(E, d)), W1=rng.normal(size=(E, h, d)) / 3, W3=rng.normal(size=(E, h, d)) / 3,
             W2=rng.normal(size=(E, d, h)) / 4)
    bias = np.linspace(1.5, 0.0, E)  # a skew, so that capacity binds
    cut = np.linspace(0, T, world + 1).astype(int)
    cut[1] += 7                       # ranks of different sizes
    cfg = dict(T=T, d=d, h=h, E=E, k=k, act="swiglu", capacity_factor=0.8, has_shared=False, lam=0.01)
    return cfg, x, w, bias, cut


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    from oracle import moe_oracle as O
    from sparse_mixture_experts_sum_b300 import ep

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, x, w, bias, cut = _problem(world)
        T, d, E, k = cfg["T"], cfg["d"], cfg["E"], cfg["k"]
        C = O.expert_capacity(T, k, E, cfg["capacity_factor"])
        xr = x[cut[rank]:cut[rank + 1]]
        Tr = xr.shape[0]
        idx, wts, _ = O.top_k_route(O.router_logits(xr, w["Wr"], bias), k)
        counts = np.zeros((k, E), dtype=np.int64)
        for j in range(k):
            np.add.at(counts[j], idx[:, j], 1)
        plan = ep.make_plan(ep.exchange_counts(torch.as_tensor(counts)), C, rank)
        # placing this rank's slots: local slot-major rank L per expert, kept
        # iff L + rank_adjust < C, at send row L + send_adjust
        run = np.zeros(E, dtype=np.int64)
        sidx = -np.ones((Tr, k), dtype=np.int64)
        for j in range(k):
            for t in range(Tr):
                e = idx[t, j]
                L = run[e]
                run[e] += 1
                if L + plan.rank_adjust[j, e] < C:
                    sidx[t, j] = L + plan.send_adjust[j, e]
        n_send = int(plan.send_splits.sum())
        assert (np.sort(sidx[sidx >= 0]) == np.arange(n_send)).all()  # every send row filled once
        Xsend = np.zeros((n_send, d))
        tt, jj = np.nonzero(sidx >= 0)
        Xsend[sidx[tt, jj]] = xr[tt]
        Xrecv = ep.all_to_all_rows(torch.as_tensor(Xsend), plan.send_splits, plan.recv_splits).numpy()
        # the owner's block: received rows at their one-GPU places
        f, l = int(plan.first[rank]), int(plan.first[rank + 1])
        Xp = np.full((plan.local_rows, d), np.nan)
        Xp[plan.recv_pos] = Xrecv
        Yp = np.zeros_like(Xp)
        for e in range(f, l):
            a, b = plan.local_offsets[e - f], plan.local_offsets[e - f + 1]
            if b > a:
                Yp[a:b] = O.expert_ffn(Xp[a:b], "swiglu", **O.expert_params(w, e, "swiglu"))
        Yback = ep.all_to_all_rows(torch.as_tensor(Yp[plan.recv_pos]), plan.recv_splits, plan.send_splits).numpy()
        y = np.zeros((Tr, d))
        for t, j in zip(tt, jj):
            y[t] += wts[t, j] * Yback[sidx[t, j]]
        q.put((rank, plan.offsets, plan.stats["kept_slots"], Xp, y))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_exchange_matches_one_batch_oracle(world):
    sys.path.insert(0, ROOT)
    from oracle import moe_oracle as O
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in range(world)), key=lambda v: v[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg, x, w, bias, cut = _problem(world)
    ref = O.layer_forward(cfg, w, x, bias)
    assert (ref["pos"] < 0).any()  # capacity binds
    from sparse_mixture_experts_sum_b300 import ep
    first = ep.expert_blocks(cfg["E"], world)
    Xp_ref = np.zeros((int(ref["offsets"][-1]), cfg["d"]))
    t_idx, j_idx = np.nonzero(ref["pos"] >= 0)
    Xp_ref[ref["pos"][t_idx, j_idx]] = x[t_idx]
    for rank, offsets, kept, Xp, y in out:
        np.testing.assert_array_equal(offsets, ref["offsets"])
        assert kept == ref["stats"]["kept_slots"]
        a, b = ref["offsets"][first[rank]], ref["offsets"][first[rank + 1]]
        np.testing.assert_array_equal(Xp, Xp_ref[a:b])  # the one-GPU rows of this rank's experts
        np.testing.assert_allclose(y, ref["y"][cut[rank]:cut[rank + 1]], rtol=0, atol=1e-12)


def test_plan_tables_on_a_hand_worked_case():
    """Two ranks of two tokens, E = 2, k = 2, C = 3.  Rank 0's tokens both
    choose (expert 0, then expert 1); rank 1's choose (0, 1) and (1, 0).
    Expert 0 sees, in priority order, rank 0's two first choices, rank 1's
    first choice, then rank 1's second choice (dropped: C = 3); expert 1 sees
    rank 1's first choice, rank 0's two second choices, then rank 1's second
    choice (dropped)."""
    sys.path.insert(0, ROOT)
    from sparse_mixture_experts_sum_b300 import ep
    counts = np.array([[[2, 0], [0, 2]],     # rank 0: [j][e]
                       [[1, 1], [1, 1]]])    # rank 1
    p0 = ep.make_plan(counts, 3, 0)
    p1 = ep.make_plan(counts, 3, 1)
    np.testing.assert_array_equal(p0.B[:, :, 0], [[0, 3], [2, 3]])  # expert 0: runs start at 0, 3 | 2, 3
    np.testing.assert_array_equal(p0.kept[:, :, 0], [[2, 0], [1, 0]])
    np.testing.assert_array_equal(p0.kept[:, :, 1], [[0, 2], [1, 0]])
    np.testing.assert_array_equal(p0.offsets, [0, 3, 6])
    assert p0.stats["kept_slots"] == 6 and p0.stats["routed_slots"] == 8
    # rank 0 owns expert 0, rank 1 expert 1; sends and receipts agree
    np.testing.assert_array_equal(p0.send_splits, [2, 2])
    np.testing.assert_array_equal(p1.send_splits, [1, 1])
    np.testing.assert_array_equal(p0.recv_splits, [2, 1])
    np.testing.assert_array_equal(p1.recv_splits, [2, 1])
    # expert 0's rows: rank 0's two (global ranks 0, 1), then rank 1's first choice (2)
    np.testing.assert_array_equal(p0.recv_pos, [0, 1, 2])
    # expert 1's rows: rank 0's second choices (ranks 1, 2), rank 1's first choice (0)
    np.testing.assert_array_equal(p1.recv_pos, [1, 2, 0])

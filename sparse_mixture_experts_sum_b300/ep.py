"""Expert parallelism for the MoE layer: experts split over ranks, tokens sent
to the experts' owners and back by all-to-all.

Sources: [P1] "'More parameters is better' is not the story..." 4.2-4.3
(experts placed on different devices, tokens dispatched to them); [P2] "MoE
mixture-of-experts architecture: principles and engineering practice" 4.1
(grouped all-to-all); [P5] "Training a 200B LLM from scratch 5/25", section
"Experts on different GPUs: a new kind of waiting".

R ranks each hold their own batch of tokens, the (replicated) router, and the
weights of a contiguous block of experts.  The layer gives, on every rank,
the rows the one-GPU layer gives for the ranks' batches concatenated in rank
order: the capacity C is the global one, and slot-major priority runs over
all ranks' first choices (rank 0's tokens, then rank 1's, ...) before any
second choice.  One small exchange makes that possible: the per-(slot,
expert) routed counts, [R, k, E] integers.  From them every rank derives the
same plan (make_plan):

  B[r,j,e]  = the slots ahead of rank r's slot-j run for expert e in priority
              order: all ranks' slots j' < j routed to e, then ranks r' < r
              at slot j
  kept      = clip(C - B, 0, counts): the slots of each run that e keeps
  offsets   = the exclusive scan over experts of sum(kept): the one-GPU
              expert-contiguous layout
  rank r's slot (t, j) routed to e, with L its rank in its run, is kept iff
  B + L < C, and sits at global row offsets[e] + B + L.

Each rank's send buffer holds its kept rows by owner, expert, slot and token
(the all-to-all splits follow); an owner places the rows it receives at their
global rows inside its block of experts, which is the one-GPU Xp slice of its
experts, runs its experts there, and returns the outputs in received order.

This module is host logic only: the plan is a handful of integer tables.
Every step on the rows runs in the library's kernels (moe_route,
moe_slot_counts, moe_dispatch_ep, moe_permute_rows, moe_expert_ffn,
moe_combine) or in torch.distributed's collectives.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np


def expert_blocks(E: int, world: int) -> np.ndarray:
    """first[o] .. first[o+1]: the experts rank o owns (contiguous blocks of
    ceil(E / world); the last ranks may own fewer, or none)."""
    per = -(-E // world)
    return np.array([min(E, o * per) for o in range(world + 1)], dtype=np.int64)


@dataclasses.dataclass
class Plan:
    """One rank's view of the expert-parallel dispatch (all int64 numpy)."""
    rank: int
    world: int
    C: int
    first: np.ndarray          # [R+1] expert blocks
    B: np.ndarray              # [R, k, E] slots ahead of each run
    kept: np.ndarray           # [R, k, E] kept slots of each run
    offsets: np.ndarray        # [E+1] one-GPU expert offsets
    rank_adjust: np.ndarray    # [k, E] this rank: B - its own earlier-slot runs
    send_adjust: np.ndarray    # [k, E] this rank: start of the run in the send buffer - the same
    send_splits: np.ndarray    # [R] rows this rank sends to each owner
    recv_splits: np.ndarray    # [R] rows this rank receives from each source
    recv_pos: np.ndarray       # [sum recv_splits] place of each received row in the local block
    local_offsets: np.ndarray  # [E_local+1] this rank's experts in its local block
    stats: dict                # routed and kept slots over all ranks, C, per-expert counts and kept

    @property
    def local_rows(self) -> int:
        return int(self.local_offsets[-1])


def make_plan(counts: np.ndarray, C: int, rank: int, first: Optional[np.ndarray] = None) -> Plan:
    """The plan of `rank` from every rank's per-(slot, expert) routed counts
    (counts[r, j, e] = #{t of rank r : idx[t, j] = e}) and the global
    capacity C (for no limit, C >= the global T)."""
    counts = np.asarray(counts, dtype=np.int64)
    R, k, E = counts.shape
    if first is None:
        first = expert_blocks(E, R)
    tot_j = counts.sum(axis=0)                                   # [k, E]
    ahead_j = np.cumsum(tot_j, axis=0) - tot_j                   # all ranks' slots j' < j
    ahead_r = np.cumsum(counts, axis=0) - counts                 # ranks r' < r at slot j
    B = ahead_j[None, :, :] + ahead_r
    kept = np.clip(C - B, 0, counts)
    fill = kept.sum(axis=(0, 1))
    offsets = np.concatenate([[0], np.cumsum(fill)]).astype(np.int64)
    # send layout of every rank: experts ascending (owners hold ascending
    # blocks, so this is owner by owner), each expert's runs by slot
    kept_re = kept.sum(axis=1)                                   # [R, E]
    e_start = np.cumsum(kept_re, axis=1) - kept_re               # [R, E]
    j_start = np.cumsum(kept, axis=1) - kept                     # [R, k, E]
    S = e_start[:, None, :] + j_start
    own_ahead = np.cumsum(counts[rank], axis=0) - counts[rank]   # this rank's slots j' < j
    f, l = int(first[rank]), int(first[rank + 1])
    send_splits = np.array([kept_re[rank, first[o]:first[o + 1]].sum() for o in range(R)], dtype=np.int64)
    recv_splits = np.array([kept_re[r, f:l].sum() for r in range(R)], dtype=np.int64)
    # the rows received from each source come expert by expert, slot by slot
    pos: List[np.ndarray] = []
    for r in range(R):
        for e in range(f, l):
            for j in range(k):
                n = int(kept[r, j, e])
                if n:
                    pos.append(offsets[e] - offsets[f] + B[r, j, e] + np.arange(n, dtype=np.int64))
    recv_pos = np.concatenate(pos) if pos else np.zeros(0, dtype=np.int64)
    routed = int(counts.sum())
    kept_total = int(fill.sum())
    stats = dict(routed_slots=routed, kept_slots=kept_total, capacity=int(C),
                 counts=tot_j.sum(axis=0), kept=fill)
    return Plan(rank=rank, world=R, C=int(C), first=first, B=B, kept=kept, offsets=offsets,
                rank_adjust=B[rank] - own_ahead, send_adjust=S[rank] - own_ahead, send_splits=send_splits,
                recv_splits=recv_splits, recv_pos=recv_pos, local_offsets=offsets[f:l + 1] - offsets[f],
                stats=stats)


def exchange_counts(counts_local, group=None) -> np.ndarray:
    """all_gather of every rank's [k, E] counts -> numpy int64 [R, k, E]."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    c = counts_local.to(torch.int64)
    out = [torch.empty_like(c) for _ in range(world)]
    dist.all_gather(out, c, group=group)
    return torch.stack(out).cpu().numpy()


def all_to_all_rows(send, send_splits, recv_splits, group=None):
    """Rows of `send` (split by destination) to their ranks; returns the
    received rows, split by source."""
    import torch
    import torch.distributed as dist
    recv = send.new_empty((int(np.sum(recv_splits)),) + tuple(send.shape[1:]))
    dist.all_to_all_single(recv, send, [int(v) for v in recv_splits], [int(v) for v in send_splits], group=group)
    return recv


def layer_forward(cfg, weights_local: dict, Wr, x, y, ws, C: int, group=None, expert_bias=None, noise=None,
                  stream=None):
    """The layer forward of this rank (bf16, slot-major priority, no shared
    expert here -- add it locally, it needs no exchange).  cfg: this rank's
    config (T = its tokens, E = all experts); weights_local: W1, W3, W2 (and
    b1, b2) of its own experts only, [E_local, ...]; Wr [E, d] replicated;
    C: the global capacity; ws: >= moe_workspace_size(cfg, 1) bytes.  Writes
    y [T, d] and returns the plan."""
    import torch
    import torch.distributed as dist
    from . import moe as M
    dev = x.device
    T, k, E, d, h = cfg.T, cfg.k, cfg.E, cfg.d, cfg.h
    rank = dist.get_rank(group)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    routed = torch.empty(E, dtype=torch.int32, device=dev)
    M.moe_route(cfg, x, Wr, expert_bias, noise, idx, w, routed, ws, stream)
    counts = torch.empty(k, E, dtype=torch.int32, device=dev)
    M.moe_slot_counts(cfg, idx, counts, stream)
    plan = make_plan(exchange_counts(counts, group), C, rank)
    adj = torch.as_tensor(plan.rank_adjust.astype(np.int32), device=dev)
    sadj = torch.as_tensor(plan.send_adjust.astype(np.int32), device=dev)
    pos = torch.empty(T, k, dtype=torch.int32, device=dev)
    Xsend = torch.empty(max(1, int(plan.send_splits.sum())), d, dtype=x.dtype, device=dev)
    M.moe_dispatch_ep(cfg, idx, x, adj, sadj, C, pos, Xsend, ws, stream)
    Xrecv = all_to_all_rows(Xsend[:int(plan.send_splits.sum())], plan.send_splits, plan.recv_splits, group)
    # this rank's experts over their rows, in the one-GPU layout of the block
    f, l = int(plan.first[rank]), int(plan.first[rank + 1])
    n_loc = plan.local_rows
    Yret = torch.empty(Xrecv.shape[0], d, dtype=x.dtype, device=dev)
    if l > f and n_loc > 0:
        rpos = torch.as_tensor(plan.recv_pos.astype(np.int32), device=dev)
        # the owner's layer view: its experts, at least n_loc rows (T*k)
        lcfg = M.make_config(-(-n_loc // k), d, h, l - f, k, "swiglu" if cfg.act == M.ACT["swiglu"] else "gelu",
                             "bf16")
        rows = lcfg.T * k
        Xl = torch.empty(rows, d, dtype=x.dtype, device=dev)
        M.moe_permute_rows(Xrecv, rpos, Xrecv.shape[0], True, Xl, stream)
        H = torch.empty(rows, h, dtype=x.dtype, device=dev)
        Yp = torch.empty(rows, d, dtype=x.dtype, device=dev)
        offs = torch.as_tensor(plan.local_offsets.astype(np.int32), device=dev)
        lws = M.workspace(lcfg, 1, device=dev)
        M.moe_expert_ffn(lcfg, Xl, offs, weights_local["W1"], weights_local.get("W3"), weights_local.get("b1"),
                         weights_local["W2"], weights_local.get("b2"), H, Yp, lws, stream)
        M.moe_permute_rows(Yp, rpos, Xrecv.shape[0], False, Yret, stream)
    Yback = all_to_all_rows(Yret, plan.recv_splits, plan.send_splits, group)
    if Yback.shape[0] == 0:  # nothing kept: every pos is -1, no row is read
        Yback = torch.empty(1, d, dtype=x.dtype, device=dev)
    M.moe_combine(cfg, Yback, pos, w, None, y, stream)
    return plan

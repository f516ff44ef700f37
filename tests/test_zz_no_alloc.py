"""moe_dispatch_static: the dispatch entry point that needs no workspace.

It serves callers that cannot allocate device memory where they dispatch (an
operator host that passes only input and output buffers, or a serving loop
that reserved all of its memory up front).  Its scratch is a fixed array
inside the library, shared by every call and keeping the previous call's
contents, so this test makes two calls in a row -- a large one, then a
smaller one over the stale scratch -- and checks each against moe_dispatch
with a caller workspace: dispatch is integer work, so the results must be
the same bits.  The file sorts last so that a run stopping at the first
failure has run every other test first."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    import sparse_mixture_experts_sum_b300 as pkg
    from sparse_mixture_experts_sum_b300 import build
    build.build()
    pkg.moe.lib()
    return pkg


def _routing(T, E, k, seed):
    """Seeded top-k indices with a skewed expert popularity (capacity binds)
    and a few tokens routed nowhere (-1), as moe_route leaves them."""
    g = torch.Generator().manual_seed(seed)
    p = torch.linspace(3.0, 1.0, E).expand(T, E)
    idx = torch.multinomial(p, k, replacement=False, generator=g).to(torch.int32)
    idx[torch.randperm(T, generator=g)[: max(1, T // 97)]] = -1
    return idx


def _dispatch_both(M, T, d, E, k, cf, seed):
    cfg = M.make_config(T, d, 64, E, k, "swiglu", "bf16", capacity_factor=cf)
    idx = _routing(T, E, k, seed).to(DEV)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16).to(DEV)
    out = []
    for static in (False, True):
        kept = torch.full((E,), -7, dtype=torch.int32, device=DEV)
        offs = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
        pos = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
        Xp = torch.zeros(T * k, d, dtype=torch.bfloat16, device=DEV)
        st = M.moe.stats_buffer()
        if static:
            M.moe.moe_dispatch_static(cfg, idx, x, kept, offs, pos, Xp, st)
        else:
            ws = M.moe.workspace(cfg, training=True)
            M.moe_dispatch(cfg, idx, x, kept, offs, pos, Xp, st, ws)
        torch.cuda.synchronize()
        out.append(dict(kept=kept.cpu(), offsets=offs.cpu(), pos=pos.cpu(), Xp=Xp.cpu(), stats=st.cpu()))
    return out


def test_static_dispatch_matches_workspace_dispatch_twice(M):
    # The dispatch cuts the slots into chunks of 1024 (T*k <= 2^18) or 4096.
    # First call: 300,000 slots, 74 chunks of 4096, 64 experts; second: 48,000
    # slots, 47 chunks of 1024, 300 experts; third: 10,000 slots, 10 chunks,
    # 16 experts -- each later call runs over the scratch the earlier ones
    # left behind.
    for T, d, E, k, cf, seed in [(150000, 128, 64, 2, 1.0, 30), (24000, 256, 300, 2, 1.0, 31),
                                 (5000, 128, 16, 2, 0.8, 32)]:
        ref, got = _dispatch_both(M, T, d, E, k, cf, seed)
        for key in ("kept", "offsets", "pos", "stats"):
            assert torch.equal(got[key], ref[key]), key
        n = int(ref["offsets"][-1])
        assert torch.equal(got["Xp"][:n], ref["Xp"][:n])
        st = M.moe.MoeStats.from_buffer_copy(bytes(ref["stats"].numpy().tobytes()))
        assert st.dropped_slots > 0 and st.kept_slots == n


def test_static_dispatch_rejects_oversize(M):
    # 2^20 slots fit at any E <= 1024; 2^21 slots at E = 1024 do not
    cfg = M.make_config(1 << 20, 64, 64, 1024, 2, "swiglu", "bf16", capacity_factor=1.0)
    with pytest.raises(M.moe.MoeError) as ei:
        M.moe.moe_dispatch_static(cfg, torch.empty(1, dtype=torch.int32, device=DEV),
                                  torch.empty(8, dtype=torch.bfloat16, device=DEV),
                                  torch.empty(1, dtype=torch.int32, device=DEV),
                                  torch.empty(1, dtype=torch.int32, device=DEV),
                                  torch.empty(1, dtype=torch.int32, device=DEV),
                                  torch.empty(8, dtype=torch.bfloat16, device=DEV), None)
    assert ei.value.status == M.moe.MOE_ERR_UNSUPPORTED

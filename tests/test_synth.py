"""Pins of the seeded input generator (no MoE arithmetic lives there)."""

import math

import numpy as np

import torch

import moe_synth as S


def test_splitmix64_published_vector():
    # splitmix64 started from state 0: first three outputs (Vigna's reference
    # implementation)
    outs = [S.mix64_int(i * S.GAMMA) for i in (1, 2, 3)]
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_torch_stream_matches_python_ints():
    for seed, tid in ((0, 1), (4, 11), (2**31 + 5, 1 + 256 * 3)):
        r = S.raw(seed, tid, 1000, 16)
        for i in range(16):
            assert (int(r[i]) & ((1 << 64) - 1)) == S.raw_int(seed, tid, 1000 + i)


def test_slices_are_independent_of_chunking():
    a = S.normal(1, 3, 0, 4096)
    b = torch.cat([S.normal(1, 3, 0, 1000), S.normal(1, 3, 1000, 3096)])
    assert torch.equal(a, b)


def test_distributions():
    z = S.normal(7, 1, 0, 200000)
    assert abs(z.mean().item()) < 0.01 and abs(z.std().item() - 1) < 0.01
    g = S.gumbel(7, 11, 0, 200000)
    assert abs(g.mean().item() - 0.5772156649) < 0.01   # Euler-Mascheroni
    assert abs(g.var().item() - math.pi ** 2 / 6) < 0.03
    u = S.uniform(7, 2, 0, 100000)
    assert u.min().item() > 0 and u.max().item() < 1


def test_bf16_storage_is_round_to_nearest_even():
    v = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20],
                     dtype=torch.float64)
    b = S.store(v, "bf16").to(torch.float64)
    assert b.tolist() == [1.0, 1.0 + 2 ** -6, -1.0, 1.0 + 2 ** -7]


def test_zipf_bias():
    p = S.zipf_pmf(64, 1.1)
    assert abs(p.sum().item() - 1) < 1e-15
    assert abs(p[0].item() - 1 / sum(i ** -1.1 for i in range(1, 65))) < 1e-15
    assert (p[:-1] > p[1:]).all()


def test_stress_workload_bias_is_log_pmf_and_overflows():
    """The large-prefill stress variant takes the Zipf(1.1) bias as ln(pmf):
    ln(1/H) for the first expert, ln(64^-1.1/H) for the last (H = the
    generalised harmonic number over 64 ranks).  Routed by the oracle it
    drops about 3/4 of the slots and leaves most experts below one 128-row
    tile, some with none."""
    import numpy as np
    from oracle import moe_oracle as O
    wl = S.WORKLOADS["large_prefill_3z"]
    t = S.make_inputs(wl, "cpu", parts=["x", "Wr", "expert_bias"])
    H = sum(i ** -1.1 for i in range(1, 65))
    b = t["expert_bias"].double()
    assert abs(b[0].item() + np.log(H)) < 1e-6 and abs(b[63].item() - (-1.1 * np.log(64) - np.log(H))) < 1e-6
    cfg = dict(T=wl.T, d=wl.d, h=wl.h, E=wl.E, k=wl.k, act=wl.act, capacity_factor=1.25, min_capacity=0,
               lam=0.01, has_shared=False)
    r = O.route_and_dispatch(cfg, t["x"], t["Wr"], t["expert_bias"])
    assert 0.70 < r["stats"]["drop_rate"] < 0.80
    assert (r["kept"] < 128).sum() >= 40 and (r["kept"] == 0).any() and (r["kept"] == 640).sum() >= 8


def test_workload_shapes_small():
    wl = S.WORKLOADS["tiny_fp32"]
    x = S.make_inputs(wl)
    assert x["x"].shape == (64, 64) and x["x"].dtype == torch.float32
    assert x["W1"].shape == (4, 128, 64) and x["W2"].shape == (4, 64, 128)
    assert abs(x["W1"].std().item() - 0.02) < 0.002
    again = S.make_inputs(wl)
    assert all(torch.equal(x[k], again[k]) for k in x)


def test_affine_rows_and_their_redraws():
    """x_affine: row t has mean ~b_t and spread ~a_t; a redrawn row keeps
    its offset and scale."""
    wl = S.WORKLOADS["small_prefill"].replace(T=16, d=4096, x_affine=True, dtype="f32")
    x = S.make_inputs(wl, parts=["x"])["x"].double()
    a, b = S._row_affine(wl, 0, wl.T, "cpu")
    assert (a >= 0.5).all() and (a <= 3.0).all() and (b.abs() <= 2.0).all()
    np.testing.assert_allclose(x.mean(1).numpy(), b.numpy(), atol=0.12)
    np.testing.assert_allclose(x.std(1).numpy(), a.numpy(), rtol=0.05)
    x2 = x.clone().float()
    S.redraw_rows(wl, x2, torch.tensor([3, 7]), 1)
    assert not torch.equal(x2[3], x[3].float()) and torch.equal(x2[4], x[4].float())
    assert abs(x2[3].double().mean().item() - b[3].item()) < 0.12
    assert abs(x2[7].double().std().item() - a[7].item()) < 0.05 * a[7].item()

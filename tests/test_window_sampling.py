"""The full-size parity tests' sampling (CPU): the windows cover what the sampling
plan names, and the oracle stepped on windows alone equals the oracle stepped on the
whole vector, restricted to the windows (the step is elementwise)."""
import numpy as np

import oracle
import synth
import gpu_util as gu


def test_windows_cover_edges_halos_and_chunks():
    rng = np.random.default_rng(0)
    ranks = [(r * 1000, (r + 1) * 1000) for r in range(7)]
    wins = gu.sample_windows(0, 6500, ranks, rng, n_chunks=3, chunk=300, edge=50, halo=4)
    covered = np.zeros(6500, bool)
    for a, b in wins:
        assert 0 <= a < b <= 6500
        covered[a:b] = True
    for (a, b), (c, _) in zip(wins, wins[1:]):
        assert b < c, "windows must be disjoint, sorted and not touching"
    for a, b in ranks:
        b = min(b, 6500)
        if a < 6500:
            assert covered[a:a + 50].all() and covered[b - 50:b].all()
            assert covered[max(0, a - 4):a + 4].all()
    assert gu.window_elements(wins) >= 3 * 50 + 2 * 50 * 6


def test_window_oracle_equals_whole_vector_oracle():
    numel, world, rank = 100_003, 4, -1
    spec_w = synth.Spec(seed=3, stream=2, sigma=0.02)
    hp = (1e-3, 0.9, 0.999, 1e-8)
    plan = oracle.plan(numel, world)
    S, P = plan["shard"], plan["padded"]
    wins = gu.sample_windows(0, numel, [(r * S, min((r + 1) * S, numel)) for r in range(world)],
                             np.random.default_rng(1), chunk=4096, edge=512)
    wo = gu.WindowOracle(numel, world, rank, wins, spec_w, hp)
    w = np.zeros(P, np.float32)
    w[:numel] = synth.fill_host(spec_w, 0, numel, synth.OUT_F32)
    m, v, p = np.zeros(P, np.float32), np.zeros(P, np.float32), np.zeros(numel, np.uint16)
    for t in (1, 2, 3):
        full = []
        for k in range(world):
            h = np.zeros(P, np.uint16)
            h[:numel] = synth.fill_host(synth.Spec(seed=3, stream=1, rank=k, step=t,
                                                   sigma=1e-3), 0, numel, synth.OUT_BF16)
            full.append(h)
        oracle.zero_step(numel, world, rank, full, w, m, v, p, *hp, t)
        wo.step(t, [[g[a:b].copy() for g in full] for a, b in wins], threads=4, sub=1000)
    for j, (a, b) in enumerate(wins):
        assert (wo.w[j].view(np.uint32) == w[a:b].view(np.uint32)).all()
        assert (wo.m[j].view(np.uint32) == m[a:b].view(np.uint32)).all()
        assert (wo.v[j].view(np.uint32) == v[a:b].view(np.uint32)).all()
        assert (wo.p[j] == p[a:b]).all()

"""The alpha-beta link model that the ring-vs-tree sweep reports beside its
measured crossover ("从零实现集合通信": the ring takes 2(N-1) steps of T/N,
the tree 2*log2(N) steps of T, and the ring wins on large messages)."""
import math

import pytest

import bench


@pytest.mark.parametrize("N", [3, 4, 5, 8, 16, 64])
def test_crossover_equalises_the_modelled_times(N):
    alpha_us, beta_gbs = 5.0, 45 / 8
    x = bench.alpha_beta_crossover(N, alpha_us, beta_gbs)
    ring, tree = bench.alpha_beta_times(N, x, alpha_us, beta_gbs)
    assert math.isclose(ring, tree, rel_tol=1e-12)
    if x > 0:
        r, t = bench.alpha_beta_times(N, x / 2, alpha_us, beta_gbs)
        assert t < r  # small messages: fewer steps win
    r, t = bench.alpha_beta_times(N, 2 * x + 1e6, alpha_us, beta_gbs)
    assert r < t  # large messages: fewer bytes per step win


def test_crossover_closed_form():
    # N = 4: L = 2, ring 6 steps of T/4, tree 4 steps of T; equal where
    # 2 alpha = 2.5 T / beta, i.e. T = 0.8 alpha beta = 0.8 * 5e-6 * 5.625e9
    assert math.isclose(bench.alpha_beta_crossover(4, 5.0, 45 / 8), 22500.0)


def test_two_ranks_have_no_crossover():
    # N = 2: the ring takes two steps of T/2, the tree two steps of T, so the
    # ring is never slower and there is no crossover
    assert bench.alpha_beta_crossover(2, 5.0, 45 / 8) is None
    r, t = bench.alpha_beta_times(2, 1 << 20, 5.0, 45 / 8)
    assert r < t

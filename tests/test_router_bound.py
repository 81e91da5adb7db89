"""The selection argument of the tensor-core router, checked by brute force on the CPU.

For large batches the library forms approximate logits a[e] on the tensor cores, where each is
within eps[e] of the defined logit l[e]; it takes theta = the k-th largest a - eps, recomputes
the defined logits of the candidates {a + eps >= theta} only, and picks the top-k among them by
(l descending, e ascending). These tests draw logits with many exact and near ties, place the
approximations anywhere in their intervals (the ends included), and check that the candidate
rule always keeps every chosen expert and that no expert left out ties with a chosen one. The
CUDA side follows the same rule (outward rounding keeps it in fp32)."""
import numpy as np
import pytest


def topk_by_rule(l, allowed, k):
    order = sorted((e for e in range(len(l)) if allowed[e]), key=lambda e: (-l[e], e))
    return order[:k]


def candidate_topk(l, a, eps, k):
    # eps covers |a - l| as computed; lo and hi rounded outward, as the kernel rounds them
    eps = np.nextafter(np.maximum(eps, np.abs(a - l)), np.inf)
    lo, hi = np.nextafter(a - eps, -np.inf), np.nextafter(a + eps, np.inf)
    theta = np.sort(lo)[::-1][k - 1]
    cand = hi >= theta
    return topk_by_rule(l, cand, k), cand


def draw_case(rng, E, spread):
    levels = rng.normal(size=max(2, E // spread))
    l = rng.choice(levels, size=E)                 # many exact ties
    l = l + rng.integers(-2, 3, size=E) * 1e-9     # and near ties
    eps = rng.uniform(1e-10, 0.3, size=E)
    u = rng.uniform(-1.0, 1.0, size=E)
    ends = rng.random(E) < 0.3                     # approximations at an interval end
    u[ends] = rng.choice([-1.0, 1.0], size=int(ends.sum()))
    a = l + u * eps
    return l, a, eps


@pytest.mark.parametrize("E,k,spread", [(8, 1, 2), (16, 3, 4), (64, 8, 3), (256, 8, 16),
                                        (40, 40, 5), (1024, 32, 64)])
def test_candidates_keep_the_exact_top_k(E, k, spread):
    rng = np.random.default_rng(E * 1000 + k)
    for _ in range(300 if E <= 256 else 40):
        l, a, eps = draw_case(rng, E, spread)
        got, cand = candidate_topk(l, a, eps, k)
        want = topk_by_rule(l, np.ones(E, bool), k)
        assert got == want
        assert cand.sum() >= k
        # no expert left out ties with or beats the k-th chosen logit
        kth = l[want[-1]]
        assert np.all(l[~cand] < kth)


def test_adversarial_interval_ends():
    # the k-th expert's approximation at the bottom of its interval, the k+1-th at the top
    E, k = 32, 4
    rng = np.random.default_rng(7)
    for _ in range(500):
        l = np.sort(rng.normal(size=E))[::-1].copy()
        eps = np.full(E, rng.uniform(0.01, 1.0))
        a = l.copy()
        a[:k] -= eps[:k]
        a[k:] += eps[k:]
        perm = rng.permutation(E)
        got, _ = candidate_topk(l[perm], a[perm], eps[perm], k)
        assert got == topk_by_rule(l[perm], np.ones(E, bool), k)


def test_all_equal_logits_pick_the_lowest_indices():  # e.g. zero token rows without a bias
    E, k = 64, 8
    l = np.zeros(E)
    eps = np.full(E, 1e-30)
    got, cand = candidate_topk(l, l.copy(), eps, k)
    assert got == list(range(k)) and cand.all()


def test_the_rule_without_the_upper_bound_fails():
    # Candidates taken as {a >= theta} instead of {a + eps >= theta} lose chosen experts: the
    # adversarial draw (the k-th expert at the bottom of its interval) finds it.
    def broken(l, a, eps, k):
        eps = np.nextafter(np.maximum(eps, np.abs(a - l)), np.inf)
        theta = np.sort(np.nextafter(a - eps, -np.inf))[::-1][k - 1]
        return topk_by_rule(l, a >= theta, k)

    E, k = 32, 4
    rng = np.random.default_rng(7)
    misses = 0
    for _ in range(200):
        l = np.sort(rng.normal(size=E))[::-1].copy()
        eps = np.full(E, rng.uniform(0.01, 1.0))
        a = l.copy()
        a[:k] -= eps[:k]
        a[k:] += eps[k:]
        misses += broken(l, a, eps, k) != topk_by_rule(l, np.ones(E, bool), k)
    assert misses > 0

"""Pins of the oracle's sampler (top-k, temperature, top-p, counter-based draws).

The generator is SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) made counter-based:
draw c of seed s is the generator's output for state s + (c + 1) * gamma.  Its
published outputs for a zero seed pin the mixing function; the sampler is pinned by
what the distribution must be (the softmax of the k largest logits at the given
temperature, cut to the top-p prefix), checked on the empirical frequencies of many
draws, by its greedy limit, and by the exact support.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W


def test_splitmix64_reference_outputs():
    # the first two outputs of SplitMix64 started from state 0
    assert O.splitmix64(0, 0) == 0xE220A8397B1DCDAF
    assert O.splitmix64(0, 1) == 0x6E789E6AA1B965F4


def test_uniform_draws_are_uniform_and_uncorrelated():
    n = 100_000
    u = np.array([O.uniform(12345, c) for c in range(n)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 0.003
    counts = np.histogram(u, bins=64, range=(0, 1))[0]
    chi2 = ((counts - n / 64) ** 2 / (n / 64)).sum()
    assert chi2 < 63 + 6 * np.sqrt(2 * 63)          # 63 degrees of freedom, ~6 sigma
    r = np.corrcoef(u[:-1], u[1:])[0, 1]
    assert abs(r) < 5 / np.sqrt(n)
    # another seed gives another sequence
    v = np.array([O.uniform(12346, c) for c in range(1000)])
    assert not np.array_equal(u[:1000], v)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_top1_is_the_greedy_argmax(seed):
    rng = np.random.default_rng(seed)
    lg = rng.normal(size=300).astype(np.float32)
    lg[[7, 200]] = lg.max() + 1.0                      # an exact tie: the lower index wins
    for u in (0.0, 0.3, 0.999999):
        i, _ = O.sample(lg, 1, 0.9, 1.0, u)
        assert i == 7
    lg2 = rng.normal(size=300).astype(np.float32)
    assert O.sample(lg2, 1, 2.0, 0.5, 0.77)[0] == int(np.argmax(lg2))


def _frequencies(lg, k, t, p, n, seed=99):
    counts = np.zeros(len(lg))
    for c in range(n):
        i, _ = O.sample(lg, k, t, p, O.uniform(seed, c))
        counts[i] += 1
    return counts / n


def _expected(lg, k, t, p):
    order = sorted(range(len(lg)), key=lambda i: (-float(lg[i]), i))[:k]
    w = np.exp((lg[order].astype(np.float64) - lg[order[0]]) / t)
    cum = np.cumsum(w)
    m = int(np.argmax(cum >= p * cum[-1])) + 1
    prob = np.zeros(len(lg))
    prob[order[:m]] = w[:m] / cum[m - 1]
    return prob


@pytest.mark.parametrize("k,t,p", [(5, 0.9, 1.0), (8, 2.0, 1.0), (6, 0.9, 0.6), (3, 0.5, 1.0)])
def test_draw_frequencies_match_the_truncated_softmax(k, t, p):
    lg = np.array([0.3, 2.0, -1.0, 1.5, 1.9, 0.0, 2.4, -3.0, 1.0, 0.7], np.float32)
    n = 40_000
    f = _frequencies(lg, k, t, p, n)
    e = _expected(lg, k, t, p)
    assert np.all(f[e == 0] == 0)                       # nothing outside the kept candidates
    sigma = np.sqrt(e * (1 - e) / n)
    assert np.all(np.abs(f - e) <= 5 * sigma + 1e-12), (f, e)


def test_temperature_limits():
    lg = np.array([0.5, 1.0, 0.9, -0.2, 0.95], np.float32)
    for c in range(200):
        assert O.sample(lg, 4, 1e-4, 1.0, O.uniform(5, c))[0] == 1      # cold: the argmax
    f = _frequencies(lg, 4, 1e4, 1.0, 20_000)                          # hot: uniform over the top 4
    assert np.all(np.abs(f[[1, 4, 2, 0]] - 0.25) < 0.02) and f[3] == 0


def test_eos_masked_entry_is_never_drawn():
    lg = np.array([1.0, 5.0, 0.5, 0.2], np.float32)
    lg[1] = -np.inf                                       # the masked id
    for c in range(500):
        assert O.sample(lg, 4, 0.9, 1.0, O.uniform(1, c))[0] != 1


def test_model_sampling_is_seeded_and_top1_is_greedy():
    s = W.TINY
    w = W.model_weights(s)
    e = W.prefill_embeds(s)

    def run(top_k, seed):
        o = O.Oracle(s, w)
        if top_k:
            o.set_sampling(top_k, 0.9, 1.0, seed)
        ids = [o.prefill(embeds=e)[0]]
        for _ in range(s.decode_steps):
            ids.append(o.step(token=ids[-1])[0])
        o.close()
        return ids

    a, b, c = run(50, 7), run(50, 7), run(50, 8)
    assert a == b and a != c
    assert run(1, 7) == run(0, 0)
    with pytest.raises(O.OracleError):
        o = O.Oracle(s, w)
        try:
            o.set_sampling(65, 0.9, 1.0, 0)
        finally:
            o.close()


def test_margin_bounds_the_decisions_sensitivity():
    """Where the reported margin exceeds eps, moving every logit by less than eps / 10
    (the logits' own scale ~1) leaves the drawn index unchanged; ties report 0."""
    rng = np.random.default_rng(11)
    eps = 1e-2
    stable = 0
    for trial in range(400):
        lg = rng.normal(size=200).astype(np.float32)
        u = O.uniform(3, trial)
        k, t, p = int(rng.integers(1, 65)), float(rng.uniform(0.5, 1.5)), float(rng.choice([1.0, 0.9]))
        i, m = O.sample(lg, k, t, p, u)
        if m > eps:
            stable += 1
            for _ in range(3):
                pert = (lg + rng.uniform(-eps / 10, eps / 10, size=lg.shape)).astype(np.float32)
                assert O.sample(pert, k, t, p, u)[0] == i
    assert stable > 100
    lg = np.array([2.0, 1.0, 2.0], np.float32)
    assert O.sample(lg, 3, 1.0, 1.0, 0.1)[1] == 0.0

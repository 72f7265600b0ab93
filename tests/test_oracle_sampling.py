"""Pins of the oracle's sampler (oracle/sampling.py) to things other than
itself: the generator's published known answers, the special cases that
reduce to greedy argmax, and the Gumbel-max identity checked statistically
against softmax(l / T)."""
import os

import numpy as np
import pytest

import synthetic
from oracle import llama as L
from oracle import sampling as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        out = S.philox4x32_10(np.array([v[:4]], np.uint32), np.array(v[4:6], np.uint32))[0]
        assert [int(x) for x in out] == v[6:], r


def test_uniforms_open_interval_and_float32_exact():
    u = S.uniforms(4096, 17, 1234)
    assert np.all((u > 0) & (u < 1))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert len(np.unique(u)) > 4000
    # the counter moves with the token index and the position, the key with the seed
    assert not np.array_equal(u, S.uniforms(4096, 18, 1234))
    assert not np.array_equal(u, S.uniforms(4096, 17, 1235))
    assert abs(u.mean() - 0.5) < 0.03


def test_greedy_special_cases():
    rng = np.random.default_rng(0)
    lg = rng.standard_normal(1000)
    assert S.select(lg, 0.0, 0, 5, 1) == L.argmax_lowest(lg)
    # top-1 keeps only the maximum, whatever the noise
    for pos in range(20):
        assert S.select(lg, 1.0, 1, pos, 9) == L.argmax_lowest(lg)
    # a temperature far below the logit gaps leaves the noise no say
    assert S.select(lg, 1e-9, 0, 3, 1) == L.argmax_lowest(lg)


def test_top_k_boundary_ties_take_lower_indices():
    lg = np.array([0.0, 3.0, 1.0, 3.0, 1.0, 1.0, -2.0])
    assert list(S.candidates(lg, 2)) == [1, 3]
    assert list(S.candidates(lg, 3)) == [1, 2, 3]      # of the three 1.0s, index 2 first
    assert list(S.candidates(lg, 4)) == [1, 2, 3, 4]
    assert list(S.candidates(lg, 0)) == list(range(7))


@pytest.mark.parametrize("T,k", [(1.0, 0), (0.7, 0), (1.3, 3)])
def test_gumbel_max_frequencies_match_softmax(T, k):
    """Draws at many positions (independent uniforms) follow softmax(l/T) over
    the candidate set: each frequency within 5 binomial sigmas."""
    lg = np.array([1.2, -0.3, 0.5, 2.0, 0.0, 1.9, -1.0, 0.4])
    n = 20000
    counts = np.zeros(len(lg))
    idx = S.candidates(lg, k)
    for pos in range(n):
        z = S.perturbed(lg, idx, T, pos, 77)
        counts[idx[np.argmax(z)]] += 1
    p = np.zeros(len(lg))
    e = np.exp(lg[idx] / T - np.max(lg[idx] / T))
    p[idx] = e / e.sum()
    sig = np.sqrt(n * p * (1 - p)) + 1e-9
    assert np.all(np.abs(counts - n * p) <= 5 * sig + 1e-9), (counts / n, p)
    if k:
        assert counts[np.setdiff1d(np.arange(len(lg)), idx)].sum() == 0


def test_generate_stops_at_eos():
    w = synthetic.get_workload("tiny").with_(n_layers=1)
    m = L.Model(w, synthetic.generate_weights(w))
    prompt = synthetic.generate_prompt(w)
    ids, lg = S.generate(m, prompt, 12, temperature=0.8, top_k=20, seed=5)
    assert len(ids) == 12
    eos = int(ids[6])
    first = int(np.flatnonzero(ids == eos)[0])
    ids2, lg2 = S.generate(m, prompt, 12, temperature=0.8, top_k=20, seed=5, eos_id=eos)
    assert len(ids2) == first + 1 and ids2[-1] == eos
    assert np.array_equal(ids2, ids[:first + 1]) and np.array_equal(lg2, lg[:first + 1])
    # greedy through the same entry point equals the greedy oracle
    g, _ = S.generate(m, prompt, 6)
    assert np.array_equal(g, L.greedy(m, prompt, 6)[0])

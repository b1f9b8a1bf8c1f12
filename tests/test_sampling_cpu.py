"""Pins of the oracle's sampling: the counter-based generator against its
published known-answer vectors, and the Gumbel-max rule against the
distribution it must produce."""

import json
import os

import numpy as np

from oracle.sampling import philox4x32_10, uniforms, gumbel, sample

KAT = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")))


def test_philox_known_answers():
    for v in KAT["vectors"]:
        ctr = np.array([int(x, 16) for x in v["ctr"]], dtype=np.uint64)
        key = np.array([int(x, 16) for x in v["key"]], dtype=np.uint64)
        out = philox4x32_10(ctr, key)
        assert [f"{int(x):08x}" for x in out] == v["out"]


def test_uniforms_in_open_interval_and_distinct_streams():
    u = uniforms(7, 3, 41, 2, 4096)
    assert u.dtype == np.float32 and u.min() > 0 and u.max() < 1
    assert abs(u.mean() - 0.5) < 0.02
    assert not np.array_equal(u, uniforms(7, 3, 42, 2, 4096))     # position
    assert not np.array_equal(u, uniforms(7, 4, 41, 2, 4096))     # sequence
    assert not np.array_equal(u, uniforms(7, 3, 41, 3, 4096))     # codebook
    assert not np.array_equal(u, uniforms(8, 3, 41, 2, 4096))     # seed
    np.testing.assert_array_equal(u[:100], uniforms(7, 3, 41, 2, 100))


def test_gumbel_max_draws_from_the_softmax():
    """Over many counters, argmax(l/T + G) follows softmax(l/T) (chi-square)."""
    rng = np.random.default_rng(0)
    logits = rng.standard_normal(6).astype(np.float32)
    T = 0.7
    p = np.exp(logits / T) / np.exp(logits / T).sum()
    n = 20000
    counts = np.zeros(6)
    for s in range(n):
        counts[sample(logits, T, 99, s, 5, 1)] += 1
    chi2 = np.sum((counts - n * p) ** 2 / (n * p))
    assert chi2 < 25.0, (counts / n, p)       # 5 dof: p-value ~ 1e-4


def test_zero_temperature_is_greedy():
    lg = np.array([0.1, 3.0, 2.9, -1.0], np.float32)
    assert sample(lg, 0.0, 1, 2, 3, 4) == 1
    # a very low temperature also picks the max almost surely
    assert sample(lg, 1e-4, 1, 2, 3, 4) == 1
    g = gumbel(5, 0, 0, 0, 8)
    assert np.all(np.isfinite(g))


def test_sampled_decode_is_reproducible_and_teacher_forcing_agrees(micro_path):
    import oracle
    from s2_inputs import random_prompt
    w = oracle.OracleWeights(micro_path, dtype=np.float64)
    p = random_prompt(w.cfg, 19, 5, seed=77)

    def run(sampling):
        o = oracle.DualAROracle(w, paged=True, pool_pages=16, sampling=sampling)
        o.prefill(3, p.tokens, p.codes, p.mask)
        return o, o.decode_frames([3], 6)[0]

    o1, c1 = run((0.9, 0.8, 1234))
    _, c2 = run((0.9, 0.8, 1234))
    _, c3 = run((0.9, 0.8, 1235))
    _, greedy = run(None)
    np.testing.assert_array_equal(c1, c2)
    assert not np.array_equal(c1, c3)
    assert not np.array_equal(c1, greedy)
    tf = o1.teacher_forced(p.tokens, p.codes, p.mask, c1, seq=3)
    np.testing.assert_array_equal(tf["pred"], c1)

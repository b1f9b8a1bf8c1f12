"""Pins of the oracle's sampling: the counter-based generator against its
published known-answer vectors, and the Gumbel-max rule against the
distribution it must produce."""

import json
import os

import numpy as np

from oracle.sampling import philox4x32_10, uniforms, gumbel, sample, nucleus, pick

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


# ---------------------------------------------------------------- top-p and EOS

def test_nucleus_matches_its_definition_by_brute_force():
    """Candidate i is kept exactly when the probability of the candidates
    strictly above it is below top_p (an O(n^2) restatement), ties included."""
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(1, 14))
        v = rng.standard_normal(n) * 2.0
        if rng.random() < 0.4:
            v = np.round(v)                      # ties
        top_p = float(rng.uniform(0.02, 0.999))
        p = np.exp(v - v.max())
        p /= p.sum()
        brute = np.array([p[v > v[i]].sum() < top_p for i in range(n)])
        np.testing.assert_array_equal(nucleus(v, top_p), brute)


def test_nucleus_special_cases():
    v = np.log(np.array([0.5, 0.3, 0.2]))        # probabilities 0.5, 0.3, 0.2
    assert nucleus(v, 1.0).all()
    np.testing.assert_array_equal(nucleus(v, 0.45), [True, False, False])
    np.testing.assert_array_equal(nucleus(v, 0.55), [True, True, False])
    np.testing.assert_array_equal(nucleus(v, 0.75), [True, True, False])
    np.testing.assert_array_equal(nucleus(v, 0.85), [True, True, True])
    # a vanishing top_p keeps only the maximum -- every copy of it
    np.testing.assert_array_equal(nucleus(np.array([1.0, 3.0, 3.0, 2.0]), 1e-9),
                                  [False, True, True, False])


def test_top_p_draws_follow_the_renormalised_nucleus():
    """Gumbel-max restricted to the nucleus samples softmax(l/T) renormalised
    over the kept candidates (chi-square), and never a dropped one."""
    rng = np.random.default_rng(3)
    logits = rng.standard_normal(8).astype(np.float32) * 1.5
    T, top_p = 0.8, 0.7
    v = logits / np.float32(T)
    keep = nucleus(v, top_p)
    p = np.exp(v - v.max()) * keep
    p /= p.sum()
    n = 20000
    counts = np.zeros(8)
    for s in range(n):
        counts[pick(logits, T, top_p, 42, s, 9, 3)] += 1
    assert counts[~keep].sum() == 0
    k = keep.nonzero()[0]
    chi2 = np.sum((counts[k] - n * p[k]) ** 2 / (n * p[k]))
    assert chi2 < 10.0 + 5.0 * len(k), (counts / n, p)   # dof = |k| - 1, generous
    # top_p = 1 and T = 0 reduce to the plain draw and to greedy
    for s in range(50):
        assert pick(logits, T, 1.0, 42, s, 9, 3) == sample(logits, T, 42, s, 9, 3)
    assert pick(logits, 0.0, 0.5, 1, 2, 3, 4) == int(np.argmax(logits))


def test_eos_ends_the_sequence_in_the_oracle(micro_path):
    """With the end-of-speech row in the Slow head's set: the frames before
    the stop are those of the run without it, the stopping frame is the first
    whose EOS logit beats every semantic logit, and -1 follows."""
    import oracle
    from s2_inputs import random_prompt
    w = oracle.OracleWeights(micro_path, dtype=np.float64)
    cfg = w.cfg
    p = random_prompt(cfg, 21, 6, seed=80)
    n = 6
    o = oracle.DualAROracle(w, paged=True, pool_pages=16, record=True)
    o.prefill(0, p.tokens, p.codes, p.mask)
    plain = o.decode_frames([0], n)[0]
    hs = [o.log[f]["h"] for f in range(n)]
    sem_max = [float((w.t["tok_emb"][cfg.sem_begin:] @ h).max()) for h in hs]

    def first_fire(t):
        for f, h in enumerate(hs):
            if float(w.t["tok_emb"][t] @ h) > sem_max[f]:
                return f
        return None
    # a text token that first beats every semantic logit after frame 0, so
    # that frames before the stop can be compared
    cands = [(first_fire(t), t) for t in range(cfg.sem_begin)]
    cands = sorted((f, t) for f, t in cands if f is not None and f >= 1)
    assert cands
    f0, eos = cands[0]
    o2 = oracle.DualAROracle(w, paged=True, pool_pages=16, eos=eos)
    o2.prefill(0, p.tokens, p.codes, p.mask)
    got = o2.decode_frames([0], n)[0]
    np.testing.assert_array_equal(got[:f0], plain[:f0])
    assert (got[f0:] == -1).all()
    assert o2.decode_frames([0], 2)[0].tolist() == [[-1] * cfg.n_codebooks] * 2

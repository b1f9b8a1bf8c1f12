"""End-of-speech stopping and top-p sampling through the C ABI against the
oracle (s2_set_stop, s2_set_top_p).

On the fp32 tiny model the codes -- including the -1 frames after a stop and
the top-p filtered draws -- equal the oracle's.  On the bf16 test model the
same features run on the CUDA-core path (batch 2) and the tensor-core path
(batch 18) and are scored teacher-forced."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from s2_inputs import TINY, MINI_BF16, ensure_weights, random_prompt  # noqa: E402


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def tiny(weights_dir):
    path = ensure_weights(TINY, weights_dir)
    return path, oracle.OracleWeights(path, dtype=np.float32)


@pytest.fixture(scope="module")
def mini(weights_dir):
    path = ensure_weights(MINI_BF16, weights_dir)
    return path, oracle.OracleWeights(path, dtype=np.float32)


def find_eos(w, prompt, n):
    """A text token whose logit first beats every semantic logit on a frame
    after the first (so frames before the stop exist), from a greedy oracle
    run; returns (token, stopping frame)."""
    cfg = w.cfg
    o = oracle.DualAROracle(w, paged=True, pool_pages=64, record=True)
    o.prefill(0, prompt.tokens, prompt.codes, prompt.mask)
    o.decode_frames([0], n)
    hs = [o.log[f]["h"] for f in range(n)]
    sem_max = [float((w.t["tok_emb"][cfg.sem_begin:] @ h).max()) for h in hs]
    best = None
    for t in range(cfg.sem_begin):
        row = w.t["tok_emb"][t]
        f = next((f for f, h in enumerate(hs) if float(row @ h) > sem_max[f]), None)
        if f is not None and f >= 1 and (best is None or f < best[1]):
            best = (t, f)
    return best


def decode(b, path, prompts, n, flags=0, eos=-1, sampling=None, top_p=None, calls=None):
    B = len(prompts)
    T = max(p.T for p in prompts)
    ctx = b.s2_create(path, max_seqs=B, max_batch=B, max_ctx=T + n + 16, max_prompt=T, flags=flags)
    try:
        if sampling:
            b.s2_set_sampling(ctx, *sampling)
        if top_p:
            b.s2_set_top_p(ctx, *top_p)
        b.s2_set_stop(ctx, eos)
        for i, p in enumerate(prompts):
            b.s2_prefill(ctx, i, p.tokens, p.codes, p.mask)
        ids = np.arange(B, dtype=np.int32)
        codes = np.concatenate([b.s2_decode_frames(ctx, ids, k) for k in (calls or [n])], axis=1)
        st = b.s2_stats(ctx)
        assert st["device_error"] == 0
        # a finished sequence can no longer be decoded; the others can
        done = [i for i in range(B) if (codes[i] == -1).any()]
        for i in done:
            with pytest.raises(b.S2Error):
                b.s2_decode_frames(ctx, [i], 1)
            b.s2_release(ctx, i)
        live = [i for i in range(B) if i not in done]
        if live:
            b.s2_decode_frames(ctx, live, 1)
        return codes
    finally:
        b.s2_destroy(ctx)


@pytest.mark.parametrize("flags", [0, 1])     # CUDA graphs, direct launches
def test_tiny_eos_stops_like_the_oracle(b, tiny, flags):
    path, w = tiny
    cfg = TINY
    # prompts for which some text token overtakes the semantic codes within
    # 8 frames (searched once with the oracle)
    prompts = [random_prompt(cfg, 20 + 5 * (s % 3), 5, seed=s) for s in (1108, 1109, 1110)]
    n = 8
    found = None
    for i, p in enumerate(prompts):
        found = find_eos(w, p, n)
        if found:
            break
    assert found, "no stopping token found for the test prompts"
    eos, f_stop = found
    o = oracle.DualAROracle(w, paged=True, pool_pages=64, eos=eos)
    for k, p in enumerate(prompts):
        o.prefill(k, p.tokens, p.codes, p.mask)
    ref = o.decode_frames(list(range(3)), n)
    assert (ref[i, f_stop:] == -1).all() and (ref[i, :f_stop] >= 0).all()
    got = decode(b, path, prompts, n, flags=flags, eos=eos)
    np.testing.assert_array_equal(got, ref)
    # split at the stop (when no row stopped before it): the second call
    # starts with the stopping frame
    if (ref[:, :f_stop] >= 0).all():
        got2 = decode(b, path, prompts, n, flags=flags, eos=eos, calls=[f_stop, n - f_stop])
        np.testing.assert_array_equal(got2, ref)


def test_tiny_top_p_draws_match_the_oracle(b, tiny):
    path, w = tiny
    prompts = [random_prompt(TINY, 25, 6, seed=1200 + i) for i in range(3)]
    samp, tp = (0.9, 0.8, 0xC0FFEE1234), (0.7, 0.85)
    got = decode(b, path, prompts, 6, sampling=samp, top_p=tp)
    o = oracle.DualAROracle(w, paged=True, pool_pages=64, sampling=samp + tp)
    for k, p in enumerate(prompts):
        o.prefill(k, p.tokens, p.codes, p.mask)
    np.testing.assert_array_equal(got, o.decode_frames([0, 1, 2], 6))
    plain = decode(b, path, prompts, 6, sampling=samp)
    assert (got != plain).any()      # the filter changed some draws


def test_tiny_eos_with_top_p_sampling(b, tiny):
    """Stopping inside a top-p sampled decode (EOS is one more candidate of
    the Slow head's draw)."""
    path, w = tiny
    p = random_prompt(TINY, 22, 5, seed=1300)
    found = find_eos(w, p, 8)
    assert found
    eos = found[0]
    samp, tp = (0.5, 0.5, 77), (0.95, 0.9)
    got = decode(b, path, [p], 8, eos=eos, sampling=samp, top_p=tp)
    o = oracle.DualAROracle(w, paged=True, pool_pages=64, sampling=samp + tp, eos=eos)
    o.prefill(0, p.tokens, p.codes, p.mask)
    np.testing.assert_array_equal(got, o.decode_frames([0], 8))


@pytest.mark.parametrize("B", [2, 18])        # CUDA-core GEMV heads, tensor-core heads
def test_mini_top_p_teacher_forced(b, mini, B):
    path, w = mini
    prompts = [random_prompt(MINI_BF16, 30 + 3 * i, 6, seed=1400 + i) for i in range(B)]
    samp, tp = (0.8, 0.9, 99), (0.8, 0.9)
    n = 6
    got = decode(b, path, prompts, n, sampling=samp, top_p=tp)
    assert ((got >= 0) & (got < MINI_BF16.codebook_size)).all()
    o = oracle.DualAROracle(w, paged=False, sampling=samp + tp)
    agree = []
    for i in (0, B - 1):   # the draws' noise is keyed by the sequence id
        p = prompts[i]
        tf = o.teacher_forced(p.tokens, p.codes, p.mask, got[i], seq=i)
        agree.append(float(np.mean(tf["pred"] == got[i])))
    assert min(agree) >= 0.95, agree


@pytest.mark.parametrize("B", [2, 18])
def test_mini_eos_marks_finished_rows(b, mini, B):
    path, w = mini
    prompts = [random_prompt(MINI_BF16, 30 + 3 * i, 6, seed=1500 + i) for i in range(B)]
    found = find_eos(w, prompts[0], 6)
    assert found
    eos, f_stop = found
    got = decode(b, path, prompts, 6, eos=eos)
    for i in range(B):
        stops = np.nonzero((got[i] == -1).all(axis=1))[0]
        if len(stops):
            s0 = stops[0]
            assert (got[i, s0:] == -1).all() and (got[i, :s0] >= 0).all()
    # row 0 stops where the oracle says (bf16 GEMV vs fp32 oracle: allow one
    # frame either side for a near-tie)
    s0 = np.nonzero((got[0] == -1).all(axis=1))[0]
    assert len(s0) and abs(int(s0[0]) - f_stop) <= 1, (s0, f_stop)

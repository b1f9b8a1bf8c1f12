"""Streaming decode (S2_FLAG_STREAM: the full frames of a call in one
persistent launch whose producer warp streams the weights through a
shared-memory ring of bulk copies) through the C ABI.

Its GEMV sums each dot product in another order than the per-frame CUDA
graph, so the two agree to rounding, not bit for bit.  Each case is scored
against the oracle by teacher forcing (>= 99% of the codes, or every
disagreement an oracle near-tie), and against the graph path: codes equal up
to the first frame where the oracle's top-2 margin is a near-tie."""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from s2_inputs import MINI_BF16, S2, ensure_weights, make_workload, random_prompt  # noqa: E402
from parity_util import score  # noqa: E402


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def mini(weights_dir):
    return ensure_weights(MINI_BF16, weights_dir)


@pytest.fixture(scope="module")
def mini_oracle(mini):
    return oracle.OracleWeights(mini, dtype=np.float32)


def decode(b, path, prompts, n, flags, sampling=None, calls=None):
    """Prefill prompts (sequence i = prompt i), decode them together; returns
    (codes [B, n, 10], kernel launches of the decode calls)."""
    B = len(prompts)
    T = max(p.T for p in prompts)
    ctx = b.s2_create(path, max_seqs=B, max_batch=B, max_ctx=T + n + 16, max_prompt=T, flags=flags)
    try:
        if sampling:
            b.s2_set_sampling(ctx, *sampling)
        for i, p in enumerate(prompts):
            b.s2_prefill(ctx, i, p.tokens, p.codes, p.mask)
        l0 = b.s2_stats(ctx)["kernel_launches"]
        parts = [b.s2_decode_frames(ctx, np.arange(B, dtype=np.int32), k) for k in (calls or [n])]
        st = b.s2_stats(ctx)
        assert st["device_error"] == 0
        return np.concatenate(parts, axis=1), st["kernel_launches"] - l0
    finally:
        b.s2_destroy(ctx)


def check_against_oracle(w, prompt, codes, tol=2e-2):
    s = score(oracle.DualAROracle(w, paged=False), prompt, codes)
    dis = s["tf"]["pred"] != codes
    assert s["agree"] >= 0.99 or bool(np.all(s["tf"]["margin"][dis] < 2 * tol)), \
        {k: v for k, v in s.items() if k != "tf"}
    return s


def check_against_graphs(w, prompt, got, ref):
    """Equal codes, or the first differing frame holds an oracle near-tie
    (after which free-running streams diverge)."""
    if np.array_equal(got, ref):
        return
    f = int(np.argmax((got != ref).any(1)))
    tf = oracle.DualAROracle(w, paged=False).teacher_forced(prompt.tokens, prompt.codes, prompt.mask,
                                                           ref[: f + 1])
    k = int(np.argmax(got[f] != ref[f]))
    assert tf["margin"][f, k] < 1e-3, (f, k, float(tf["margin"][f, k]))


@pytest.mark.parametrize("B", [1, 2])
def test_mini_stream_against_oracle_and_graphs(b, mini, mini_oracle, B):
    prompts = [random_prompt(MINI_BF16, 30 + 11 * i, 9 + i, seed=1900 + i) for i in range(B)]
    n = 12
    got, launches = decode(b, mini, prompts, n, b.S2_FLAG_STREAM)
    ref, launches_ref = decode(b, mini, prompts, n, 0)
    # frames 1.. ran in one launch (frame 0 of a fresh prompt is a graph)
    assert launches < launches_ref / 3, (launches, launches_ref)
    for i, p in enumerate(prompts):
        check_against_oracle(mini_oracle, p, got[i])
        check_against_graphs(mini_oracle, p, got[i], ref[i])


def test_mini_stream_split_calls_and_continuing_rows(b, mini, mini_oracle):
    """Calls of 1, 4 and 7 frames continue the same sequences; every call
    after the first runs all its frames in the streaming kernel."""
    prompts = [random_prompt(MINI_BF16, 40, 12, seed=1910), random_prompt(MINI_BF16, 23, 5, seed=1911)]
    got, _ = decode(b, mini, prompts, 12, b.S2_FLAG_STREAM, calls=[1, 4, 7])
    one, _ = decode(b, mini, prompts, 12, b.S2_FLAG_STREAM)
    np.testing.assert_array_equal(got, one)
    for i, p in enumerate(prompts):
        check_against_oracle(mini_oracle, p, got[i])


def test_mini_stream_sampling_matches_graph_draws(b, mini, mini_oracle):
    """Temperature draws (Gumbel noise in the GEMV's arg-max epilogue) with
    the same seed pick the same codes as the graph path unless a sampled
    score is a near-tie."""
    prompts = [random_prompt(MINI_BF16, 35, 7, seed=1920)]
    samp = (0.8, 0.9, 1234)
    got, _ = decode(b, mini, prompts, 9, b.S2_FLAG_STREAM, sampling=samp)
    ref, _ = decode(b, mini, prompts, 9, 0, sampling=samp)
    greedy, _ = decode(b, mini, prompts, 9, b.S2_FLAG_STREAM)
    assert (got != greedy).any()
    assert np.mean(got == ref) >= 0.9, (got, ref)


def test_mini_stream_falls_back_where_it_does_not_run(b, mini):
    """Batch 3 and a bf16 KV cache replay the graphs: same codes as flags 0."""
    prompts = [random_prompt(MINI_BF16, 20 + i, 3, seed=1930 + i) for i in range(3)]
    got, _ = decode(b, mini, prompts, 5, b.S2_FLAG_STREAM)
    ref, _ = decode(b, mini, prompts, 5, 0)
    np.testing.assert_array_equal(got, ref)
    got, _ = decode(b, mini, prompts[:1], 5, b.S2_FLAG_STREAM | b.S2_FLAG_KV_BF16)
    ref, _ = decode(b, mini, prompts[:1], 5, b.S2_FLAG_KV_BF16)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------ full-size S2 model

@pytest.fixture(scope="module")
def s2w(weights_dir):
    if os.environ.get("S2_SKIP_FULL"):
        pytest.skip("full-size model skipped")
    return ensure_weights(S2, weights_dir)


@pytest.mark.slow
def test_s2_stream_batch1_prompt41_60_frames(b, s2w):
    """The bench's workload: 41-token prompt, 60 frames, every frame scored
    against the oracle (teacher forced) and against the graph path."""
    wl = make_workload(1)
    p = wl.prompts[0]
    got, launches = decode(b, s2w, wl.prompts, wl.n_frames, b.S2_FLAG_STREAM)
    ref, launches_ref = decode(b, s2w, wl.prompts, wl.n_frames, 0)
    assert launches < launches_ref / 10, (launches, launches_ref)
    w = oracle.OracleWeights(s2w, dtype=np.float32)
    s = check_against_oracle(w, p, got[0])
    print("S2 stream b1:", {k: v for k, v in s.items() if k != "tf"})
    check_against_graphs(w, p, got[0], ref[0])

"""Persistent decode (S2_FLAG_PERSIST: all full frames of a call in one
cooperative launch) against the per-frame CUDA graphs through the C ABI.

Both paths run the same kernel code with the same arguments and the same
split of every operation over CTAs and warps, so the codes must be identical
-- greedy and sampled, at every batch size, across calls that mix continuing
and fresh sequences.  The graph path itself is held to the oracle by
test_model_gpu.py; here the persistent path is also scored against the
oracle directly (teacher-forced) on the bf16 test model."""

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


def decode(b, path, prompts, n, flags=None, sampling=None, calls=None):
    """Prefill prompts (sequence i = prompt i), decode them together; returns
    (codes [B, n, 10], kernel launches of the decode calls)."""
    B = len(prompts)
    T = max(p.T for p in prompts)
    flags = b.S2_FLAG_PERSIST if flags is None else flags
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


# The persistent kernel runs every GEMV of a frame with one batch instance,
# sized for the Fast AR's first pass (two rows per sequence): B = 1 -> 2-row,
# 2 -> 4-row, 3 -> 8-row; at B = 5 that pass's 10 rows run in two chunks.
@pytest.mark.parametrize("B", [1, 2, 3, 5])
def test_mini_persistent_codes_equal_graphs(b, mini, B):
    prompts = [random_prompt(MINI_BF16, 30 + 11 * i, 9 + i, seed=900 + i) for i in range(B)]
    n = 10
    got, launches = decode(b, mini, prompts, n)
    ref, launches_ref = decode(b, mini, prompts, n, flags=0)
    np.testing.assert_array_equal(got, ref)
    # the persistent kernel ran: frames 1.. are one launch instead of ~100 each
    assert launches < launches_ref / 3, (launches, launches_ref)


def test_mini_persistent_split_calls_and_kv_bf16(b, mini):
    prompts = [random_prompt(MINI_BF16, 40, 12, seed=910), random_prompt(MINI_BF16, 23, 5, seed=911)]
    for flags in (0, b.S2_FLAG_KV_BF16):
        got, _ = decode(b, mini, prompts, 12, flags=flags | b.S2_FLAG_PERSIST, calls=[1, 4, 7])
        ref, _ = decode(b, mini, prompts, 12, flags=flags, calls=[1, 4, 7])
        np.testing.assert_array_equal(got, ref)


def test_mini_persistent_sampling_equals_graphs(b, mini):
    prompts = [random_prompt(MINI_BF16, 35 + i, 7, seed=920 + i) for i in range(3)]
    samp = (0.8, 0.9, 1234)
    got, _ = decode(b, mini, prompts, 9, sampling=samp)
    ref, _ = decode(b, mini, prompts, 9, flags=0, sampling=samp)
    np.testing.assert_array_equal(got, ref)
    greedy, _ = decode(b, mini, prompts, 9)
    assert (got != greedy).any()   # the draws did change codes


def test_mini_persistent_continuous_batching(b, mini):
    """Sequences join and leave between calls; each call's first frame mixes
    continuing and fresh rows (graph path), the rest run persistent."""
    ps = [random_prompt(MINI_BF16, 20 + 9 * i, 4 + i, seed=930 + i) for i in range(4)]

    def run(flags):
        ctx = b.s2_create(mini, max_seqs=4, max_batch=4, max_ctx=128, max_prompt=64, flags=flags)
        out = []
        try:
            for i in (0, 1):
                b.s2_prefill(ctx, i, ps[i].tokens, ps[i].codes, ps[i].mask)
            out.append(b.s2_decode_frames(ctx, [1, 0], 3))
            b.s2_prefill(ctx, 2, ps[2].tokens, ps[2].codes, ps[2].mask)
            out.append(b.s2_decode_frames(ctx, [2, 0, 1], 4))
            b.s2_release(ctx, 0)
            b.s2_prefill(ctx, 3, ps[3].tokens, ps[3].codes, ps[3].mask)
            out.append(b.s2_decode_frames(ctx, [1, 3, 2], 5))
            assert b.s2_stats(ctx)["device_error"] == 0
        finally:
            b.s2_destroy(ctx)
        return out

    for g, r in zip(run(b.S2_FLAG_PERSIST), run(0)):
        np.testing.assert_array_equal(g, r)


def test_mini_persistent_teacher_forced_against_oracle(b, mini):
    w = oracle.OracleWeights(mini, dtype=np.float32)
    p = random_prompt(MINI_BF16, 90, 50, seed=940)
    codes, _ = decode(b, mini, [p], 14)
    s = score(oracle.DualAROracle(w, paged=False), p, codes[0])
    # >= 99% agreement, or every disagreement an oracle near-tie (top-2
    # margin below twice the 2e-2 logit tolerance)
    dis = s["tf"]["pred"] != codes[0]
    assert s["agree"] >= 0.99 or bool(np.all(s["tf"]["margin"][dis] < 4e-2)), \
        {k: v for k, v in s.items() if k != "tf"}


# ------------------------------------------------------------------ full-size S2 model

@pytest.fixture(scope="module")
def s2w(weights_dir):
    if os.environ.get("S2_SKIP_FULL"):
        pytest.skip("full-size model skipped")
    return ensure_weights(S2, weights_dir)


@pytest.mark.slow
@pytest.mark.parametrize("B", [1, 4])
def test_s2_persistent_codes_equal_graphs(b, s2w, B):
    """The bench's 41-token prompt (batch 1) and four different prompts."""
    if B == 1:
        prompts = make_workload(1).prompts
    else:
        prompts = [random_prompt(S2, 41 + 13 * i, 10 + i, seed=950 + i) for i in range(B)]
    n = 12
    got, launches = decode(b, s2w, prompts, n)
    ref, launches_ref = decode(b, s2w, prompts, n, flags=0)
    np.testing.assert_array_equal(got, ref)
    assert launches < launches_ref / 3, (launches, launches_ref)

"""Model-level parity through the C ABI (include/s2.h) against the oracle.

Tolerances (from the benchmark definition): on the tiny fp32 model the codes
are identical to the oracle's free-running decode; on bf16 models, per frame
slow-hidden cosine >= 0.9999, max-abs logit error <= 2e-2 and >= 99% greedy
code agreement, all scored teacher-forced (the oracle replays the GPU's
frames in one causal pass)."""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from s2_inputs import (TINY, MINI_BF16, S2, ensure_weights, make_workload,  # noqa: E402
                       random_prompt, Prompt)
from parity_util import run_library, score, cosine, small_model_agreement_ok  # noqa: E402


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


def oracle_free_run(w, prompts, n, pool_pages=256, perm_seed=None):
    o = oracle.DualAROracle(w, paged=True, pool_pages=pool_pages, perm_seed=perm_seed)
    cached = [o.prefill(i, p.tokens, p.codes, p.mask) for i, p in enumerate(prompts)]
    return o.decode_frames(list(range(len(prompts))), n), cached


# ------------------------------------------------------------------ tiny model: bit-exact codes

@pytest.mark.parametrize("flags", [0, 1, 4])   # graphs+PDL, no graphs, no PDL
def test_tiny_workload_codes_bit_exact(b, tiny, flags):
    path, w = tiny
    wl = make_workload(0)
    r = run_library(b, path, wl.prompts, wl.n_frames, flags=flags)
    ref, _ = oracle_free_run(w, wl.prompts, wl.n_frames)
    np.testing.assert_array_equal(r["codes"], ref)
    assert r["stats"]["device_error"] == 0


def test_tiny_logits_and_hidden_match(b, tiny):
    path, w = tiny
    wl = make_workload(0)
    r = run_library(b, path, wl.prompts, wl.n_frames, debug=True)
    o = oracle.DualAROracle(w, paged=False)
    s = score(o, wl.prompts[0], r["codes"][0], r["logits"][0], r["hidden"][0])
    assert s["agree"] == 1.0
    assert s["max_logit_err"] < 1e-3, s["max_logit_err"]
    assert s["min_cos"] > 0.999999


def test_tiny_debug_sinks_in_host_memory(b, tiny):
    """Host buffers given as debug sinks receive exactly what device sinks
    receive (the library fills them from its own device copies)."""
    path, _ = tiny
    wl = make_workload(0)
    dev = run_library(b, path, wl.prompts, wl.n_frames, debug=True)
    p = wl.prompts[0]
    n = wl.n_frames
    ctx = b.s2_create(path, max_seqs=1, max_batch=1, max_ctx=p.T + n + 16, max_prompt=p.T)
    try:
        dims = b.s2_model_dims(ctx)
        C, d, L = dims["codebook_size"], dims["d"], dims["n_slow"]
        lg = np.zeros((1, n, 10, C), np.float32)
        hd = np.zeros((1, n, d), np.float32)
        ly = np.zeros((n, L, 1, d), np.float32)
        b.s2_set_debug_sinks(ctx, lg, hd, ly, n)
        b.s2_prefill(ctx, 0, p.tokens, p.codes, p.mask)
        codes = b.s2_decode_frames(ctx, np.zeros(1, np.int32), n)
    finally:
        b.s2_destroy(ctx)
    np.testing.assert_array_equal(codes, dev["codes"])
    np.testing.assert_array_equal(lg, dev["logits"])
    np.testing.assert_array_equal(hd, dev["hidden"])
    np.testing.assert_array_equal(ly, dev["layers"])
    assert np.abs(lg).sum() > 0 and np.abs(ly[1:]).sum() > 0


def test_tiny_continuation_equals_one_call(b, tiny):
    path, _ = tiny
    wl = make_workload(0, n_frames=9)
    one = run_library(b, path, wl.prompts, 9)["codes"]
    parts = run_library(b, path, wl.prompts, 9, split_calls=[1, 3, 5])["codes"]
    np.testing.assert_array_equal(one, parts)


def test_tiny_batch_with_radix_prefix_and_scattered_pages(b, tiny):
    """Five sequences, two sharing a 32-position VQ prefix, decoded as one
    batch over scattered pages: codes equal the oracle's, and the second
    sharer reuses two pages."""
    path, w = tiny
    cfg = TINY
    base = random_prompt(cfg, 45, 32, seed=41, masked_positions=np.arange(32))
    other = random_prompt(cfg, 40, 5, seed=42)
    shared = Prompt(np.concatenate([base.tokens[:35], other.tokens[:12]]),
                    np.concatenate([base.codes[:, :35], other.codes[:, :12]], axis=1),
                    np.concatenate([base.mask[:35], other.mask[:12]]))
    prompts = [base, shared, other, random_prompt(cfg, 1, 0, seed=43), random_prompt(cfg, 63, 20, seed=44)]
    n = 6
    r = run_library(b, path, prompts, n, perm_seed=12345, pool_pages=64)
    ref, cached = oracle_free_run(w, prompts, n)
    assert r["cached"] == cached == [0, 32, 0, 0, 0]
    np.testing.assert_array_equal(r["codes"], ref)


@pytest.mark.parametrize("order", [None, [4, 1, 2, 0, 3]])
def test_tiny_batched_prefill_equals_oracle(b, tiny, order):
    """The radix batch prefilled in one s2_prefill_batch call: the second
    sharer still reuses the pages the first inserts in the same call (it
    starts a second group), and the codes equal the oracle's.  In the other
    order the sharer comes first and nothing is reused."""
    path, w = tiny
    cfg = TINY
    base = random_prompt(cfg, 45, 32, seed=41, masked_positions=np.arange(32))
    other = random_prompt(cfg, 40, 5, seed=42)
    shared = Prompt(np.concatenate([base.tokens[:35], other.tokens[:12]]),
                    np.concatenate([base.codes[:, :35], other.codes[:, :12]], axis=1),
                    np.concatenate([base.mask[:35], other.mask[:12]]))
    prompts = [base, shared, other, random_prompt(cfg, 1, 0, seed=43), random_prompt(cfg, 63, 20, seed=44)]
    n = 6
    r = run_library(b, path, prompts, n, perm_seed=12345, pool_pages=64, batch_prefill=True, order=order)
    seq = run_library(b, path, prompts, n, perm_seed=12345, pool_pages=64, order=order)
    assert r["cached"] == seq["cached"]
    assert r["cached"] == ([0, 32, 0, 0, 0] if order is None else [32, 0, 0, 0, 0])
    np.testing.assert_array_equal(r["codes"], seq["codes"])
    if order is None:
        ref, _ = oracle_free_run(w, prompts, n)
        np.testing.assert_array_equal(r["codes"], ref)


@pytest.mark.parametrize("prefill_rows", [0, 4096])
def test_mini_bf16_batched_prefill_tensor_core(b, mini, prefill_rows):
    """Twenty ragged prompts, eight of them sharing a 48-position VQ prefix,
    prefilled in one call on the tensor-core path (segmented RoPE / KV append,
    one tcgen05 attention launch over every prompt's query tiles; passes of at
    most max_prompt rows, or all prompts after the first group in one pass):
    the same cached lengths as separate calls, and the decode scored
    teacher-forced against the oracle."""
    path, w = mini
    cfg = MINI_BF16
    rng = np.random.default_rng(77)
    head = random_prompt(cfg, 48, 48, seed=300, masked_positions=np.arange(48))
    prompts = []
    for i in range(20):
        tail = random_prompt(cfg, int(rng.integers(5, 60)), int(rng.integers(0, 4)), seed=310 + i)
        if i % 5 in (1, 3):
            prompts.append(Prompt(np.concatenate([head.tokens, tail.tokens]),
                                  np.concatenate([head.codes, tail.codes], axis=1),
                                  np.concatenate([head.mask, tail.mask])))
        else:
            prompts.append(tail)
    n = 5
    r = run_library(b, path, prompts, n, perm_seed=5, debug=True, batch_prefill=True, max_batch=20,
                    prefill_rows=prefill_rows)
    seq = run_library(b, path, prompts, n, perm_seed=5)
    assert r["cached"] == seq["cached"]
    assert sorted(set(r["cached"])) == [0, 48]
    o = oracle.DualAROracle(w, paged=False)
    worst = {}
    for i in (0, 1, 3, 8, 19):
        sc = score(o, prompts[i], r["codes"][i], r["logits"][i], r["hidden"][i])
        worst[i] = (sc["max_logit_err"], sc["min_cos"], sc["agree"], sc["near_ties"])
        assert sc["max_logit_err"] <= 2e-2, (i, worst[i])
        assert sc["min_cos"] >= 0.9999, (i, worst[i])
        assert small_model_agreement_ok(sc), (i, worst[i])
    print("batched prefill:", worst)


def test_pool_exhaustion_leaves_state_unchanged(b, tiny):
    path, _ = tiny
    wl = make_workload(0)
    p = wl.prompts[0]
    ctx = b.s2_create(path, max_seqs=2, max_batch=2, kv_pool_pages=2, max_ctx=64, max_prompt=32)
    try:
        b.s2_prefill(ctx, 0, p.tokens, p.codes, p.mask)          # 1 page
        with pytest.raises(b.S2Error) as e:
            b.s2_decode_frames(ctx, [0], 40)                      # needs 3 pages
        assert e.value.status == b.S2_ENOMEM
        c = b.s2_decode_frames(ctx, [0], 4)                       # still primed, fits
        assert c.shape == (1, 4, 10)
        with pytest.raises(b.S2Error) as e:
            b.s2_prefill(ctx, 1, np.concatenate([p.tokens] * 2), None, None)
        assert e.value.status == b.S2_ENOMEM
        assert b.s2_stats(ctx)["pages_used"] == 2
    finally:
        b.s2_destroy(ctx)


def test_invalid_calls_are_rejected(b, tiny):
    path, _ = tiny
    wl = make_workload(0)
    p = wl.prompts[0]
    ctx = b.s2_create(path, max_seqs=3, max_batch=3, max_ctx=64, max_prompt=32)
    try:
        bad = p.codes.copy()
        bad[3, np.nonzero(p.mask)[0][0]] = TINY.codebook_size     # out of range code
        with pytest.raises(b.S2Error) as e:
            b.s2_prefill(ctx, 0, p.tokens, bad, p.mask)
        assert e.value.status == b.S2_EINVAL
        b.s2_prefill(ctx, 0, p.tokens, p.codes, p.mask)
        b.s2_prefill(ctx, 1, p.tokens, p.codes, p.mask)
        b.s2_decode_frames(ctx, [0], 2)
        with pytest.raises(b.S2Error) as e:                        # not prefilled
            b.s2_decode_frames(ctx, [0, 2], 2)
        assert e.value.status == b.S2_ESTATE
        with pytest.raises(b.S2Error) as e:                        # prefill of a live id
            b.s2_prefill(ctx, 0, p.tokens, p.codes, p.mask)
        assert e.value.status == b.S2_ESTATE
        with pytest.raises(b.S2Error) as e:                        # duplicate id
            b.s2_decode_frames(ctx, [1, 1], 2)
        assert e.value.status == b.S2_EINVAL
        b.s2_release(ctx, 0)
        # a one-page prompt cannot reuse its page: at least one position is computed
        assert b.s2_prefill(ctx, 0, p.tokens, p.codes, p.mask) == 0
    finally:
        b.s2_destroy(ctx)


@pytest.mark.parametrize("flags", [0, 1])
def test_tiny_continuous_batching_matches_oracle(b, tiny, flags):
    """Sequences join a running batch between calls: a decode call mixes
    continuing sequences with freshly prefilled ones, in any order."""
    path, w = tiny
    cfg = TINY
    ps = [random_prompt(cfg, 20 + 7 * i, 4 + i, seed=500 + i) for i in range(4)]
    o = oracle.DualAROracle(w, paged=True, pool_pages=64)
    ctx = b.s2_create(path, max_seqs=4, max_batch=4, max_ctx=128, max_prompt=64, flags=flags)
    try:
        for i in (0, 1):
            b.s2_prefill(ctx, i, ps[i].tokens, ps[i].codes, ps[i].mask)
            o.prefill(i, ps[i].tokens, ps[i].codes, ps[i].mask)
        g = b.s2_decode_frames(ctx, [1, 0], 3)
        np.testing.assert_array_equal(g, o.decode_frames([1, 0], 3))
        b.s2_prefill(ctx, 2, ps[2].tokens, ps[2].codes, ps[2].mask)
        o.prefill(2, ps[2].tokens, ps[2].codes, ps[2].mask)
        g = b.s2_decode_frames(ctx, [2, 0, 1], 4)       # 2 is fresh, 0 and 1 continue
        np.testing.assert_array_equal(g, o.decode_frames([2, 0, 1], 4))
        b.s2_release(ctx, 0)
        o.release(0)
        b.s2_prefill(ctx, 3, ps[3].tokens, ps[3].codes, ps[3].mask)
        o.prefill(3, ps[3].tokens, ps[3].codes, ps[3].mask)
        g = b.s2_decode_frames(ctx, [1, 3, 2], 5)
        np.testing.assert_array_equal(g, o.decode_frames([1, 3, 2], 5))
    finally:
        b.s2_destroy(ctx)


def test_radix_lru_eviction_makes_room(b, tiny):
    """Cached pages nobody uses are evicted, oldest first, when the pool is
    short; results do not change."""
    path, w = tiny
    cfg = TINY
    a = random_prompt(cfg, 48, 10, seed=601)
    c2 = random_prompt(cfg, 48, 10, seed=602)
    ctx = b.s2_create(path, max_seqs=2, max_batch=2, kv_pool_pages=5, max_ctx=80, max_prompt=48)
    try:
        b.s2_prefill(ctx, 0, a.tokens, a.codes, a.mask)          # 3 pages, all 3 cached
        ga = b.s2_decode_frames(ctx, [0], 3)
        b.s2_release(ctx, 0)                                       # pages stay in the tree
        assert b.s2_stats(ctx)["radix_pages"] == 3
        assert b.s2_prefill(ctx, 1, c2.tokens, c2.codes, c2.mask) == 0   # needs 3 of 5 pages
        st = b.s2_stats(ctx)
        assert st["evicted_pages"] >= 1
        gc = b.s2_decode_frames(ctx, [1], 3)
        b.s2_release(ctx, 1)
        b.s2_prefill(ctx, 0, a.tokens, a.codes, a.mask)
        np.testing.assert_array_equal(b.s2_decode_frames(ctx, [0], 3), ga)
    finally:
        b.s2_destroy(ctx)
    ref, _ = oracle_free_run(w, [c2], 3)
    np.testing.assert_array_equal(gc, ref)


# ------------------------------------------------------------------ mid-size bf16 model

@pytest.mark.parametrize("flags", [2, 0])     # CUDA-core GEMV prefill, tcgen05 prefill
def test_mini_bf16_teacher_forced(b, mini, flags):
    path, w = mini
    cfg = MINI_BF16
    prompts = [random_prompt(cfg, 100, 60, seed=51)]
    n = 16
    r = run_library(b, path, prompts, n, flags=flags, debug=True)
    o = oracle.DualAROracle(w, paged=False)
    s = score(o, prompts[0], r["codes"][0], r["logits"][0], r["hidden"][0])
    assert s["max_logit_err"] <= 2e-2, s
    assert s["min_cos"] >= 0.9999, s
    assert small_model_agreement_ok(s), {k: v for k, v in s.items() if k != "tf"}


def test_mini_bf16_batch_radix_matches_oracle(b, mini):
    """Batch of 6 over scattered pages, 4 sharing a 48-position VQ prefix."""
    path, w = mini
    cfg = MINI_BF16
    base = random_prompt(cfg, 60, 60, seed=61, masked_positions=np.arange(60))
    prompts = []
    for i in range(4):
        tail = random_prompt(cfg, 9 + 3 * i, 0, seed=70 + i)
        prompts.append(Prompt(np.concatenate([base.tokens[:50], tail.tokens]),
                              np.concatenate([base.codes[:, :50], tail.codes], axis=1),
                              np.concatenate([base.mask[:50], tail.mask])))
    prompts += [random_prompt(cfg, 33, 10, seed=80), random_prompt(cfg, 17, 0, seed=81)]
    n = 8
    r = run_library(b, path, prompts, n, perm_seed=7, debug=True)
    assert r["cached"] == [0, 48, 48, 48, 0, 0]
    o = oracle.DualAROracle(w, paged=False)
    for i, p in enumerate(prompts):
        s = score(o, p, r["codes"][i], r["logits"][i], r["hidden"][i])
        brief = {k: v for k, v in s.items() if k != "tf"}
        assert s["max_logit_err"] <= 2e-2, (i, brief)
        assert s["min_cos"] >= 0.9999, (i, brief)
        assert small_model_agreement_ok(s), (i, brief)


def test_mini_bf16_prefix_hit_equals_cold_on_gpu(b, mini):
    """On the CUDA-core path every row's arithmetic is independent of the
    batch, so a radix hit reproduces a cold prefill's codes exactly."""
    path, _ = mini
    cfg = MINI_BF16
    base = random_prompt(cfg, 70, 64, seed=91, masked_positions=np.arange(64))
    tail = random_prompt(cfg, 20, 0, seed=92)
    second = Prompt(np.concatenate([base.tokens[:66], tail.tokens]),
                    np.concatenate([base.codes[:, :66], tail.codes], axis=1),
                    np.concatenate([base.mask[:66], tail.mask]))
    hot = run_library(b, path, [base, second], 6, flags=2)
    cold = run_library(b, path, [second], 6, flags=2)
    assert hot["cached"][1] == 64
    np.testing.assert_array_equal(hot["codes"][1], cold["codes"][0])


# ------------------------------------------------------------------ full-size S2 model

@pytest.fixture(scope="module")
def s2w(weights_dir):
    if os.environ.get("S2_SKIP_FULL"):
        pytest.skip("full-size model skipped")
    path = ensure_weights(S2, weights_dir)
    return path


@pytest.fixture(scope="module")
def s2_oracle(s2w):
    return oracle.OracleWeights(s2w, dtype=np.float32)


@pytest.mark.slow
@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_s2_batch1_prompt41_60_frames(b, s2w, s2_oracle, kv):
    """Full-size model, 41-token prompt, 60 frames (the bench's workload),
    with the Slow AR KV cache in fp32 (default) or bf16."""
    wl = make_workload(1)
    flags = 0 if kv == "f32" else 64
    r = run_library(b, s2w, wl.prompts, wl.n_frames, debug=True, flags=flags)
    o = oracle.DualAROracle(s2_oracle, paged=False)
    p = wl.prompts[0]
    T = p.T
    frames = [1, wl.n_frames // 2, wl.n_frames - 1]
    rows = [T - 1 + f for f in frames]
    s = score(o, p, r["codes"][0], r["logits"][0], r["hidden"][0])
    tf = o.teacher_forced(p.tokens, p.codes, p.mask, r["codes"][0], capture_rows=rows)
    layer_cos = [[cosine(r["layers"][f, l, 0], tf["layers"][l, j]) for l in range(S2.n_slow)]
                 for j, f in enumerate(frames)]
    brief = {k: v for k, v in s.items() if k != "tf"}
    brief["min_layer_cos"] = float(np.min(layer_cos))
    brief["layer_cos_first_frame"] = [round(c, 7) for c in layer_cos[0][::5]]
    print(f"S2 b1 kv={kv}:", brief)
    assert s["min_cos"] >= 0.9999, brief
    assert np.min(layer_cos) >= 0.9999, brief
    if kv == "f32":
        assert s["max_logit_err"] <= 2e-2, brief
        assert s["agree"] >= 0.99, brief
        # the graph-replayed decode runs the same kernels on the same
        # inputs as the debug run: identical codes, every frame
        r2 = run_library(b, s2w, wl.prompts, wl.n_frames)
        np.testing.assert_array_equal(r2["codes"], r["codes"])


def test_mini_bf16_batched_tensor_core_decode(b, mini):
    """Batch of 20 (>= 16 rows: projections and heads on tcgen05; Fast AR
    pass 1 has 40 rows), ragged prompts, scattered pages."""
    path, w = mini
    cfg = MINI_BF16
    rng = np.random.default_rng(99)
    prompts = [random_prompt(cfg, int(rng.integers(5, 90)), int(rng.integers(0, 5)), seed=200 + i)
               for i in range(20)]
    n = 6
    r = run_library(b, path, prompts, n, perm_seed=3, debug=True)
    o = oracle.DualAROracle(w, paged=False)
    worst = {}
    for i in (0, 7, 13, 19):
        s = score(o, prompts[i], r["codes"][i], r["logits"][i], r["hidden"][i])
        worst[i] = (s["max_logit_err"], s["min_cos"], s["agree"], s["near_ties"])
        assert s["max_logit_err"] <= 2e-2, (i, worst[i])
        assert s["min_cos"] >= 0.9999, (i, worst[i])
        assert small_model_agreement_ok(s), (i, worst[i])
    print("batched tc:", worst)


# ------------------------------------------------------------------ full-size workloads 2-4 (scaled frames)

def _score_sampled(o, prompts, r, idx):
    out = []
    for i in idx:
        s = score(o, prompts[i], r["codes"][i], r["logits"][i], r["hidden"][i])
        out.append((i, s["agree"], s["max_logit_err"], s["min_cos"]))
        assert s["max_logit_err"] <= 2e-2, (i, s)
        assert s["min_cos"] >= 0.9999, (i, s)
    return out


@pytest.mark.slow
def test_s2_voice_clone_prefill_1024(b, s2w, s2_oracle):
    """Workload 2 in full: 900 VQ positions + 124 text tokens prefilled on the
    tensor cores (GEMMs and attention), then all 200 frames, every frame
    teacher-forced against the oracle."""
    wl = make_workload(2)
    assert wl.n_frames == 200
    r = run_library(b, s2w, wl.prompts, wl.n_frames, debug=True, debug_layers=False)
    o = oracle.DualAROracle(s2_oracle, paged=False)
    res = _score_sampled(o, wl.prompts, r, [0])
    print("S2 w2:", res)
    assert res[0][1] >= 0.99


@pytest.mark.slow
def test_s2_batch32_shared_radix_prefix(b, s2w, s2_oracle):
    """Workload 3 in full: 32 sequences on one cached 900-position VQ prefix,
    300 frames each; four sequences (the cold one and three that hit the
    896 cached positions) teacher-forced over every frame."""
    wl = make_workload(3)
    r = run_library(b, s2w, wl.prompts, wl.n_frames, debug=True, pool_pages=wl.pool_pages,
                    debug_layers=False)
    assert r["cached"][0] == 0 and all(c == 896 for c in r["cached"][1:])
    o = oracle.DualAROracle(s2_oracle, paged=False)
    res = _score_sampled(o, wl.prompts, r, [0, 1, 17, 31])
    print("S2 w3:", res)
    assert all(x[1] >= 0.99 for x in res), res


@pytest.mark.slow
def test_s2_batch128_scattered_pages(b, s2w, s2_oracle):
    """Workload 4 shape: 128 x 200-token prompts over a seeded-scattered pool."""
    wl = make_workload(4, n_frames=4)
    r = run_library(b, s2w, wl.prompts, wl.n_frames, debug=True, pool_pages=wl.pool_pages,
                    perm_seed=wl.page_perm_seed, debug_layers=False)
    o = oracle.DualAROracle(s2_oracle, paged=False)
    res = _score_sampled(o, wl.prompts, r, [0, 127])
    print("S2 w4:", res)
    assert np.mean([x[1] for x in res]) >= 0.99


@pytest.mark.slow
def test_s2_batch128_long_context_1700_keys(b, s2w, s2_oracle):
    """The batch-128 workload at its defining context length without its
    1,500 frames: 128 sequences with 1,650-token prompts decode 50 frames over
    the seeded-scattered pool of 128 x ceil(1700/16) = 13,696 pages, so the
    last slow steps attend over 1,698 keys; four sequences teacher-forced
    over every frame."""
    wl = make_workload(4)
    prompts = [random_prompt(S2, 1650, 0, seed=4000 + i) for i in range(128)]
    n = 50
    r = run_library(b, s2w, prompts, n, debug=True, pool_pages=wl.pool_pages, perm_seed=wl.page_perm_seed,
                    max_ctx=1700, debug_layers=False)
    o = oracle.DualAROracle(s2_oracle, paged=False)
    res = _score_sampled(o, prompts, r, [0, 41, 86, 127])
    print("S2 w4 long:", res)
    assert all(x[1] >= 0.99 for x in res), res


# ------------------------------------------------------------------ INT8 per-channel weights

def test_tiny_int8_codes_bit_exact(b, tiny):
    """INT8 weights quantised on the device equal the oracle's quantisation,
    so the tiny model's codes stay identical."""
    path, _ = tiny
    w8 = oracle.OracleWeights(path, dtype=np.float32, quant="int8")
    wl = make_workload(0, n_frames=6)
    r = run_library(b, path, wl.prompts, wl.n_frames, flags=16)
    ref, _ = oracle_free_run(w8, wl.prompts, wl.n_frames)
    np.testing.assert_array_equal(r["codes"], ref)


def test_mini_int8_teacher_forced(b, mini):
    path, _ = mini
    w8 = oracle.OracleWeights(path, dtype=np.float32, quant="int8")
    prompts = [random_prompt(MINI_BF16, 70, 30, seed=301)]
    r = run_library(b, path, prompts, 12, flags=16, debug=True)
    o = oracle.DualAROracle(w8, paged=False)
    s = score(o, prompts[0], r["codes"][0], r["logits"][0], r["hidden"][0])
    assert s["max_logit_err"] <= 2e-2, s
    assert s["min_cos"] >= 0.9999, s
    assert small_model_agreement_ok(s), {k: v for k, v in s.items() if k != "tf"}


@pytest.mark.slow
def test_s2_int8_batch1(b, s2w):
    """Full-size model with INT8 weights against the oracle's INT8 model
    (same quantised weights); the agreement with the bf16 model is printed
    as the fidelity of the 8-bit path."""
    wl = make_workload(1, n_frames=20)
    w8 = oracle.OracleWeights(s2w, dtype=np.float32, quant="int8")
    r = run_library(b, s2w, wl.prompts, wl.n_frames, flags=16, debug=True)
    o = oracle.DualAROracle(w8, paged=False)
    s = score(o, wl.prompts[0], r["codes"][0], r["logits"][0], r["hidden"][0])
    print("S2 int8:", {k: v for k, v in s.items() if k != "tf"})
    assert s["max_logit_err"] <= 2e-2, s
    assert s["min_cos"] >= 0.9999, s
    assert s["agree"] >= 0.99, s


# ------------------------------------------------------------------ temperature sampling

def test_tiny_sampling_reproduces_oracle_draws(b, tiny):
    """Gumbel-max sampling with the counter-based generator: the library's
    draws equal the oracle's on the same seed (fp32 tiny model)."""
    path, w = tiny
    cfg = TINY
    prompts = [random_prompt(cfg, 25, 6, seed=700 + i) for i in range(3)]
    samp = (0.9, 0.7, 0x1234ABCD5678)
    ctx = b.s2_create(path, max_seqs=3, max_batch=3, max_ctx=96, max_prompt=32)
    try:
        b.s2_set_sampling(ctx, *samp)
        for i, p in enumerate(prompts):
            b.s2_prefill(ctx, i, p.tokens, p.codes, p.mask)
        g = np.concatenate([b.s2_decode_frames(ctx, [0, 1, 2], 3),
                            b.s2_decode_frames(ctx, [2, 0, 1], 4)[[1, 2, 0]]], axis=1)
    finally:
        b.s2_destroy(ctx)
    o = oracle.DualAROracle(w, paged=True, pool_pages=64, sampling=samp)
    for i, p in enumerate(prompts):
        o.prefill(i, p.tokens, p.codes, p.mask)
    ref = np.concatenate([o.decode_frames([0, 1, 2], 3), o.decode_frames([2, 0, 1], 4)[[1, 2, 0]]], axis=1)
    np.testing.assert_array_equal(g, ref)
    greedy, _ = oracle_free_run(w, prompts, 7)
    assert not np.array_equal(g, greedy)


def test_mini_sampling_batched_tensor_core_path(b, mini):
    """Sampled decode on the tensor-core batch path scored teacher-forced
    against the oracle's draws for the GPU's own frames."""
    path, w = mini
    prompts = [random_prompt(MINI_BF16, 30 + i, 4, seed=800 + i) for i in range(18)]
    samp = (1.0, 0.8, 77)
    ctx = b.s2_create(path, max_seqs=18, max_batch=18, max_ctx=64, max_prompt=48)
    try:
        b.s2_set_sampling(ctx, *samp)
        for i, p in enumerate(prompts):
            b.s2_prefill(ctx, i, p.tokens, p.codes, p.mask)
        g = b.s2_decode_frames(ctx, list(range(18)), 5)
    finally:
        b.s2_destroy(ctx)
    o = oracle.DualAROracle(w, paged=False, sampling=samp)
    agree = []
    for i in (0, 9, 17):
        tf = o.teacher_forced(prompts[i].tokens, prompts[i].codes, prompts[i].mask, g[i], seq=i)
        agree.append(float(np.mean(tf["pred"] == g[i])))
    assert np.mean(agree) >= 0.98, agree

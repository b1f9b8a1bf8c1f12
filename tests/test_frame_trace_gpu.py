"""The frame timeline (S2_FRAME_TRACE): while a decode frame is enqueued, every
GEMV, tensor-core GEMM, RMSNorm-rows and decode-attention launch gets a slot in
which thread 0 of each CTA stamps the global timer at entry, after the wait on
the previous kernel, at the end of its prologue (main loop) and at exit; after
each decode call the last frame's stamps go to the file.  Measurement only: the
decoded codes must not change, and every stamped CTA's four stamps must be in
order."""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from s2_inputs import MINI_BF16, TINY, ensure_weights, random_prompt  # noqa: E402


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_dual_ar_gb300 import buildlib
    buildlib.build()
    from serving_dual_ar_gb300 import binding
    return binding


def decode(b, path, cfg, trace_file, batch):
    if trace_file:
        os.environ["S2_FRAME_TRACE"] = trace_file
    try:
        ctx = b.s2_create(path, max_seqs=batch, max_batch=batch, max_ctx=128, max_prompt=64)
    finally:
        os.environ.pop("S2_FRAME_TRACE", None)
    try:
        for i in range(batch):
            p = random_prompt(cfg, 20 + i, 4, seed=1300 + i)
            b.s2_prefill(ctx, i, p.tokens, p.codes, p.mask)
        return b.s2_decode_frames(ctx, np.arange(batch, dtype=np.int32), 4)
    finally:
        b.s2_destroy(ctx)


def read_trace(path):
    kinds, rows = {}, {}
    for line in open(path):
        f = line.split()
        if f[0] == "launch":
            kinds[int(f[1])] = " ".join(f[2:])
        else:
            rows.setdefault(int(f[0]), []).append([int(x) for x in f[1:6]])
    return kinds, {k: np.array(v, dtype=np.int64) for k, v in rows.items()}


@pytest.mark.parametrize("model,batch", [("tiny", 1), ("mini", 16)])
def test_frame_trace_is_complete_ordered_and_changes_nothing(b, weights_dir, tmp_path, model, batch):
    """Batch 1 on the tiny model (GEMV path) and batch 16 on the bf16 mini model
    (tensor-core path with RMSNorm-rows launches)."""
    cfg = TINY if model == "tiny" else MINI_BF16
    path = ensure_weights(cfg, weights_dir)
    ref = decode(b, path, cfg, None, batch)
    tf = str(tmp_path / "frame.txt")
    got = decode(b, path, cfg, tf, batch)
    np.testing.assert_array_equal(got, ref)
    kinds, rows = read_trace(tf)
    assert kinds and set(kinds) == set(rows), "every traced launch has stamped CTAs"
    assert any(k.startswith("attn") for k in kinds.values())
    want = "gemv" if model == "tiny" else "tc"
    assert any(k.startswith(want) for k in kinds.values())
    if model == "mini":
        assert any(k.startswith("rms") for k in kinds.values())
    for i, t in rows.items():
        stamps = t[:, 1:5]
        # drop rows an earlier graph left in the slot (far from this launch's entries)
        stamps = stamps[np.abs(stamps[:, 0] - np.median(stamps[:, 0])) < 1_000_000]
        assert len(stamps), i
        assert (np.diff(stamps, axis=1) >= 0).all(), (i, kinds[i])
    # launches of one frame run in order: each one's first exit after the previous one's first entry
    ids = sorted(rows)
    firsts = [int(rows[i][:, 1].min()) for i in ids]
    exits = [int(rows[i][:, 4].max()) for i in ids]
    assert all(exits[k] >= firsts[k - 1] for k in range(1, len(ids)))

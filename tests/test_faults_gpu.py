"""Failure paths on the GPU, made on the host (no GPU fault is provoked).

* S2_FAULT_ALLOC_AT=n: the context's n-th device allocation fails as if the
  device were out of memory.  s2_create must return S2_ENOMEM and give back
  everything it had allocated; a failing debug-sink allocation returns
  S2_ENOMEM and leaves the context working as before.
* S2_FAULT_BARRIER=1: in the persistent decode kernel one CTA skips its
  arrival at the grid barrier before the first attention operation, where no
  copy is in flight, and the barrier's budget is cut to 50 ms.  Every CTA's
  wait must run out and return (no hang), the device error word must read 2
  (a bounded wait gave up), and a new context must decode correctly after it.
"""

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from s2_inputs import MINI_BF16, ensure_weights, random_prompt  # noqa: E402


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


class env_var:
    def __init__(self, name, value):
        self.name, self.value = name, value

    def __enter__(self):
        self.old = os.environ.get(self.name)
        os.environ[self.name] = self.value

    def __exit__(self, *exc):
        if self.old is None:
            del os.environ[self.name]
        else:
            os.environ[self.name] = self.old


def create(b, path, flags=0):
    return b.s2_create(path, max_seqs=2, max_batch=2, max_ctx=128, max_prompt=64, flags=flags)


def creation_allocations(b, path):
    """How many device allocations s2_create makes (weights, KV pool, the
    shared-prefix operand images when that path is on, work buffers, RoPE
    cos and sin): the fault index past which a create succeeds, less one."""
    for n in range(1, 16):
        with env_var("S2_FAULT_ALLOC_AT", str(n)):
            try:
                ctx = create(b, path)
            except b.S2Error as e:
                assert e.status == b.S2_ENOMEM, n
                continue
        b.s2_destroy(ctx)
        return n - 1
    raise AssertionError("s2_create failed at every fault index")


def decode_one(b, ctx, p, n):
    b.s2_prefill(ctx, 0, p.tokens, p.codes, p.mask)
    return b.s2_decode_frames(ctx, np.zeros(1, np.int32), n)


def test_failed_allocation_in_create_returns_enomem_and_frees_everything(b, mini):
    ctx = create(b, mini)          # warm the CUDA context and the weight file cache
    b.s2_destroy(ctx)
    torch.cuda.synchronize()
    n_alloc = creation_allocations(b, mini)
    assert n_alloc >= 5, n_alloc
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for n in range(1, n_alloc + 1):
        with env_var("S2_FAULT_ALLOC_AT", str(n)):
            with pytest.raises(b.S2Error) as ei:
                create(b, mini)
        assert ei.value.status == b.S2_ENOMEM, n
        torch.cuda.synchronize()
        assert abs(torch.cuda.mem_get_info()[0] - free0) <= (4 << 20), n
    ctx = create(b, mini)
    b.s2_destroy(ctx)


def test_failed_debug_sink_allocation_changes_nothing(b, mini):
    p = random_prompt(MINI_BF16, 30, 6, seed=1201)
    ctx = create(b, mini)
    try:
        ref = decode_one(b, ctx, p, 4)
    finally:
        b.s2_destroy(ctx)
    first_after = creation_allocations(b, mini) + 1
    with env_var("S2_FAULT_ALLOC_AT", str(first_after)):   # the first allocation after creation
        ctx = create(b, mini)
    try:
        lg = np.zeros((1, 4, 10, MINI_BF16.codebook_size), np.float32)
        with pytest.raises(b.S2Error) as ei:
            b.s2_set_debug_sinks(ctx, lg, None, None, 4)
        assert ei.value.status == b.S2_ENOMEM
        got = decode_one(b, ctx, p, 4)          # decodes as before, no sink set
        assert not lg.any()
        assert b.s2_stats(ctx)["device_error"] == 0
    finally:
        b.s2_destroy(ctx)
    np.testing.assert_array_equal(got, ref)


def test_persistent_barrier_wait_runs_out_and_returns(b, mini):
    p = random_prompt(MINI_BF16, 30, 6, seed=1202)
    ctx = create(b, mini)
    try:
        ref = decode_one(b, ctx, p, 6)
    finally:
        b.s2_destroy(ctx)
    with env_var("S2_FAULT_BARRIER", "1"):
        ctx = create(b, mini, flags=b.S2_FLAG_PERSIST)
    try:
        decode_one(b, ctx, p, 6)                # frames 1..5 in the persistent kernel
        st = b.s2_stats(ctx)                    # synchronises: every CTA has returned
        assert st["device_error"] == 2, st
    finally:
        b.s2_destroy(ctx)
    ctx = create(b, mini, flags=b.S2_FLAG_PERSIST)
    try:
        again = decode_one(b, ctx, p, 6)
        assert b.s2_stats(ctx)["device_error"] == 0
    finally:
        b.s2_destroy(ctx)
    np.testing.assert_array_equal(again, ref)

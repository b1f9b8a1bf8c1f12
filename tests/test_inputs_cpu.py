"""The five synthetic workloads against the input recipe, on CPU.

Shapes and structure follow the benchmark configurations: the tiny model's
16-position prompt with 8 VQ positions, the 41-token prompt of 60 frames (the
one workload the pages themselves time, "s2pro-native", Where it stands), the
1,024-position voice-clone prompt (900 VQ positions of reference audio, then
text), 32 prompts behind one shared 900-position reference-audio prefix, and
128 independent 200-token prompts in a scattered pool of 128 x 1,700
positions.  At a VQ position the token is the semantic id of the first code.
"""
import numpy as np
import pytest

from oracle.radix import RadixCache, position_keys
from s2_inputs import S2, TINY, make_workload


def _check_prompt(p, cfg):
    T = p.T
    assert p.tokens.dtype == np.int32 and p.codes.shape == (cfg.n_codebooks, T) and p.mask.shape == (T,)
    m = p.mask.astype(bool)
    assert (p.tokens[m] == cfg.sem_begin + p.codes[0, m]).all()
    assert ((p.codes[:, m] >= 0) & (p.codes[:, m] < cfg.codebook_size)).all()
    assert not p.codes[:, ~m].any()
    assert ((p.tokens[~m] >= 0) & (p.tokens[~m] < cfg.sem_begin)).all()


def test_tiny_workload():
    wl = make_workload(0)
    assert wl.model == TINY and wl.batch == 1 and wl.n_frames == 4
    p = wl.prompts[0]
    assert p.T == 16 and int(p.mask.sum()) == 8
    _check_prompt(p, TINY)


def test_batch1_text_prompt():
    wl = make_workload(1)
    assert wl.model == S2 and wl.batch == 1 and wl.n_frames == 60
    p = wl.prompts[0]
    assert p.T == 41 and not p.mask.any()
    _check_prompt(p, S2)


def test_voice_clone_prompt():
    wl = make_workload(2)
    assert wl.batch == 1 and wl.n_frames == 200
    p = wl.prompts[0]
    assert p.T == 1024
    assert p.mask[:900].all() and not p.mask[900:].any()
    _check_prompt(p, S2)


def test_shared_prefix_batch():
    wl = make_workload(3)
    assert wl.batch == 32 and wl.n_frames == 300 and wl.shared_prefix == 900
    first = wl.prompts[0]
    for p in wl.prompts:
        assert p.T == 940
        _check_prompt(p, S2)
        assert (p.tokens[:900] == first.tokens[:900]).all()
        assert (p.codes[:, :900] == first.codes[:, :900]).all() and p.mask[:900].all()
    suffixes = {tuple(p.tokens[900:]) for p in wl.prompts}
    assert len(suffixes) == 32
    # whole pages only: after the first prompt, every other one finds the 56
    # full pages (896 positions) of the shared prefix, not the partial 57th
    rc = RadixCache(16)
    keys0 = position_keys(first.tokens, first.codes, first.mask)
    rc.insert(keys0, list(range(-(-first.T // 16))))
    for p in wl.prompts[1:]:
        keys = position_keys(p.tokens, p.codes, p.mask)
        assert len(rc.match(keys, (p.T - 1) // 16)) == 56


def test_batch128_scattered_pool():
    wl = make_workload(4)
    assert wl.batch == 128 and wl.n_frames == 1500
    assert wl.pool_pages == 128 * 107 == 13_696       # 1,700 positions = 106.25 pages each
    assert wl.page_perm_seed is not None
    for p in wl.prompts:
        assert p.T == 200 and not p.mask.any()
        _check_prompt(p, S2)
    assert len({tuple(p.tokens) for p in wl.prompts}) == 128


@pytest.mark.parametrize("i", range(5))
def test_workloads_are_deterministic(i):
    a, b = make_workload(i), make_workload(i)
    for p, q in zip(a.prompts, b.prompts):
        assert (p.tokens == q.tokens).all() and (p.codes == q.codes).all() and (p.mask == q.mask).all()


@pytest.mark.parametrize("i", range(1, 5))
def test_pool_holds_every_sequence_to_its_last_frame(i):
    wl = make_workload(i)
    need = sum(-(-(p.T + wl.n_frames) // 16) for p in wl.prompts)
    if wl.shared_prefix:
        need -= (wl.batch - 1) * (wl.shared_prefix // 16)
    assert wl.pool_pages >= need

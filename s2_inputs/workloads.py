"""Seeded prompts of the five benchmark workloads.

Each prompt is (tokens int32 [T], codes int32 [n_codebooks, T], mask uint8 [T]).
Column t of ``codes`` is meaningful only where ``mask[t]`` is 1; elsewhere it
is zero.  At a masked (VQ) position the token id is ``sem_begin + codes[0, t]``
(the semantic id of the frame's first code); text positions draw ids
uniformly from the text range [0, sem_begin).  Prompt randomness comes from
``numpy.random.default_rng(100 + i)`` for workload i.
"""

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from .config import ModelConfig, TINY, S2

PAGE = 16


@dataclass
class Prompt:
    tokens: np.ndarray
    codes: np.ndarray
    mask: np.ndarray

    @property
    def T(self):
        return int(self.tokens.shape[0])


@dataclass
class Workload:
    name: str
    model: ModelConfig
    prompts: List[Prompt]
    n_frames: int
    page_size: int = PAGE
    pool_pages: int = 0
    page_perm_seed: Optional[int] = None
    shared_prefix: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return len(self.prompts)


def _vq_prompt(rng, cfg, n_vq, text_tail, vq_codes=None):
    """n_vq masked positions followed by ``text_tail`` text positions."""
    T = n_vq + len(text_tail)
    tokens = np.zeros(T, np.int32)
    codes = np.zeros((cfg.n_codebooks, T), np.int32)
    mask = np.zeros(T, np.uint8)
    if n_vq:
        c = vq_codes if vq_codes is not None else rng.integers(
            0, cfg.codebook_size, (cfg.n_codebooks, n_vq))
        codes[:, :n_vq] = c
        tokens[:n_vq] = cfg.sem_begin + c[0]
        mask[:n_vq] = 1
    tokens[n_vq:] = text_tail
    return Prompt(tokens, codes, mask)


def random_prompt(cfg: ModelConfig, T: int, n_masked: int, seed: int,
                  masked_positions=None):
    """A prompt of T positions with ``n_masked`` VQ positions at random places."""
    rng = np.random.default_rng(seed)
    tokens = rng.integers(0, cfg.sem_begin, T).astype(np.int32)
    codes = np.zeros((cfg.n_codebooks, T), np.int32)
    mask = np.zeros(T, np.uint8)
    if masked_positions is None:
        masked_positions = rng.choice(T, n_masked, replace=False) if n_masked else []
    masked_positions = np.asarray(masked_positions, dtype=np.int64)
    if masked_positions.size:
        c = rng.integers(0, cfg.codebook_size,
                         (cfg.n_codebooks, masked_positions.size))
        codes[:, masked_positions] = c
        tokens[masked_positions] = cfg.sem_begin + c[0]
        mask[masked_positions] = 1
    return Prompt(tokens, codes, mask)


def _pages_for(T, n):
    return -(-(T + n) // PAGE)


def make_workload(i: int, n_frames: Optional[int] = None) -> Workload:
    """Workload i (0..4) of the benchmark definition; ``n_frames`` overrides."""
    rng = np.random.default_rng(100 + i)
    if i == 0:
        cfg = TINY
        # 16 positions, 8 of them VQ-masked, interleaved with text.
        tokens = rng.integers(0, cfg.sem_begin, 16).astype(np.int32)
        pos = rng.choice(16, 8, replace=False)
        codes = np.zeros((cfg.n_codebooks, 16), np.int32)
        codes[:, pos] = rng.integers(0, cfg.codebook_size, (cfg.n_codebooks, 8))
        mask = np.zeros(16, np.uint8)
        mask[pos] = 1
        tokens[pos] = cfg.sem_begin + codes[0, pos]
        n = 4 if n_frames is None else n_frames
        return Workload("tiny_b1_t16_f4", cfg, [Prompt(tokens, codes, mask)], n,
                        pool_pages=8 + _pages_for(16, n))
    if i == 1:
        cfg = S2
        tokens = rng.integers(0, cfg.sem_begin, 41).astype(np.int32)
        p = Prompt(tokens, np.zeros((cfg.n_codebooks, 41), np.int32),
                   np.zeros(41, np.uint8))
        n = 60 if n_frames is None else n_frames
        return Workload("s2_b1_prompt41_f60", cfg, [p], n,
                        pool_pages=8 + _pages_for(41, n))
    if i == 2:
        cfg = S2
        text = rng.integers(0, cfg.sem_begin, 124)
        codes = rng.integers(0, cfg.codebook_size, (cfg.n_codebooks, 900))
        p = _vq_prompt(rng, cfg, 900, text, vq_codes=codes)
        n = 200 if n_frames is None else n_frames
        return Workload("s2_b1_voiceclone1024_f200", cfg, [p], n,
                        pool_pages=8 + _pages_for(1024, n))
    if i == 3:
        cfg = S2
        codes = rng.integers(0, cfg.codebook_size, (cfg.n_codebooks, 900))
        suffixes = rng.integers(0, cfg.sem_begin, (32, 40))
        prompts = [_vq_prompt(rng, cfg, 900, suffixes[b], vq_codes=codes)
                   for b in range(32)]
        n = 300 if n_frames is None else n_frames
        shared = 900 // PAGE
        private = _pages_for(940, n) - shared + 1
        return Workload("s2_b32_radix900_suffix40_f300", cfg, prompts, n,
                        pool_pages=8 + shared + 32 * private, shared_prefix=900)
    if i == 4:
        cfg = S2
        toks = rng.integers(0, cfg.sem_begin, (128, 200)).astype(np.int32)
        prompts = [Prompt(toks[b].copy(),
                          np.zeros((cfg.n_codebooks, 200), np.int32),
                          np.zeros(200, np.uint8)) for b in range(128)]
        n = 1500 if n_frames is None else n_frames
        # a pool sized for 128 x 1,700 tokens in whole pages
        return Workload("s2_b128_prompt200_f1500", cfg, prompts, n,
                        pool_pages=128 * -(-1700 // PAGE), page_perm_seed=104)
    raise ValueError(f"no workload {i}")


WORKLOADS = {i: (lambda i=i: make_workload(i)) for i in range(5)}

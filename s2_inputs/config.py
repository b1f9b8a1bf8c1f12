"""Model shapes of the Dual-AR configurations used by tests and the bench."""

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class ModelConfig:
    """Shape of one Dual-AR model (Slow AR over time, Fast AR over depth).

    ``sem_begin`` is the first semantic-token id; semantic ids run to
    ``vocab - 1`` and number ``codebook_size``.  ``wdtype`` is the stored
    weight type of the file ("f32" or "bf16").
    """

    name: str
    d: int
    n_heads: int
    n_kv: int
    head_dim: int
    ffn: int
    n_slow: int
    n_fast: int
    vocab: int
    sem_begin: int
    n_codebooks: int
    codebook_size: int
    wdtype: str
    seed: int
    eps: float = 1e-6
    rope_theta: float = 1e6
    init_std: float = 0.02

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv * self.head_dim

    def with_(self, **kw):
        return replace(self, **kw)


# Tiny model (fp32, seed 0): 2+2 layers, d=256, 4/2 heads of 64, FFN 768,
# vocab 512 with semantic ids 448..511, 10 codebooks x 64.
TINY = ModelConfig(name="tiny", d=256, n_heads=4, n_kv=2, head_dim=64, ffn=768,
                   n_slow=2, n_fast=2, vocab=512, sem_begin=448,
                   n_codebooks=10, codebook_size=64, wdtype="f32", seed=0)

# Full-size S2-shaped model (bf16, seed 1).
S2 = ModelConfig(name="s2", d=2560, n_heads=32, n_kv=8, head_dim=128, ffn=9728,
                 n_slow=36, n_fast=4, vocab=151936 + 4096, sem_begin=151936,
                 n_codebooks=10, codebook_size=4096, wdtype="bf16", seed=1)

# Micro model for CPU-only oracle pins (fp32, small enough for fp64 brute force).
MICRO = ModelConfig(name="micro", d=64, n_heads=4, n_kv=2, head_dim=16, ffn=128,
                    n_slow=2, n_fast=2, vocab=96, sem_begin=64,
                    n_codebooks=10, codebook_size=32, wdtype="f32", seed=7)

# Mid-size bf16 model with the S2 head size (128) for GPU parity at sizes that
# span several kernel tiles but that the oracle finishes in seconds.
MINI_BF16 = ModelConfig(name="mini_bf16", d=1024, n_heads=8, n_kv=2,
                        head_dim=128, ffn=2816, n_slow=3, n_fast=2,
                        vocab=2048 + 512, sem_begin=2048, n_codebooks=10,
                        codebook_size=512, wdtype="bf16", seed=3)

MODELS = {m.name: m for m in (TINY, S2, MICRO, MINI_BF16)}


def param_counts(cfg: ModelConfig):
    """Parameter counts (elements) of the pieces of a model.

    Returns a dict with the per-layer matrix count, the slow and fast stacks,
    the embeddings and heads, and the total.  Norm gains are counted
    separately because they are negligible in bytes.
    """
    d, F = cfg.d, cfg.ffn
    layer = (cfg.q_dim * d + 2 * cfg.kv_dim * d + d * cfg.q_dim + 3 * F * d)
    layer_gains = 2 * d + 2 * cfg.head_dim
    tok = cfg.vocab * d
    table = cfg.n_codebooks * cfg.codebook_size * d
    out = {
        "layer": layer,
        "slow_layers": cfg.n_slow * layer,
        "fast_layers": cfg.n_fast * layer,
        "tok_emb": tok,
        "vq_emb": table,
        "fast_in_emb": table,
        "fast_head": table,
        "sem_head_slice": cfg.codebook_size * d,
        "fast_head_slice": cfg.codebook_size * d,
        "gains": (cfg.n_slow + cfg.n_fast) * layer_gains + 2 * d,
    }
    out["total"] = (out["slow_layers"] + out["fast_layers"] + tok + 3 * table
                    + out["gains"])
    return out

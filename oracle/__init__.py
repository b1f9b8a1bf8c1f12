"""Dual-AR frame-decode oracle: a plain, slow CPU implementation.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes anything in this package: only ``tests/``, ``__graft_entry__.smoke``
and the CPU-baseline / reference legs of ``bench.py`` use it.  It shares no
code with the CUDA path; both take their seeded inputs from ``s2_inputs``.

Every function cites the passage it follows.  The pages are:
  * "SGLang Day-0 Support for FishAudio S2 Text-to-Speech" (sections
    Architecture, Optimizations with SGLang Omni, Engineering Appendix),
  * "s2pro-native" (sections What happens to a sentence, Where it stands,
    The gate that says no),
  * "Fish Audio Abre Código do S2" (section Por Dentro do Modelo:
    Arquitetura Dual-AR; Streaming de Produção via SGLang).
Where they are silent the reading taken is stated beside the code.
"""

from .model import (DualAROracle, OracleWeights, rms_norm, rope_table,
                    apply_rope, softmax, gqa_attention, swiglu, silu,
                    bf16_round, embed_prompt, feedback_embedding,
                    masked_argmax, ContiguousKV, PagedKV,
                    quantize_rows_int8, dequantize_rows_int8)
from .radix import RadixCache, position_keys

__all__ = [
    "DualAROracle", "OracleWeights", "rms_norm", "rope_table", "apply_rope",
    "softmax", "gqa_attention", "swiglu", "silu", "bf16_round",
    "embed_prompt", "feedback_embedding", "masked_argmax", "ContiguousKV",
    "PagedKV", "RadixCache", "position_keys", "quantize_rows_int8",
    "dequantize_rows_int8",
]

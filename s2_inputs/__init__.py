"""Seeded synthetic inputs shared by the oracle, the tests and the bench.

This module holds data only: model shapes, the random-init weight file
(format, writer, reader) and the seeded prompts of each workload.  It holds
none of the Dual-AR arithmetic; the oracle (``oracle/``) and the CUDA path
(``serving_dual_ar_gb300``) each implement that on their own.

Sources for the shapes: the SGLang S2 page ("Architecture", Stage 2: a Slow AR
over time plus a 4-layer Fast AR emitting 9 residual codebook tokens) and the
Fish Audio S2 release post ("Dual-AR architecture": 10 RVQ codebooks at about
21 Hz, 4B parameters on the time axis and 400M on the depth axis).  The
concrete dimensions are the tiny and S2-shaped configurations of the
benchmark definition (d=2560, 32/8 heads of 128, FFN 9728, 36 + 4 layers,
151,936 text + 4,096 semantic ids, 10 codebooks of 4,096).
"""

from .config import (ModelConfig, TINY, S2, MICRO, MINI_BF16, MODELS,
                     param_counts)
from .weights import (tensor_specs, write_weights, WeightFile,
                      ensure_weights, weights_path)
from .workloads import (Prompt, Workload, make_workload, WORKLOADS,
                        random_prompt)

__all__ = [
    "ModelConfig", "TINY", "S2", "MICRO", "MINI_BF16", "MODELS",
    "param_counts", "tensor_specs", "write_weights", "WeightFile",
    "ensure_weights", "weights_path", "Prompt", "Workload", "make_workload",
    "WORKLOADS", "random_prompt",
]

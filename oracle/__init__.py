"""CPU oracle of the DeepSeekMoE layer forward (fp64, numpy).

Test infrastructure: only tests/, the smoke check and the benchmark's CPU
baseline leg import this package. The CUDA library never does.
"""
from . import moe_oracle  # noqa: F401

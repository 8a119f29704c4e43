"""DeepSeekMoE layer forward for one B300 GPU (sm_103a).

The compute lives in the CUDA library lib/libmoe_b300.so behind the C ABI of
include/moe_b300.h; `binding` marshals torch tensors into it. Importing this
package loads nothing: binding.load() does, and raises if the library is
missing.
"""

__all__ = ["binding", "build", "inputs", "workloads"]

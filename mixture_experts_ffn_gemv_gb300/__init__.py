"""GB300-native MoE FFN layer forward (router, softmax top-k, permute, grouped
SwiGLU experts, weighted unpermute-reduce, shared-expert add) behind a C-ABI
CUDA library.

The compute lives in ``libmoe_ffn_gb300.so`` (hand-written sm_103a kernels);
``binding`` marshals torch tensors into its entry points.  The library is
loaded on first use and its absence is an error: there is no fallback path.
"""
from .inputs import LayerShape, Workload, WORKLOADS, TINY, QWEN3_30B_A3B, DEEPSEEK_V3  # noqa: F401

__all__ = ["LayerShape", "Workload", "WORKLOADS", "TINY", "QWEN3_30B_A3B", "DEEPSEEK_V3"]


def __getattr__(name):
    # the binding (and with it the CUDA library) loads only when asked for
    if name in ("binding", "MoeLayer", "build_library"):
        import importlib
        binding = importlib.import_module(__name__ + ".binding")
        if name == "binding":
            return binding
        return getattr(binding, name)
    raise AttributeError(name)

"""GB300 (sm_103a) FlashAttention-2 forward: a C-ABI CUDA library and its thin binding.

``exact_attention_10_gb300.fa`` holds the ctypes binding of ``include/fa.h``;
importing this package does not load the CUDA library, so the CPU-only parts
(``inputs``, ``accounting``) work on machines without a GPU.  Every compute
call goes to the CUDA kernels; there is no CPU fallback.
"""

__all__ = ["fa", "inputs", "accounting"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)

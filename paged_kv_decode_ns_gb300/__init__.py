"""GB300-native paged-KV attention: the data-parallel hot path of a
nanoserve-style LLM server (KV append, split-KV paged decode with online
softmax, chunked prefill), as hand-written sm_103a CUDA kernels behind a C
ABI (``include/ns_paged.h``).

``binding`` holds the Python names of the C entry points; ``workloads``
builds seeded synthetic inputs.  Importing the package loads nothing: the
shared library is opened on the first call into ``binding``.
"""

__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)

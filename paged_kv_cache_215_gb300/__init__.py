"""GB300-native paged KV-cache decode attention.

``paged_kv_cache_215_gb300.pkv`` is the binding of the CUDA library (built by
``paged_kv_cache_215_gb300.build.build()``); ``workloads`` draws seeded inputs.
The binding is imported on first use so that the input generator works on a
machine without the library; using the binding without the library raises.
"""
import importlib

__all__ = ["pkv", "workloads", "build", "dp"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)

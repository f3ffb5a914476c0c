"""GB300-native MLA verify attention (absorbed and materialised branches).

The compute lives in libmla.so (CUDA for sm_103a behind a C ABI declared in
include/mla.h); ``binding`` forwards to it with the same function names.
Importing this package does not load the library; the first call does, and
raises if it has not been built.
"""

import importlib

__all__ = [
    "mla_max_absorbed_queries", "mla_max_absorbed_queries_batch", "mla_select_branch",
    "mla_workspace_bytes", "mla_verify_attention", "make_geometry", "MlaError",
]


def __getattr__(name):
    if name in __all__ or name in ("lib", "status_string", "mla_last_error"):
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)

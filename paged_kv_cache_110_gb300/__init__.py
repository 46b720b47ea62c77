"""GB300-native attention over a block-paged KV cache.

The product is ``libpa.so`` (CUDA kernels for sm_103a behind the C ABI in
``include/pa.h``) and its thin Python binding, ``paged_kv_cache_110_gb300.binding``
(imported explicitly; it raises if the library has not been built).
``workloads`` draws seeded synthetic inputs.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "build"]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)

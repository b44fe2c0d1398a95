"""GB300 (sm_103a) query-centric KV-cache fusion for RAG prefill.

`qcf` holds the binding of the C ABI (include/qcf.h), `model` the device model,
chunk store and request wrappers.  The compiled library (libqcf.so, built by
`build.py`) is loaded on first use; without it every call raises.
"""
from ._lib import LIB_PATH, QcfError  # noqa: F401

__all__ = ["LIB_PATH", "QcfError"]

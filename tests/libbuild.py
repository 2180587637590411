"""Test helper: make sure libpagedkv.so exists (nvcc cross-compiles without a GPU)."""
import os

from paged_kv_cache_146_gb300 import _native, build


def ensure_built():
    srcs = [os.path.join(build.CSRC, s) for s in os.listdir(build.CSRC)]
    srcs.append(os.path.join(build.INCLUDE, "pagedkv.h"))
    newest = max(os.path.getmtime(s) for s in srcs)
    if not os.path.exists(_native.LIB_PATH) or os.path.getmtime(_native.LIB_PATH) < newest:
        build.build()
    return _native.lib()

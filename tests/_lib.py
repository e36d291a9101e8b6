"""Test helper: make sure libzl.so exists (build it in-tree when it does not)."""
import os

from coalesced_packed_attention_gb300 import build as _build
from coalesced_packed_attention_gb300 import zl


def ensure_library():
    if not os.path.exists(zl.LIB_PATH):
        _build.build()
    return zl.load_library()

"""Shared test helper: make sure libpkv.so is built (here or on a GPU machine)."""

import os

from paged_kv_cache_56_gb300 import build as _build, pkv


def ensure_built():
    if not os.path.exists(pkv.LIB_PATH) or any(
            os.path.getmtime(p) > os.path.getmtime(pkv.LIB_PATH) for p in _build._sources() + _build._headers()):
        _build.build()
    return pkv.lib()

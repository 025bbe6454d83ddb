"""The C-ABI library loads and exports every function include/pa.h declares."""

import ctypes
import os
import re

from paged_kv_cache_40_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = f.read()
    return re.findall(r"^PA_API\s+[\w\s\*]+?\b(pa_\w+)\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for must in ("pa_append_kv", "pa_copy_blocks", "pa_decode_attention",
                 "pa_decode_workspace_bytes", "pa_alloc_create", "pa_alloc_append_slot",
                 "pa_alloc_free_seq", "pa_alloc_fork", "pa_alloc_export_state"):
        assert must in names


def test_every_declared_symbol_is_exported(libpa):
    lib = ctypes.CDLL(_lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(_lib.SIGNATURES), "binding signatures out of date"


def test_only_the_api_is_exported(libpa):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_functions())


def test_version_and_status_strings(libpa):
    lib = libpa.lib()
    assert lib.pa_version() == 200
    assert lib.pa_status_string(2) == b"PA_ERR_OUT_OF_BLOCKS"
    assert lib.pa_status_string(6) == b"PA_ERR_TIMEOUT"

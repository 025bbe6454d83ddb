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
    assert lib.pa_version() == 300
    assert lib.pa_status_string(2) == b"PA_ERR_OUT_OF_BLOCKS"
    assert lib.pa_status_string(6) == b"PA_ERR_TIMEOUT"


def _declarations():
    """{name: (return type, [parameter types])} of every PA_API function,
    types as written in the header (whitespace normalised, names dropped)."""
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = re.sub(r"/\*.*?\*/", " ", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"PA_API\s+([\w\s\*]+?)\b(pa_\w+)\((.*?)\);", text, flags=re.S):
        ret, name, params = m.group(1), m.group(2), " ".join(m.group(3).split())
        types = []
        if params and params != "void":
            for p in params.split(","):
                p = p.strip()
                # drop the parameter name (the last identifier, after any '*')
                t = re.sub(r"\b\w+$", "", p).strip()
                types.append(" ".join(t.replace("*", " * ").split()))
        out[name] = (" ".join(ret.replace("*", " * ").split()), types)
    return out


def _kind(c_type: str) -> str:
    """The ctypes kind a C parameter type calls for."""
    if "*" in c_type:
        return "pointer"
    base = c_type.replace("const", "").strip()
    # on LP64 ctypes has one type for size_t and uint64_t (c_ulong)
    return {"int": "int32", "int32_t": "int32", "int64_t": "int64", "uint64_t": "size",
            "size_t": "size",
            "float": "float", "pa_status": "int32", "pa_stream_t": "pointer",
            "pa_allocator": "pointer"}.get(base, "unknown:" + base)


def _ctypes_kind(t) -> str:
    if t in (ctypes.c_void_p, ctypes.c_char_p) or isinstance(t, type(ctypes.POINTER(ctypes.c_int))):
        return "pointer"
    return {ctypes.c_int: "int32", ctypes.c_int32: "int32", ctypes.c_int64: "int64",
            ctypes.c_uint64: "size", ctypes.c_size_t: "size",
            ctypes.c_float: "float"}.get(t, "unknown")


def test_binding_signatures_match_the_header_argument_by_argument():
    """Every argument of every declaration has a ctypes type of the same kind
    (32/64-bit integer, size, float, pointer) at the same position: a
    binding that drifted from the header would pass garbage to a kernel."""
    decls = _declarations()
    assert set(decls) == set(_lib.SIGNATURES)
    for name, (ret, params) in decls.items():
        restype, argtypes = _lib.SIGNATURES[name]
        kinds = [_kind(p) for p in params]
        assert not [k for k in kinds if k.startswith("unknown")], (name, params)
        assert kinds == [_ctypes_kind(a) for a in argtypes], (name, params)
        assert _kind(ret) == _ctypes_kind(restype) or (ret.startswith("void") and restype is None), \
            (name, ret)

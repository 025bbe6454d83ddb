"""ctypes loader for libpa.so and the C signatures of include/pa.h.

Loading never falls back: if the library is missing or lacks a symbol the
header declares, the import of the binding fails with a message that says how
to build it.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK = 0
STATUS_NAMES = {
    0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_OUT_OF_BLOCKS",
    3: "PA_ERR_BAD_BLOCK_ID", 4: "PA_ERR_UNSUPPORTED", 5: "PA_ERR_CUDA",
    6: "PA_ERR_TIMEOUT",
}
PA_DEVERR_BAD_BLOCK = 1
PA_DEVERR_BAD_SLOT = 2
PA_DEVERR_BAD_LEN = 4
PA_DEVERR_TIMEOUT = 8


class PaError(RuntimeError):
    """A libpa call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{self.status_name}: {message}")


class OutOfBlocksError(PaError):
    pass


class AllocStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "num_blocks", "free_blocks", "used_blocks", "shared_blocks",
        "cow_copies", "alloc_failures", "total_refs", "num_seqs")]


_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f32 = ctypes.c_float
_pi32 = ctypes.POINTER(ctypes.c_int32)
_pi64 = ctypes.POINTER(ctypes.c_int64)
_pint = ctypes.POINTER(ctypes.c_int)

SIGNATURES = {
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_version": (_i32, []),
    "pa_device_error": (_i32, [_vp, _pi32]),
    "pa_set_wait_limit_ns": (_i32, [ctypes.c_uint64]),
    "pa_kernel_launches": (ctypes.c_uint64, []),
    "pa_append_kv": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _vp]),
    "pa_copy_blocks": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _vp]),
    "pa_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_decode_workspace_init": (_i32, [_vp, _sz, _i32, _i32, _vp]),
    "pa_decode_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                   _i32, _i32, _i64, _f32, _vp, _vp, _sz, _i32, _vp]),
    "pa_decode_append_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                          _i32, _i32, _i32, _i32, _i32, _i64, _f32, _vp, _vp,
                                          _sz, _i32, _vp]),
    "pa_decode_attention_fixed_scratch": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                                 _i32, _i32, _i32, _i64, _f32, _vp, _i32, _vp]),
    "pa_append_kv_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                _i64, _vp]),
    "pa_copy_blocks_fp8": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _vp]),
    "pa_decode_attention_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                       _i32, _i32, _i32, _i64, _f32, _vp, _vp, _sz, _i32, _vp]),
    "pa_decode_shared_prefix_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_decode_attention_shared_prefix": (_i32, [_vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32,
                                                 _i32, _i32, _i32, _i32, _i32, _i64, _f32, _vp,
                                                 _vp, _sz, _vp]),
    "pa_alloc_create": (_i32, [_i32, _i32, _pi32, ctypes.POINTER(_vp)]),
    "pa_alloc_destroy": (None, [_vp]),
    "pa_alloc_add_seq": (_i32, [_vp, _i64, _i64]),
    "pa_alloc_fork": (_i32, [_vp, _i64, _i64]),
    "pa_alloc_append_slot": (_i32, [_vp, _i64, _pi32, _pi32, _pi32]),
    # the per-step calls take their arrays as plain addresses (numpy buffers)
    "pa_alloc_append_slots": (_i32, [_vp, _vp, _i32, _vp, _vp, _pint, _pint]),
    "pa_alloc_free_seq": (_i32, [_vp, _i64]),
    "pa_alloc_get_table": (_i32, [_vp, _i64, _pi32, _i32, _pint]),
    "pa_alloc_seq_len": (_i32, [_vp, _i64, _pi64]),
    "pa_alloc_build_tables": (_i32, [_vp, _vp, _i32, _i32, ctypes.c_int32, _vp, _vp]),
    "pa_alloc_plan_step": (_i32, [_vp, _vp, _i32, _i32, ctypes.c_int32, _vp, _vp, _pint, _vp,
                                  _vp]),
    "pa_decode_step": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _pint, _vp, _vp, _vp,
                              _vp, _vp, _i32, _i32, _i32, _i32, _i64, ctypes.c_float, _vp, _vp,
                              _sz, _i32, _vp]),
    "pa_decode_step_fp8": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _pint, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64,
                                  ctypes.c_float, _vp, _vp, _sz, _i32, _vp]),
    "pa_alloc_shared_prefix": (_i32, [_vp, _vp, _i32, _vp, _i32, _pint]),
    "pa_alloc_stats": (_i32, [_vp, ctypes.POINTER(AllocStats)]),
    "pa_alloc_export_state": (_i32, [_vp, _pi32, _pint, _pi32]),
    "pa_alloc_add_host_pool": (_i32, [_vp, _i32, _pi32]),
    "pa_alloc_swap_out": (_i32, [_vp, _i64, _pi32, _i32, _pint]),
    "pa_alloc_swap_in": (_i32, [_vp, _i64, _pi32, _i32, _pint]),
    "pa_alloc_export_host_state": (_i32, [_vp, _pi32, _pint, _pi64]),
    "pa_swap_blocks": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _i32, _i64, _vp, _i32, _i32, _vp]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libpa.so once, with every declared signature attached."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "or `python paged_kv_cache_40_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)  # AttributeError if a declared symbol is missing
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int) -> None:
    """Raise PaError (with the thread's last message) for a non-OK status."""
    if status == PA_OK:
        return
    msg = load().pa_last_error().decode(errors="replace")
    if status == 2:
        raise OutOfBlocksError(status, msg)
    raise PaError(status, msg)

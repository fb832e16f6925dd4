"""ctypes declarations of include/sdm.h (the library's only interface)."""

from __future__ import annotations

import ctypes
import os

from ._build import LIB

c_i32, c_i64, c_p, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t

SDM_OK = 0
SDM_F32, SDM_BF16 = 0, 1
SDM_DEV_BAD_SLOT = 0x1

# every symbol include/sdm.h declares
EXPORTS = ("sdm_workspace_bytes", "sdm_workspace_init", "sdm_phase1", "sdm_dw", "sdm_forward_chunks",
           "sdm_phase1_saving", "sdm_dw_saving", "sdm_forward_chunks_saving", "sdm_forward_chunks_noalloc", "sdm_read", "sdm_pa", "sdm_gwr", "sdm_gds",
           "sdm_device_status",
           "sdm_status_string")
NOALLOC_SCRATCH_BYTES = 16 << 20


class Shape(ctypes.Structure):
    _fields_ = [("P", c_i32), ("C", c_i32), ("W", c_i32), ("R", c_i32), ("hd", c_i32), ("valid_last", c_i32),
                ("steps", c_i64), ("S", c_i64), ("val_dtype", c_i32), ("dv_dtype", c_i32), ("bank_dtype", c_i32),
                ("gate_per_entry", c_i32), ("dw_log_buckets", c_i32), ("p1_warps", c_i32)]


P1_FIELDS = ("log_k", "rex", "cpe", "k_eff", "is_last", "is_only", "pos_k", "log_q", "q_w", "pos_q", "q_last",
             "q_only", "A", "QK", "sorted_k", "sorted_q", "repeats", "ngroups", "stats")


class P1Out(ctypes.Structure):
    _fields_ = [(f, c_p) for f in P1_FIELDS]


_lib = None


def load(path: str = LIB):
    """Load the CUDA library. Raises if it has not been built: there is no other code path."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsdm_gb300.so is missing ({path}); build it with sparse_slot_memory_gb300.build()")
    lib = ctypes.CDLL(path)
    sp = ctypes.POINTER(Shape)
    op = ctypes.POINTER(P1Out)
    lib.sdm_workspace_bytes.restype = c_sz
    lib.sdm_workspace_bytes.argtypes = [sp]
    lib.sdm_workspace_init.restype = c_i32
    lib.sdm_workspace_init.argtypes = [c_p, c_sz, c_p]
    lib.sdm_phase1.restype = c_i32
    lib.sdm_phase1.argtypes = [sp, c_p, c_p, c_p, c_p, c_p, op, c_i64, c_i64, c_p, c_sz, c_p]
    lib.sdm_dw.restype = c_i32
    lib.sdm_dw.argtypes = [sp, c_p, c_p, c_i64, c_i64, c_p, c_sz, c_p]
    lib.sdm_forward_chunks.restype = c_i32
    lib.sdm_forward_chunks.argtypes = [sp, c_p, c_p, c_p, c_p, c_p, c_p, c_p, op, c_i64, c_i64, c_p, c_sz, c_p]
    lib.sdm_phase1_saving.restype = c_i32
    lib.sdm_phase1_saving.argtypes = [sp, c_p, c_p, c_p, c_p, c_p, op, c_i64, c_i64, c_p, c_sz, c_p]
    lib.sdm_dw_saving.restype = c_i32
    lib.sdm_dw_saving.argtypes = [sp, c_p, c_p, c_p, c_i64, c_i64, c_p, c_sz, c_p]
    lib.sdm_forward_chunks_saving.restype = c_i32
    lib.sdm_forward_chunks_saving.argtypes = [sp, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, op, c_i64, c_i64, c_p, c_sz,
                                              c_p]
    lib.sdm_forward_chunks_noalloc.restype = c_i32
    lib.sdm_forward_chunks_noalloc.argtypes = [sp, c_p, c_p, c_p, c_p, c_p, c_p, c_p, op, c_i64, c_i64, c_p, c_p]
    lib.sdm_pa.restype = c_i32
    lib.sdm_pa.argtypes = [sp, c_i32] + [c_p] * 12 + [c_i64, c_i64, c_p, c_p]
    lib.sdm_read.restype = c_i32
    lib.sdm_read.argtypes = [sp] + [c_p] * 4 + [c_i64, c_i64, c_p, c_p]
    lib.sdm_gwr.restype = c_i32
    lib.sdm_gwr.argtypes = [sp, c_i32] + [c_p] * 6 + [c_i64, c_i64, c_p, c_p]
    lib.sdm_gds.restype = c_i32
    lib.sdm_gds.argtypes = [sp, c_i32] + [c_p] * 8 + [c_i64, c_i64, c_p, c_p]
    lib.sdm_device_status.restype = c_i32
    lib.sdm_device_status.argtypes = [c_p, ctypes.POINTER(c_i32), c_i32, c_p]
    lib.sdm_status_string.restype = ctypes.c_char_p
    lib.sdm_status_string.argtypes = [c_i32]
    _lib = lib
    return lib

"""ctypes declarations of the C ABI in include/sdm.h (argument marshalling only)."""

from __future__ import annotations

import ctypes
import os

from . import build as _build

MAX_FACTORS = 4
MAX_K = 128
MAX_CANDIDATES = 1024
MAX_CHUNK = 256
ABI_VERSION = 4

SDM_OK, SDM_ERR_INVALID_ARG, SDM_ERR_UNSUPPORTED, SDM_ERR_ALIAS, SDM_ERR_WORKSPACE, \
    SDM_ERR_CUDA, SDM_ERR_DEVICE = range(7)
SDM_F32, SDM_BF16, SDM_F16 = 0, 1, 2
KERNEL_KINDS = ("bank_copy", "score", "select", "plan_sort", "plan_link", "write_read", "decode",
                "bwd_flags", "bwd_sweep", "bwd_reduce", "bwd_subkeys", "layer_gates", "layer_gemm", "layer_grad")

# Every function include/sdm.h declares, in header order.
EXPORTS = (
    "sdm_write_read_workspace_size", "sdm_decode_workspace_size", "sdm_write_read",
    "sdm_write_read_static", "sdm_snapshot_bytes", "sdm_write_read_train",
    "sdm_write_read_backward_workspace_size", "sdm_write_read_backward", "sdm_layer_workspace_size",
    "sdm_layer_forward", "sdm_layer_forward_train", "sdm_layer_backward_workspace_size", "sdm_layer_backward",
    "sdm_decode_step", "sdm_last_device_error", "sdm_status_string", "sdm_last_error_message",
    "sdm_abi_version", "sdm_launch_count", "sdm_profile_begin", "sdm_profile_end",
    "sdm_kernel_name", "sdm_test_stall_decode_copy",
    "sdm_test_force_write_read_layout", "sdm_test_force_simt_scorer", "sdm_test_factor_scores",
)
STATIC_SCRATCH_BYTES = 16 << 20


class SdmShape(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
        ("d_sub", ctypes.c_int64), ("d_v", ctypes.c_int64),
        ("F", ctypes.c_int32), ("factor_dims", ctypes.c_int32 * MAX_FACTORS),
        ("W", ctypes.c_int32), ("R", ctypes.c_int32), ("chunk_size", ctypes.c_int32),
        ("act_dtype", ctypes.c_int32), ("bank_dtype", ctypes.c_int32),
    ]


class SdmLayerSaved(ctypes.Structure):
    _fields_ = [("q_w", ctypes.c_void_p), ("q_r", ctypes.c_void_p), ("k_val", ctypes.c_void_p),
                ("gates", ctypes.c_void_p), ("y", ctypes.c_void_p), ("idx_w", ctypes.c_void_p),
                ("wt_w", ctypes.c_void_p), ("idx_r", ctypes.c_void_p), ("wt_r", ctypes.c_void_p),
                ("snapshot", ctypes.c_void_p), ("snapshot_bytes", ctypes.c_size_t), ("snapshot_dtype", ctypes.c_int32)]


class SdmLayerGrads(ctypes.Structure):
    _fields_ = [("dx", ctypes.c_void_p), ("dw_qw", ctypes.c_void_p), ("dw_qr", ctypes.c_void_p),
                ("dw_v", ctypes.c_void_p), ("dw_g", ctypes.c_void_p), ("dw_o", ctypes.c_void_p),
                ("d_subkeys", ctypes.c_void_p), ("dbank", ctypes.c_void_p), ("d_bank_init", ctypes.c_void_p)]


class KernelTimes(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * len(KERNEL_KINDS)),
                ("ms", ctypes.c_double * len(KERNEL_KINDS))]


class SdmError(RuntimeError):
    """A non-OK status from the library; .status holds the code."""

    def __init__(self, status: int, func: str, message: str):
        self.status = status
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)}: {message}")


STATUS_NAMES = {
    SDM_OK: "ok", SDM_ERR_INVALID_ARG: "invalid argument", SDM_ERR_UNSUPPORTED: "unsupported",
    SDM_ERR_ALIAS: "alias", SDM_ERR_WORKSPACE: "workspace", SDM_ERR_CUDA: "cuda",
    SDM_ERR_DEVICE: "device",
}

_P = ctypes.c_void_p
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libsdm_gb300.so.  Raises ImportError when it is not built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"SDM CUDA library not built ({path}); run "
                              "`python gated_delta_rule_factor_gb300/build.py`")
        _build.build()
    lib = ctypes.CDLL(path)
    sp = ctypes.POINTER(SdmShape)
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.sdm_write_read_workspace_size.argtypes = [sp, szp]
    lib.sdm_decode_workspace_size.argtypes = [sp, szp]
    lib.sdm_write_read.argtypes = [sp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   ctypes.c_size_t, _P]
    lib.sdm_write_read_static.argtypes = [sp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.sdm_snapshot_bytes.argtypes = [sp, ctypes.c_int32, szp]
    lib.sdm_write_read_train.argtypes = [sp] + [_P] * 13 + [ctypes.c_size_t, ctypes.c_int32, _P,
                                                            ctypes.c_size_t, _P]
    lib.sdm_write_read_backward_workspace_size.argtypes = [sp, szp]
    lib.sdm_write_read_backward.argtypes = [sp] + [_P] * 10 + [ctypes.c_size_t, ctypes.c_int32] + \
        [_P] * 9 + [ctypes.c_size_t, _P]
    lib.sdm_layer_workspace_size.argtypes = [sp, ctypes.c_int64, szp]
    lib.sdm_layer_forward.argtypes = [sp, ctypes.c_int64] + [_P] * 16 + [ctypes.c_size_t, _P]
    lib.sdm_layer_forward_train.argtypes = [sp, ctypes.c_int64] + [_P] * 10 + [ctypes.POINTER(SdmLayerSaved), _P,
                                                                          ctypes.c_size_t, _P]
    lib.sdm_layer_backward_workspace_size.argtypes = [sp, ctypes.c_int64, szp]
    lib.sdm_layer_backward.argtypes = [sp, ctypes.c_int64] + [_P] * 9 + [ctypes.POINTER(SdmLayerSaved),
                                                                        ctypes.POINTER(SdmLayerGrads), _P,
                                                                        ctypes.c_size_t, _P]
    lib.sdm_decode_step.argtypes = [sp, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_int, _P,
                                    _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sdm_last_device_error.argtypes = [_P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int32), _P]
    lib.sdm_status_string.argtypes = [ctypes.c_int]
    lib.sdm_status_string.restype = ctypes.c_char_p
    lib.sdm_last_error_message.argtypes = []
    lib.sdm_last_error_message.restype = ctypes.c_char_p
    lib.sdm_abi_version.restype = ctypes.c_int32
    lib.sdm_launch_count.restype = ctypes.c_uint64
    lib.sdm_profile_begin.argtypes = []
    lib.sdm_profile_end.argtypes = [ctypes.POINTER(KernelTimes)]
    lib.sdm_kernel_name.argtypes = [ctypes.c_int32]
    lib.sdm_kernel_name.restype = ctypes.c_char_p
    lib.sdm_test_stall_decode_copy.argtypes = [ctypes.c_int]
    lib.sdm_test_force_write_read_layout.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.sdm_test_force_simt_scorer.argtypes = [ctypes.c_int]
    lib.sdm_test_factor_scores.argtypes = [sp, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    for name in ("sdm_write_read_workspace_size", "sdm_decode_workspace_size", "sdm_write_read",
                 "sdm_write_read_static", "sdm_decode_step", "sdm_last_device_error", "sdm_profile_begin", "sdm_profile_end",
                 "sdm_snapshot_bytes", "sdm_write_read_train", "sdm_write_read_backward_workspace_size",
                 "sdm_write_read_backward", "sdm_layer_workspace_size", "sdm_layer_forward",
                 "sdm_layer_forward_train", "sdm_layer_backward_workspace_size", "sdm_layer_backward",
                 "sdm_test_factor_scores"):
        getattr(lib, name).restype = ctypes.c_int
    if lib.sdm_abi_version() != ABI_VERSION:
        raise ImportError(f"SDM library ABI {lib.sdm_abi_version()} != binding ABI {ABI_VERSION}")
    _lib = lib
    return lib


def check(status: int, func: str) -> None:
    if status != SDM_OK:
        msg = load().sdm_last_error_message().decode(errors="replace")
        raise SdmError(status, func, msg)

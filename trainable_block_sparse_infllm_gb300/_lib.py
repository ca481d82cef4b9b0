"""ctypes binding of libinfllmv2.so (include/infllmv2.h).

Argument marshalling only: every call forwards device pointers, sizes and the
current CUDA stream to the C ABI, and raises ``InfLLMv2Error`` on a non-zero
return code.  There is no fallback: if the library is missing the import of
this module fails.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# INFLLMV2_LIBRARY=checked loads the checked build (libinfllmv2_checked.so,
# build_lib.build(checked=True)) instead of the product library.
LIB_PATH = os.path.join(_PKG, "libinfllmv2_checked.so" if os.environ.get("INFLLMV2_LIBRARY") == "checked"
                        else "libinfllmv2.so")

OK = 0
INVALID_ARGUMENT = 1
UNSUPPORTED = 2
WORKSPACE_TOO_SMALL = 3
CUDA_ERROR = 4
DEVICE_BAD_KV_LEN = 0x1
DEVICE_TIMEOUT = 0x2
DEVICE_BOUNDS = 0x4
OP_SELECT = 1
OP_DECODE = 2
OP_PREFILL = 3
OP_DECODE_STEP = 4
OP_BACKWARD = 5


class InfLLMv2Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{status_string(code)}: {message}")
        self.code = code


class Params(ctypes.Structure):
    """Mirror of ``infllmv2_params``."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("kernel_size", ctypes.c_int32),
        ("kernel_stride", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("n_init_blocks", ctypes.c_int32),
        ("n_local_blocks", ctypes.c_int32),
        ("topk_includes_forced", ctypes.c_int32),
        ("max_kv_len", ctypes.c_int32),
        ("score_scale", ctypes.c_float),
        ("attn_scale", ctypes.c_float),
    ]

    def __repr__(self):
        return "Params(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with build_lib.build() "
                      "(there is no CPU fallback for this library)")

lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_P = ctypes.POINTER(Params)
_i32 = ctypes.c_int32

lib.infllmv2_default_params.argtypes = [_P, _i32, _i32, _i32, _i32, _i32]
lib.infllmv2_default_params.restype = None
lib.infllmv2_max_selected.argtypes = [_P]
lib.infllmv2_max_selected.restype = _i32
lib.infllmv2_num_kernels.argtypes = [_P]
lib.infllmv2_num_kernels.restype = _i32
lib.infllmv2_workspace_size.argtypes = [_P, _i32, _i32]
lib.infllmv2_workspace_size.restype = ctypes.c_size_t
lib.infllmv2_compress_keys.argtypes = [_P, _vp, _vp, _i32, _i32, _vp, _vp]
lib.infllmv2_compress_keys.restype = ctypes.c_int
lib.infllmv2_select_blocks.argtypes = [_P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
lib.infllmv2_select_blocks.restype = ctypes.c_int
lib.infllmv2_select_blocks_static.argtypes = [_P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
lib.infllmv2_select_blocks_static.restype = ctypes.c_int
for _name in ("infllmv2_sparse_attn_decode", "infllmv2_sparse_attn_prefill"):
    getattr(lib, _name).argtypes = [_P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    ctypes.c_size_t, _vp]
    getattr(lib, _name).restype = ctypes.c_int
lib.infllmv2_is_checked_build.argtypes = []
lib.infllmv2_is_checked_build.restype = ctypes.c_int
lib.infllmv2_test_hooks.argtypes = [ctypes.c_uint32]
lib.infllmv2_test_hooks.restype = ctypes.c_int
lib.infllmv2_coarse_means.argtypes = [_P, _vp, _vp, _i32, _vp, _vp]
lib.infllmv2_coarse_means.restype = ctypes.c_int
lib.infllmv2_select_blocks_coarse_lse.argtypes = [_P, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
lib.infllmv2_select_blocks_coarse_lse.restype = ctypes.c_int
lib.infllmv2_decode_step.argtypes = [_P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     ctypes.c_size_t, _vp]
lib.infllmv2_decode_step.restype = ctypes.c_int
lib.infllmv2_append_kv.argtypes = [_P, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
lib.infllmv2_append_kv.restype = ctypes.c_int
lib.infllmv2_append_decode_step.argtypes = [_P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
lib.infllmv2_append_decode_step.restype = ctypes.c_int
lib.infllmv2_sparse_attn_backward.argtypes = [_P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
lib.infllmv2_sparse_attn_backward.restype = ctypes.c_int
lib.infllmv2_status_string.argtypes = [ctypes.c_int]
lib.infllmv2_status_string.restype = ctypes.c_char_p
lib.infllmv2_last_error.argtypes = []
lib.infllmv2_last_error.restype = ctypes.c_char_p
lib.infllmv2_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
lib.infllmv2_get_device_status.restype = ctypes.c_int

EXPORTED = (
    "infllmv2_default_params", "infllmv2_max_selected", "infllmv2_num_kernels",
    "infllmv2_workspace_size", "infllmv2_compress_keys", "infllmv2_select_blocks",
    "infllmv2_select_blocks_static",
    "infllmv2_sparse_attn_decode", "infllmv2_sparse_attn_prefill", "infllmv2_decode_step",
    "infllmv2_coarse_means", "infllmv2_select_blocks_coarse_lse", "infllmv2_sparse_attn_backward",
    "infllmv2_append_kv", "infllmv2_append_decode_step",
    "infllmv2_status_string",
    "infllmv2_last_error", "infllmv2_get_device_status",
)


def status_string(code: int) -> str:
    return lib.infllmv2_status_string(code).decode()


def check(rc: int) -> None:
    if rc != OK:
        raise InfLLMv2Error(rc, lib.infllmv2_last_error().decode())

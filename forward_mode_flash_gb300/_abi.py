"""ctypes view of the C ABI in ``include/jvp_attn.h``.

Loads ``_build/libjvp_attn.so`` (built by ``forward_mode_flash_gb300.build``)
and declares every exported entry point.  There is no fallback: if the library
is missing or fails to load, importing the binding raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libjvp_attn.so")

JVP_OK, JVP_ERR_INVALID_ARG, JVP_ERR_UNSUPPORTED, JVP_ERR_ALIGNMENT = 0, 1, 2, 3
JVP_ERR_CUDA, JVP_ERR_DEVICE_TIMEOUT, JVP_ERR_WORKSPACE, JVP_ERR_BOUNDS = 4, 5, 6, 7
# fixed device scratch of jvp_attn_bwd_dual_noalloc (JVP_BWD_NOALLOC_SCRATCH_BYTES)
JVP_BWD_NOALLOC_SCRATCH_BYTES = 4 << 20
JVP_F32, JVP_F16, JVP_BF16 = 0, 1, 2
JVP_MASK_NONE, JVP_MASK_BOOL, JVP_MASK_ADDITIVE, JVP_MASK_CAUSAL = 0, 1, 2, 3
JVP_MASK_BOOL_CAUSAL, JVP_MASK_ADDITIVE_CAUSAL = 4, 5

# Every function the header declares (checked against the library's exports).
EXPORTS = (
    "jvp_attn_fwd_dual",
    "jvp_attn_fwd_dual_ws",
    "jvp_attn_fwd_dual_workspace_size",
    "jvp_attn_fwd_dual_host",
    "jvp_attn_fwd_dual_host_workspace_size",
    "jvp_attn_fwd",
    "jvp_attn_bwd_dual",
    "jvp_attn_bwd_dual_workspace_size",
    "jvp_attn_bwd_dual_noalloc",
    "jvp_attn_bwd",
    "jvp_attn_bwd_workspace_size",
    "jvp_attn_get_device_status",
    "jvp_attn_status_string",
    "jvp_attn_last_error",
    "jvp_attn_version",
    "jvp_attn_selftest_wait_timeout",
    "jvp_attn_debug_last_path",
    "jvp_attn_debug_set_cluster_split",
)


class Shape(ctypes.Structure):
    # Hkv = 0 means Hkv = H (no grouped-query attention)
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Nq", ctypes.c_int64),
                ("Nk", ctypes.c_int64), ("D", ctypes.c_int64), ("Hkv", ctypes.c_int64)]


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64),
                ("d", ctypes.c_int64)]


class Mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_h", ctypes.c_int64), ("stride_q", ctypes.c_int64),
                ("stride_k", ctypes.c_int64)]


_lock = threading.Lock()
_libs = {}           # path -> loaded library
_debug_path = None   # when set, load() returns this debug build instead


class JvpAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"jvp_attn status {status}: {message}")
        self.status = status


def use_debug_build(path: str | None) -> None:
    """Route load() to a debug build of the library (device-side bounds checks;
    forward_mode_flash_gb300.build.build(debug=True) makes it), or back to the
    ordinary build with None."""
    global _debug_path
    _debug_path = path


def load(path: str | None = None):
    """Load (once per file) and return the library with argument types declared."""
    with _lock:
        p = path or _debug_path or LIB_PATH
        if p in _libs:
            return _libs[p]
        if not os.path.exists(p):
            raise ImportError(
                f"{p} is missing: build it with forward_mode_flash_gb300.build.build() "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(p)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        SP, STP, MP = ctypes.POINTER(Shape), ctypes.POINTER(Strides), ctypes.POINTER(Mask)
        lib.jvp_attn_fwd_dual.argtypes = [SP, i32, vp, vp, vp, vp, vp, vp, STP, MP, f32, vp, vp,
                                          STP, vp, vp, vp]
        lib.jvp_attn_fwd_dual.restype = i32
        lib.jvp_attn_fwd_dual_ws.argtypes = lib.jvp_attn_fwd_dual.argtypes[:-1] + \
            [vp, ctypes.c_size_t, vp]
        lib.jvp_attn_fwd_dual_ws.restype = i32
        lib.jvp_attn_fwd_dual_workspace_size.argtypes = [SP, i32]
        lib.jvp_attn_fwd_dual_workspace_size.restype = ctypes.c_size_t
        lib.jvp_attn_fwd_dual_host.argtypes = [SP, i32] + [vp] * 6 + [MP, f32, vp, vp, vp, vp,
                                                                        i32, vp, ctypes.c_size_t,
                                                                        vp]
        lib.jvp_attn_fwd_dual_host.restype = i32
        lib.jvp_attn_fwd_dual_host_workspace_size.argtypes = [SP, i32, i32]
        lib.jvp_attn_fwd_dual_host_workspace_size.restype = ctypes.c_size_t
        lib.jvp_attn_fwd.argtypes = [SP, i32, vp, vp, vp, STP, MP, f32, vp, STP, vp, vp]
        lib.jvp_attn_fwd.restype = i32
        lib.jvp_attn_bwd_dual.argtypes = [SP, i32] + [vp] * 8 + [vp, vp] + [vp, vp] + [STP, MP, f32] + \
            [vp] * 6 + [STP, vp, ctypes.c_size_t, vp]
        lib.jvp_attn_bwd_dual.restype = i32
        lib.jvp_attn_bwd_dual_noalloc.argtypes = lib.jvp_attn_bwd_dual.argtypes[:-3] + [vp]
        lib.jvp_attn_bwd_dual_noalloc.restype = i32
        lib.jvp_attn_bwd_dual_workspace_size.argtypes = [SP, i32]
        lib.jvp_attn_bwd_dual_workspace_size.restype = ctypes.c_size_t
        # shape, dtype, q k v o lse g_o, in_strides, mask, scale, g_q g_k g_v,
        # out_strides, workspace, bytes, stream
        lib.jvp_attn_bwd.argtypes = [SP, i32] + [vp] * 6 + [STP, MP, f32] + [vp] * 3 + \
            [STP, vp, ctypes.c_size_t, vp]
        lib.jvp_attn_bwd.restype = i32
        lib.jvp_attn_bwd_workspace_size.argtypes = [SP, i32]
        lib.jvp_attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.jvp_attn_get_device_status.argtypes = [vp]
        lib.jvp_attn_get_device_status.restype = i32
        lib.jvp_attn_status_string.argtypes = [i32]
        lib.jvp_attn_status_string.restype = ctypes.c_char_p
        lib.jvp_attn_last_error.argtypes = []
        lib.jvp_attn_last_error.restype = ctypes.c_char_p
        lib.jvp_attn_version.argtypes = []
        lib.jvp_attn_version.restype = i32
        lib.jvp_attn_selftest_wait_timeout.argtypes = [ctypes.c_int64, vp]
        lib.jvp_attn_selftest_wait_timeout.restype = i32
        lib.jvp_attn_debug_last_path.argtypes = []
        lib.jvp_attn_debug_last_path.restype = i32
        lib.jvp_attn_debug_set_cluster_split.argtypes = [i32]
        lib.jvp_attn_debug_set_cluster_split.restype = i32
        _libs[p] = lib
        return lib


def check(status: int) -> None:
    """Raise JvpAttnError with the library's message if status is not JVP_OK."""
    if status != JVP_OK:
        msg = load().jvp_attn_last_error().decode(errors="replace")
        raise JvpAttnError(status, msg or load().jvp_attn_status_string(status).decode())

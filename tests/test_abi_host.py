"""Host-side checks of the C ABI that need no GPU.

The library must load without a device, export every function that
``include/jvp_attn.h`` declares, and reject bad arguments with the documented
status before it touches the device.
"""

import ctypes
import os
import re

import pytest

from forward_mode_flash_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "jvp_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jvp_attn_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(_abi.EXPORTS)


def test_library_loads_and_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert lib.jvp_attn_version() == 200


def test_status_strings(lib):
    for code in range(7):
        assert lib.jvp_attn_status_string(code)
    assert lib.jvp_attn_status_string(0) == b"ok"


def _strides(n, shape):
    B, H, N, D = shape
    arr = (_abi.Strides * n)()
    for i in range(n):
        arr[i] = _abi.Strides(H * N * D, N * D, D, 1)
    return arr


def call_fwd_dual(lib, shape=(1, 2, 64, 64), dtype=_abi.JVP_BF16, ptrs=0x1000, mask=None,
                  scale=0.125, in_strides=None, out_strides=None, hkv=0):
    B, H, N, D = shape
    sh = _abi.Shape(B, H, N, N, D, hkv)
    p = ctypes.c_void_p(ptrs) if ptrs else None
    ins = in_strides if in_strides is not None else _strides(6, shape)
    outs = out_strides if out_strides is not None else _strides(2, shape)
    m = ctypes.byref(mask) if mask is not None else None
    return lib.jvp_attn_fwd_dual(ctypes.byref(sh), dtype, p, p, p, p, p, p, ins, m, scale, p, p,
                                 outs, None, None, None)


def test_validation_rejects_bad_arguments_without_a_device(lib):
    assert lib.jvp_attn_fwd_dual(None, 2, None, None, None, None, None, None, None, None, 1.0,
                                 None, None, None, None, None, None) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, shape=(1, 1, 8, 0)) == _abi.JVP_ERR_INVALID_ARG       # D = 0
    assert call_fwd_dual(lib, shape=(1, 1, 8, 256)) == _abi.JVP_ERR_UNSUPPORTED     # D > 128
    assert call_fwd_dual(lib, shape=(-1, 1, 8, 64)) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, dtype=7) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, scale=float("nan")) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, scale=float("inf")) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, ptrs=0) == _abi.JVP_ERR_INVALID_ARG                   # null inputs
    assert call_fwd_dual(lib, ptrs=0x1001) == _abi.JVP_ERR_ALIGNMENT                # odd address
    bad = _strides(6, (1, 2, 64, 64))
    bad[2] = _abi.Strides(8192, 4096, 64, 2)
    assert call_fwd_dual(lib, in_strides=bad) == _abi.JVP_ERR_INVALID_ARG           # d stride != 1
    causal_with_tensor = _abi.Mask(_abi.JVP_MASK_CAUSAL, 0x2000, 0, 0, 64, 1)
    assert call_fwd_dual(lib, mask=causal_with_tensor) == _abi.JVP_ERR_INVALID_ARG
    bool_without_tensor = _abi.Mask(_abi.JVP_MASK_BOOL, None, 0, 0, 64, 1)
    assert call_fwd_dual(lib, mask=bool_without_tensor) == _abi.JVP_ERR_INVALID_ARG
    unknown = _abi.Mask(9, None, 0, 0, 0, 0)
    assert call_fwd_dual(lib, mask=unknown) == _abi.JVP_ERR_INVALID_ARG
    assert b"causal" in lib.jvp_attn_last_error() or lib.jvp_attn_last_error()


def test_empty_problems_succeed_without_a_device(lib):
    assert call_fwd_dual(lib, shape=(0, 2, 64, 64), ptrs=0) == _abi.JVP_OK
    assert call_fwd_dual(lib, shape=(1, 0, 64, 64), ptrs=0) == _abi.JVP_OK
    assert call_fwd_dual(lib, shape=(1, 2, 0, 64), ptrs=0) == _abi.JVP_OK
    assert lib.jvp_attn_debug_last_path() == 0


def test_selftest_rejects_bad_limits(lib):
    assert lib.jvp_attn_selftest_wait_timeout(0, None) == _abi.JVP_ERR_INVALID_ARG
    assert lib.jvp_attn_selftest_wait_timeout(1 << 31, None) == _abi.JVP_ERR_INVALID_ARG


def test_grouped_heads_and_combined_masks_are_validated_without_a_device(lib):
    # H must be a multiple of Hkv; Hkv = 0 means H
    assert call_fwd_dual(lib, shape=(1, 8, 64, 64), hkv=3) == _abi.JVP_ERR_INVALID_ARG
    assert b"multiple of Hkv" in lib.jvp_attn_last_error()
    assert call_fwd_dual(lib, shape=(1, 8, 64, 64), hkv=-2) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, shape=(0, 8, 64, 64), hkv=2, ptrs=0) == _abi.JVP_OK
    assert call_fwd_dual(lib, shape=(0, 8, 64, 64), hkv=8, ptrs=0) == _abi.JVP_OK
    # the combined kinds need a mask tensor; CAUSAL alone takes none
    for kind in (_abi.JVP_MASK_BOOL_CAUSAL, _abi.JVP_MASK_ADDITIVE_CAUSAL):
        assert call_fwd_dual(lib, mask=_abi.Mask(kind, None, 0, 0, 64, 1)) == \
            _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, mask=_abi.Mask(6, 0x2000, 0, 0, 64, 1)) == _abi.JVP_ERR_INVALID_ARG
    assert call_fwd_dual(lib, mask=_abi.Mask(_abi.JVP_MASK_CAUSAL, 0x2000, 0, 0, 64, 1)) == \
        _abi.JVP_ERR_INVALID_ARG
    assert b"BOOL_CAUSAL" in lib.jvp_attn_last_error()


def test_split_workspace_size_is_zero_without_a_device_or_for_other_shapes(lib):
    sh = _abi.Shape(1, 2, 1000, 1000, 64, 0)
    assert lib.jvp_attn_fwd_dual_workspace_size(ctypes.byref(sh), _abi.JVP_BF16) == 0  # no GPU here
    sh32 = _abi.Shape(1, 2, 1000, 1000, 40, 0)
    assert lib.jvp_attn_fwd_dual_workspace_size(ctypes.byref(sh32), _abi.JVP_BF16) == 0
    assert lib.jvp_attn_fwd_dual_workspace_size(None, _abi.JVP_BF16) == 0


def test_host_buffer_entry_point_validates_before_touching_a_device(lib):
    sh = _abi.Shape(2, 4, 256, 256, 64, 0)
    need = lib.jvp_attn_fwd_dual_host_workspace_size(ctypes.byref(sh), _abi.JVP_BF16, 4)
    # two slots of 2 (b, h) pairs: q, dq, o, t_o, k, v, dk, dv of 2*256*64 bf16, lse and mu
    assert need == 2 * (8 * 2 * 256 * 64 * 2 + 2 * 2 * 256 * 4)
    p = ctypes.c_void_p(0x10000)

    def call(shape=sh, chunks=4, ws=0x100000, ws_bytes=need, mask=None):
        m = ctypes.byref(mask) if mask is not None else None
        return lib.jvp_attn_fwd_dual_host(ctypes.byref(shape), _abi.JVP_BF16, p, p, p, p, p, p,
                                          m, 0.125, p, p, None, None, chunks,
                                          ctypes.c_void_p(ws), ws_bytes, None)
    assert call(chunks=0) == _abi.JVP_ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == _abi.JVP_ERR_WORKSPACE
    assert call(ws=0x100010) == _abi.JVP_ERR_ALIGNMENT
    assert call(shape=_abi.Shape(2, 4, 256, 256, 64, 2)) == _abi.JVP_ERR_UNSUPPORTED
    per_head = _abi.Mask(_abi.JVP_MASK_BOOL, 0x2000, 0, 256 * 256, 256, 1)
    assert call(mask=per_head) == _abi.JVP_ERR_INVALID_ARG
    assert b"shared by every" in lib.jvp_attn_last_error()



def _bwd_args(n):
    return [ctypes.c_void_p(0x10000)] * n


def test_sizes_that_would_overflow_are_rejected_without_a_device(lib):
    # Sizes above 2^31 - 1, and products of sizes that would wrap int64 (or
    # wrap to zero: B = H = 2^32), are rejected before anything else happens.
    big, wrap = (1 << 31) - 1, 1 << 32
    for B, H, N in ((wrap, wrap, 64), (big, big, big), (1 << 31, 1, 64), (big, big, 64)):
        assert call_fwd_dual(lib, shape=(B, H, N, 64)) == _abi.JVP_ERR_UNSUPPORTED, (B, H, N)
        sh = _abi.Shape(B, H, N, N, 64, 0)
        ins = _strides(10, (1, 1, 64, 64))
        outs = _strides(6, (1, 1, 64, 64))
        none = _abi.Mask(_abi.JVP_MASK_NONE, None, 0, 0, 0, 0)
        st = lib.jvp_attn_bwd_dual(ctypes.byref(sh), _abi.JVP_BF16, *_bwd_args(10), *_bwd_args(2),
                                   ins, ctypes.byref(none), 0.125, *_bwd_args(6), outs,
                                   ctypes.c_void_p(0x100000), 1 << 40, None)
        assert st == _abi.JVP_ERR_UNSUPPORTED, (B, H, N, st)
        # the no-allocation backward: such a problem never fits its fixed scratch
        st = lib.jvp_attn_bwd_dual_noalloc(ctypes.byref(sh), _abi.JVP_BF16, *_bwd_args(10),
                                           *_bwd_args(2), ins, ctypes.byref(none), 0.125,
                                           *_bwd_args(6), outs, None)
        assert st == _abi.JVP_ERR_WORKSPACE, (B, H, N, st)
        assert lib.jvp_attn_bwd_dual_workspace_size(ctypes.byref(sh), _abi.JVP_BF16) == \
            ctypes.c_size_t(-1).value
        assert lib.jvp_attn_fwd_dual_workspace_size(ctypes.byref(sh), _abi.JVP_BF16) == 0
        assert lib.jvp_attn_fwd_dual_host_workspace_size(ctypes.byref(sh), _abi.JVP_BF16, 4) == 0
    # the forward-only entry point shares the checks
    sh = _abi.Shape(wrap, wrap, 64, 64, 64, 0)
    p = ctypes.c_void_p(0x10000)
    st = lib.jvp_attn_fwd(ctypes.byref(sh), _abi.JVP_BF16, p, p, p, _strides(3, (1, 1, 64, 64)),
                          None, 0.125, p, _strides(1, (1, 1, 64, 64)), None, None)
    assert st == _abi.JVP_ERR_UNSUPPORTED
    assert b"2^31" in lib.jvp_attn_last_error() or b"too large" in lib.jvp_attn_last_error()


def test_debug_build_compiles_and_exports_the_same_functions():
    # The bounds-checking build (-DJVP_DEBUG_CHECKS) of every translation unit.
    path = build.build(debug=True)
    dbg = ctypes.CDLL(path)
    for n in header_functions():
        assert hasattr(dbg, n), n
    dbg.jvp_attn_status_string.restype = ctypes.c_char_p
    assert dbg.jvp_attn_status_string(_abi.JVP_ERR_BOUNDS).startswith(b"device-side bounds")


def test_primal_backward_validates_before_touching_a_device(lib):
    # jvp_attn_bwd: the dual backward's checks on its own argument list
    # (q, k, v, o, lse, g_o; g_q, g_k, g_v), then the device lookup.
    p = ctypes.c_void_p(0x10000)
    ws = ctypes.c_void_p(0x100000)
    none = _abi.Mask(_abi.JVP_MASK_NONE, None, 0, 0, 0, 0)

    def call(shape=(1, 2, 64, 64), ptr=p, ins=None, outs=None, scale=0.125, ws_bytes=1 << 20,
             lse=p):
        B, H, N, D = shape
        sh = _abi.Shape(B, H, N, N, D, 0)
        ins = ins if ins is not None else _strides(5, shape)
        outs = outs if outs is not None else _strides(3, shape)
        return lib.jvp_attn_bwd(ctypes.byref(sh), _abi.JVP_BF16, ptr, ptr, ptr, ptr, lse, ptr, ins,
                                ctypes.byref(none), scale, ptr, ptr, ptr, outs, ws, ws_bytes, None)

    assert lib.jvp_attn_bwd(None, _abi.JVP_BF16, p, p, p, p, p, p, None, None, 0.125, p, p, p,
                            None, ws, 1 << 20, None) == _abi.JVP_ERR_INVALID_ARG
    assert call(shape=(1, 1, 8, 256)) == _abi.JVP_ERR_UNSUPPORTED
    assert call(scale=float("nan")) == _abi.JVP_ERR_INVALID_ARG
    assert call(ptr=None) == _abi.JVP_ERR_INVALID_ARG                      # null tensors
    assert call(ptr=ctypes.c_void_p(0x10001)) == _abi.JVP_ERR_ALIGNMENT    # odd address
    assert call(lse=None) == _abi.JVP_ERR_INVALID_ARG                      # lse is required
    bad = _strides(5, (1, 2, 64, 64))
    bad[4] = _abi.Strides(8192, 4096, 64, 2)
    assert call(ins=bad) == _abi.JVP_ERR_INVALID_ARG                       # d stride != 1
    assert call(ws_bytes=8) == _abi.JVP_ERR_WORKSPACE                      # 8*B*H*Nq needed
    assert call(shape=(0, 2, 64, 64), ptr=None) == _abi.JVP_OK            # empty problem
    sh = _abi.Shape(2, 8, 2048, 2048, 64, 0)
    assert lib.jvp_attn_bwd_workspace_size(ctypes.byref(sh), _abi.JVP_BF16) == \
        lib.jvp_attn_bwd_dual_workspace_size(ctypes.byref(sh), _abi.JVP_BF16) == 8 * 2 * 8 * 2048
    big = _abi.Shape(1 << 32, 1 << 32, 64, 64, 64, 0)
    assert lib.jvp_attn_bwd_workspace_size(ctypes.byref(big), _abi.JVP_BF16) == \
        ctypes.c_size_t(-1).value

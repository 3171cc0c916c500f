"""Thin ctypes binding of the gbconv C ABI (include/gbconv.h), same names.

Argument marshalling only: every function forwards to the C entry point of the
same name in the in-tree libgbconv.so, which does all the work in CUDA
kernels.  Device pointers are plain integers (e.g. ``tensor.data_ptr()``),
streams are integer handles (``torch.cuda.current_stream().cuda_stream``) or
None for the legacy default stream.  A non-OK status raises GbconvError
carrying the status name and the library's detail string.

There is no fallback: if libgbconv.so is missing or fails to load, importing
the library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgbconv.so")

CONV_BF16, CONV_F32, CONV_INT8 = 0, 1, 2
CONV_NHWC, CONV_NCHW, CONV_NC32HW32 = 0, 1, 2
CONV_ACT_NONE, CONV_ACT_RELU, CONV_ACT_RELU6 = 0, 1, 2

CONV_ALGO_AUTO = -1
CONV_ALGO_DIRECT = 0
CONV_ALGO_IGEMM_N64 = 1
CONV_ALGO_IGEMM_N128 = 2
CONV_ALGO_IGEMM_N256 = 3
CONV_ALGO_WINO_F2 = 4
CONV_ALGO_WINO_F6 = 5
CONV_ALGO_DEPTHWISE = 6
CONV_ALGO_INT8_MMA = 7
CONV_ALGO_INT8_TC = 8
CONV_ALGO_IM2COL_GEMM = 9
CONV_ALGO_STEM_S2D = 10
CONV_ALGO_IGEMM_TF32 = 11
CONV_ALGO_INT8_WINO_F2 = 12
CONV_ALGO_STEM_S2D4 = 13
CONV_ALGO_IGEMM_2SM = 14
CONV_ALGO_INT8_TC_CHUNK = 15
CONV_ALGO_IGEMM_STRIP = 16
CONV_ALGO_COUNT = 17

STATUS_NAMES = {
    0: "CONV_OK", 1: "CONV_ERR_BAD_PARAM", 2: "CONV_ERR_UNSUPPORTED", 3: "CONV_ERR_ALIGNMENT",
    4: "CONV_ERR_WORKSPACE", 5: "CONV_ERR_CUDA", 6: "CONV_ERR_TIMEOUT", 7: "CONV_ERR_INTERNAL",
    8: "CONV_ERR_FASTRUN_FILE", 9: "CONV_ERR_NOT_FOUND",
}

# Every symbol include/gbconv.h declares, with (restype, argtypes).
_i, _sz, _p, _f = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
_cp = ctypes.c_char_p
SIGNATURES = {
    "conv_desc_create": (_i, [ctypes.POINTER(_p)] + [_i] * 12),
    "conv_desc_destroy": (_i, [_p]),
    "conv_desc_set_layout": (_i, [_p, _i]),
    "conv_desc_set_epilogue": (_i, [_p, _i, _i]),
    "conv_desc_set_input_shuffle": (_i, [_p, _i]),
    "conv_desc_set_requant": (_i, [_p, _p]),
    "conv_desc_get_output_dims": (_i, [_p, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "conv_algo_count": (_i, [_p, ctypes.POINTER(_i)]),
    "conv_algo_info": (_i, [_p, _i, ctypes.POINTER(_i), ctypes.POINTER(_cp), ctypes.POINTER(_i)]),
    "conv_algo_resolve": (_i, [_p, ctypes.POINTER(_i)]),
    "conv_workspace_size": (_i, [_p, _i, ctypes.POINTER(_sz)]),
    "conv_weights_packed_size": (_i, [_p, _i, ctypes.POINTER(_sz)]),
    "conv_weights_prepack": (_i, [_p, _i, _p, _p, _p]),
    "conv_fwd": (_i, [_p, _p, _p, _p, _p, _p, _i, _p, _sz, _p]),
    "conv_fwd_host_scratch_size": (_i, [_p, _i, _i, ctypes.POINTER(_sz)]),
    "conv_fwd_host": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _p, _sz, _p]),
    "conv_fwd_noalloc": (_i, [_p, _p, _p, _p, _p, _p, _i, _p]),
    "conv_mbv2_block_packed_size": (_i, [_i, _i, _i, ctypes.POINTER(_sz)]),
    "conv_mbv2_block_prepack": (_i, [_i, _i, _i, _p, _p, _p, _p, _p, _p]),
    "conv_mbv2_block_fwd": (_i, [_i] * 6 + [_p, _p, _p, _p, _i, _p, _p]),
    "conv_fastrun_select": (_i, [_p, _p, ctypes.POINTER(_i), ctypes.POINTER(_f)]),
    "conv_fastrun_lookup": (_i, [_p, ctypes.POINTER(_i)]),
    "conv_fastrun_save": (_i, [_cp]),
    "conv_fastrun_load": (_i, [_cp]),
    "conv_fastrun_clear": (_i, []),
    "conv_nchw_f32_to_nhwc_bf16": (_i, [_p, _p, _i, _i, _i, _i, _i, _p]),
    "conv_nchw_i8_to_nc32hw32": (_i, [_p, _p, _i, _i, _i, _i, _p]),
    "conv_nc32hw32_to_nchw_i8": (_i, [_p, _p, _i, _i, _i, _i, _p]),
    "conv_nhwc_bf16_to_nchw_f32": (_i, [_p, _p, _i, _i, _i, _i, _i, _p]),
    "conv_maxpool2d_nhwc_bf16": (_i, [_p, _p, _i, _i, _i, _i, _i, _i, _i, _p]),
    "conv_global_avgpool_nhwc_bf16": (_i, [_p, _p, _i, _i, _i, _i, _p]),
    "conv_sync_status": (_i, [_p]),
    "conv_selftest_wait_timeout": (_i, [ctypes.c_uint, _p]),
    "conv_status_string": (_cp, [_i]),
    "conv_last_error_detail": (_cp, []),
    "conv_version": (_cp, []),
    "conv_launch_count": (_i, [ctypes.POINTER(ctypes.c_ulonglong)]),
}


class GbconvError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, f"status {status}")
        self.detail = detail
        super().__init__(f"{func}: {self.status_name}: {detail}")


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgbconv.so (built by build.py) and declare every signature."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise ImportError(f"{path} is missing: run cnn_convolution_gemm_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(st: int, func: str):
    if st != 0:
        detail = load_library().conv_last_error_detail().decode(errors="replace")
        raise GbconvError(st, func, detail)


def _ptr(v):
    return None if v is None or v == 0 else ctypes.c_void_p(int(v))


def _stream(s):
    return None if s is None else ctypes.c_void_p(int(s))


def conv_desc_create(N, C, H, W, K, R, S, stride=1, pad=0, dilation=1, groups=1,
                     dtype=CONV_BF16):
    d = ctypes.c_void_p()
    _check(load_library().conv_desc_create(ctypes.byref(d), N, C, H, W, K, R, S, stride, pad,
                                           dilation, groups, dtype), "conv_desc_create")
    return d


def conv_desc_destroy(desc):
    _check(load_library().conv_desc_destroy(desc), "conv_desc_destroy")


def conv_desc_set_layout(desc, layout):
    _check(load_library().conv_desc_set_layout(desc, layout), "conv_desc_set_layout")


def conv_desc_set_epilogue(desc, act, has_residual):
    _check(load_library().conv_desc_set_epilogue(desc, act, 1 if has_residual else 0),
           "conv_desc_set_epilogue")


def conv_desc_set_input_shuffle(desc, groups):
    _check(load_library().conv_desc_set_input_shuffle(desc, groups), "conv_desc_set_input_shuffle")


def conv_desc_set_requant(desc, scale_ptr):
    _check(load_library().conv_desc_set_requant(desc, _ptr(scale_ptr)), "conv_desc_set_requant")


def conv_desc_get_output_dims(desc):
    oh, ow = ctypes.c_int(), ctypes.c_int()
    _check(load_library().conv_desc_get_output_dims(desc, ctypes.byref(oh), ctypes.byref(ow)),
           "conv_desc_get_output_dims")
    return oh.value, ow.value


def conv_algo_count(desc):
    n = ctypes.c_int()
    _check(load_library().conv_algo_count(desc, ctypes.byref(n)), "conv_algo_count")
    return n.value


def conv_algo_info(desc, i):
    a, name, ap = ctypes.c_int(), ctypes.c_char_p(), ctypes.c_int()
    _check(load_library().conv_algo_info(desc, i, ctypes.byref(a), ctypes.byref(name),
                                         ctypes.byref(ap)), "conv_algo_info")
    return a.value, name.value.decode(), bool(ap.value)


def conv_algo_resolve(desc):
    a = ctypes.c_int()
    _check(load_library().conv_algo_resolve(desc, ctypes.byref(a)), "conv_algo_resolve")
    return a.value


def conv_workspace_size(desc, algo):
    n = ctypes.c_size_t()
    _check(load_library().conv_workspace_size(desc, algo, ctypes.byref(n)), "conv_workspace_size")
    return n.value


def conv_weights_packed_size(desc, algo):
    n = ctypes.c_size_t()
    _check(load_library().conv_weights_packed_size(desc, algo, ctypes.byref(n)),
           "conv_weights_packed_size")
    return n.value


def conv_weights_prepack(desc, algo, w_ptr, wpack_ptr, stream=None):
    _check(load_library().conv_weights_prepack(desc, algo, _ptr(w_ptr), _ptr(wpack_ptr),
                                               _stream(stream)), "conv_weights_prepack")


def conv_fwd(desc, x_ptr, wpack_ptr, bias_ptr, residual_ptr, y_ptr, algo=CONV_ALGO_AUTO,
             ws_ptr=None, ws_bytes=0, stream=None):
    _check(load_library().conv_fwd(desc, _ptr(x_ptr), _ptr(wpack_ptr), _ptr(bias_ptr),
                                   _ptr(residual_ptr), _ptr(y_ptr), algo, _ptr(ws_ptr), ws_bytes,
                                   _stream(stream)), "conv_fwd")


def conv_fwd_host_scratch_size(desc, algo=CONV_ALGO_AUTO, n_chunk=0):
    n = ctypes.c_size_t()
    _check(load_library().conv_fwd_host_scratch_size(desc, algo, n_chunk, ctypes.byref(n)),
           "conv_fwd_host_scratch_size")
    return n.value


def conv_fwd_host(desc, x_host_ptr, wpack_ptr, bias_ptr, residual_host_ptr, y_host_ptr,
                  algo=CONV_ALGO_AUTO, n_chunk=0, scratch_ptr=None, scratch_bytes=0, stream=None):
    """x, residual and y in host memory (page-locked for overlap); wpack, bias on
    the device.  Stream-ordered like conv_fwd."""
    _check(load_library().conv_fwd_host(desc, _ptr(x_host_ptr), _ptr(wpack_ptr), _ptr(bias_ptr),
                                        _ptr(residual_host_ptr), _ptr(y_host_ptr), algo, n_chunk,
                                        _ptr(scratch_ptr), scratch_bytes, _stream(stream)),
           "conv_fwd_host")


def conv_fwd_noalloc(desc, x_ptr, wpack_ptr, bias_ptr, residual_ptr, y_ptr, algo, stream=None):
    _check(load_library().conv_fwd_noalloc(desc, _ptr(x_ptr), _ptr(wpack_ptr), _ptr(bias_ptr),
                                           _ptr(residual_ptr), _ptr(y_ptr), algo, _stream(stream)),
           "conv_fwd_noalloc")


def conv_mbv2_block_packed_size(C_in, E, C_out):
    n = ctypes.c_size_t()
    _check(load_library().conv_mbv2_block_packed_size(C_in, E, C_out, ctypes.byref(n)),
           "conv_mbv2_block_packed_size")
    return n.value


def conv_mbv2_block_prepack(C_in, E, C_out, w_expand_ptr, b_expand_ptr, w_dw_ptr, w_project_ptr,
                            wpack_ptr, stream=None):
    _check(load_library().conv_mbv2_block_prepack(C_in, E, C_out, _ptr(w_expand_ptr),
                                                  _ptr(b_expand_ptr), _ptr(w_dw_ptr),
                                                  _ptr(w_project_ptr), _ptr(wpack_ptr),
                                                  _stream(stream)), "conv_mbv2_block_prepack")


def conv_mbv2_block_fwd(N, H, W, C_in, E, C_out, x_ptr, wpack_ptr, b_dw_ptr, b_project_ptr,
                        has_residual, y_ptr, stream=None):
    _check(load_library().conv_mbv2_block_fwd(N, H, W, C_in, E, C_out, _ptr(x_ptr),
                                              _ptr(wpack_ptr), _ptr(b_dw_ptr),
                                              _ptr(b_project_ptr), 1 if has_residual else 0,
                                              _ptr(y_ptr), _stream(stream)),
           "conv_mbv2_block_fwd")


def conv_fastrun_select(desc, stream=None):
    best = ctypes.c_int()
    times = (ctypes.c_float * CONV_ALGO_COUNT)()
    _check(load_library().conv_fastrun_select(desc, _stream(stream), ctypes.byref(best), times),
           "conv_fastrun_select")
    return best.value, [float(t) for t in times]


def conv_fastrun_lookup(desc):
    a = ctypes.c_int()
    _check(load_library().conv_fastrun_lookup(desc, ctypes.byref(a)), "conv_fastrun_lookup")
    return a.value


def conv_fastrun_save(path):
    _check(load_library().conv_fastrun_save(os.fsencode(path)), "conv_fastrun_save")


def conv_fastrun_load(path):
    _check(load_library().conv_fastrun_load(os.fsencode(path)), "conv_fastrun_load")


def conv_fastrun_clear():
    _check(load_library().conv_fastrun_clear(), "conv_fastrun_clear")


def conv_nchw_i8_to_nc32hw32(x_ptr, y_ptr, N, C, H, W, stream=None):
    _check(load_library().conv_nchw_i8_to_nc32hw32(_ptr(x_ptr), _ptr(y_ptr), N, C, H, W,
                                                   _stream(stream)), "conv_nchw_i8_to_nc32hw32")


def conv_nc32hw32_to_nchw_i8(x_ptr, y_ptr, N, C, H, W, stream=None):
    _check(load_library().conv_nc32hw32_to_nchw_i8(_ptr(x_ptr), _ptr(y_ptr), N, C, H, W,
                                                   _stream(stream)), "conv_nc32hw32_to_nchw_i8")


def conv_nchw_f32_to_nhwc_bf16(x_ptr, y_ptr, N, C, H, W, C_out, stream=None):
    _check(load_library().conv_nchw_f32_to_nhwc_bf16(_ptr(x_ptr), _ptr(y_ptr), N, C, H, W, C_out,
                                                     _stream(stream)),
           "conv_nchw_f32_to_nhwc_bf16")


def conv_nhwc_bf16_to_nchw_f32(x_ptr, y_ptr, N, C, H, W, C_in, stream=None):
    _check(load_library().conv_nhwc_bf16_to_nchw_f32(_ptr(x_ptr), _ptr(y_ptr), N, C, H, W, C_in,
                                                     _stream(stream)),
           "conv_nhwc_bf16_to_nchw_f32")


def conv_maxpool2d_nhwc_bf16(x_ptr, y_ptr, N, C, H, W, k, stride, pad, stream=None):
    _check(load_library().conv_maxpool2d_nhwc_bf16(_ptr(x_ptr), _ptr(y_ptr), N, C, H, W, k,
                                                   stride, pad, _stream(stream)),
           "conv_maxpool2d_nhwc_bf16")


def conv_global_avgpool_nhwc_bf16(x_ptr, y_ptr, N, C, H, W, stream=None):
    _check(load_library().conv_global_avgpool_nhwc_bf16(_ptr(x_ptr), _ptr(y_ptr), N, C, H, W,
                                                        _stream(stream)),
           "conv_global_avgpool_nhwc_bf16")


def conv_sync_status(stream=None):
    _check(load_library().conv_sync_status(_stream(stream)), "conv_sync_status")


def conv_selftest_wait_timeout(limit_us, stream=None):
    _check(load_library().conv_selftest_wait_timeout(limit_us, _stream(stream)),
           "conv_selftest_wait_timeout")


def conv_status_string(st):
    return load_library().conv_status_string(st).decode()


def conv_last_error_detail():
    return load_library().conv_last_error_detail().decode(errors="replace")


def conv_version():
    return load_library().conv_version().decode()


def conv_launch_count():
    """Kernels the library has enqueued since it was loaded."""
    n = ctypes.c_ulonglong(0)
    _check(load_library().conv_launch_count(ctypes.byref(n)), "conv_launch_count")
    return n.value

"""Python binding of liboidnx (the C ABI in include/oidnx.h).

Argument marshalling only: every function below calls the C function of the
same name; all compute runs in the library's CUDA kernels.  Device pointers
and streams are plain integers (e.g. ``tensor.data_ptr()`` and
``torch.cuda.current_stream().cuda_stream``).  A non-OK status raises
``OidnxError`` carrying the status code and ``oidnx_last_error()``.

Importing fails loudly when the library has not been built (there is no
fallback): build it with ``python conv2d_implicit_gemm_gb300/build.py``.
"""

import ctypes
import json
import os
import struct

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboidnx.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build the CUDA library first "
        "(python conv2d_implicit_gemm_gb300/build.py)")
_lib = ctypes.CDLL(_LIB_PATH)

OK = 0
ERR_INVALID_ARGUMENT = 1
ERR_INVALID_MODEL = 2
ERR_UNSUPPORTED = 3
ERR_OUT_OF_MEMORY = 4
ERR_CUDA = 5
ERR_RELEASED = 6
ERR_TIMEOUT = 7
ERR_NOT_COMMITTED = 8

IMAGE_COLOR, IMAGE_ALBEDO, IMAGE_NORMAL, IMAGE_OUTPUT = 0, 1, 2, 3
PRECISION_AUTO, PRECISION_FP32, PRECISION_FP16 = 0, 1, 2
TRANSFER_PU, TRANSFER_LOG = 0, 1

LAYER_NAMES = (
    "enc_conv0", "enc_conv1", "enc_conv2", "enc_conv3", "enc_conv4",
    "enc_conv5a", "enc_conv5b", "dec_conv4a", "dec_conv4b", "dec_conv3a",
    "dec_conv3b", "dec_conv2a", "dec_conv2b", "dec_conv1a", "dec_conv1b",
    "dec_conv0",
)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_st = ctypes.c_int


def _sig(name, res, *args):
    fn = getattr(_lib, name)
    fn.restype = res
    fn.argtypes = list(args)
    return fn


_sig("oidnx_filter_create", _st, _vp, _sz, _i, ctypes.POINTER(_vp))
_sig("oidnx_filter_set_image", _st, _vp, _i, _vp, _sz)
_sig("oidnx_filter_set_int", _st, _vp, ctypes.c_char_p, _i)
_sig("oidnx_filter_get_int", _st, _vp, ctypes.c_char_p, ctypes.POINTER(_i))
_sig("oidnx_filter_set_float", _st, _vp, ctypes.c_char_p, ctypes.c_float)
_sig("oidnx_filter_commit", _st, _vp)
_sig("oidnx_filter_execute", _st, _vp, _vp)
_sig("oidnx_filter_execute_host", _st, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("oidnx_filter_execute_host_async", _st, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("oidnx_filter_wait_host", _st, _vp)
_sig("oidnx_network_execute", _st, _vp, _vp, _i, _i, _vp, _vp)
_sig("oidnx_network_execute_noalloc", _st, _vp, _vp, _i, _i, _vp, _vp)
_sig("oidnx_output_pass", _st, _vp, _vp, _i, _i, _vp, _sz, _vp, _sz, _i, ctypes.c_float, _vp)
_sig("oidnx_filter_sync_status", _st, _vp)
_sig("oidnx_debug_wait_probe", _st, _vp, ctypes.c_uint, _vp)
_sig("oidnx_profile_next", _st, _vp)
_sig("oidnx_get_profile", _st, _vp, ctypes.c_char_p, _sz)
_sig("oidnx_get_resource_info", _st, _vp, ctypes.c_char_p, _sz)
_sig("oidnx_debug_read_activation", _st, _vp, _i, _vp, _sz, ctypes.POINTER(_sz))
_sig("oidnx_last_error", ctypes.c_char_p)
_sig("oidnx_filter_release", None, _vp)
_sig("oidnx_conv_create", _st, _vp, _vp, _i, _i, _i, ctypes.POINTER(_vp))
_sig("oidnx_conv_execute", _st, _vp, _vp, _vp, _i, _i, _i, _vp)
_sig("oidnx_conv_release", None, _vp)
_sig("oidnx_plan_tiles", _st, _i, _i, _i, _i, ctypes.POINTER(_i), _i, ctypes.POINTER(_i))
_sig("oidnx_default_overlap", _i)
_sig("oidnx_version", ctypes.c_char_p)

LIBRARY_PATH = _LIB_PATH


class OidnxError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"oidnx status {status}: {message}")
        self.status = status


def _check(status):
    if status != OK:
        raise OidnxError(status, oidnx_last_error())


def _host_ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def oidnx_last_error():
    return _lib.oidnx_last_error().decode()


def oidnx_version():
    return _lib.oidnx_version().decode()


def oidnx_default_overlap():
    return _lib.oidnx_default_overlap()


def oidnx_filter_create(blob, precision=PRECISION_AUTO):
    handle = _vp()
    buf = ctypes.create_string_buffer(bytes(blob), len(blob))
    _check(_lib.oidnx_filter_create(buf, len(blob), precision, ctypes.byref(handle)))
    return handle.value


def oidnx_filter_set_image(f, which, device_ptr, row_stride_bytes=0):
    _check(_lib.oidnx_filter_set_image(f, which, device_ptr, row_stride_bytes))


def oidnx_filter_set_int(f, name, value):
    _check(_lib.oidnx_filter_set_int(f, name.encode(), int(value)))


def oidnx_filter_get_int(f, name):
    v = _i()
    _check(_lib.oidnx_filter_get_int(f, name.encode(), ctypes.byref(v)))
    return v.value


def oidnx_filter_set_float(f, name, value):
    _check(_lib.oidnx_filter_set_float(f, name.encode(), float(value)))


def oidnx_filter_commit(f):
    _check(_lib.oidnx_filter_commit(f))


def oidnx_filter_execute(f, stream=0):
    _check(_lib.oidnx_filter_execute(f, stream))


def oidnx_filter_execute_host(f, color, albedo, normal, output, stream=0):
    _check(_lib.oidnx_filter_execute_host(f, _host_ptr(color), _host_ptr(albedo),
                                          _host_ptr(normal), _host_ptr(output), stream))


def oidnx_filter_execute_host_async(f, color, albedo, normal, output, stream=0):
    """Enqueue only: the arrays must stay alive and unchanged, and `output`
    unread, until oidnx_filter_wait_host(f) returns."""
    _check(_lib.oidnx_filter_execute_host_async(f, _host_ptr(color), _host_ptr(albedo),
                                                _host_ptr(normal), _host_ptr(output), stream))


def oidnx_filter_wait_host(f):
    _check(_lib.oidnx_filter_wait_host(f))


def oidnx_network_execute(f, packed_in, w, h, out, stream=0):
    _check(_lib.oidnx_network_execute(f, packed_in, w, h, out, stream))


def oidnx_network_execute_noalloc(f, packed_in, w, h, out, stream=0):
    """Network forward without device allocation (intermediates in the
    library's fixed 48 MiB device array; limits in oidnx.h)."""
    _check(_lib.oidnx_network_execute_noalloc(f, packed_in, w, h, out, stream))


def oidnx_output_pass(f, net, w, h, color, output, hdr, input_scale, stream=0,
                      color_stride=0, output_stride=0):
    """The output pass on device buffers (net [h][w] float4, colour and
    output float4 images)."""
    _check(_lib.oidnx_output_pass(f, net, w, h, color, color_stride, output, output_stride,
                                  int(hdr), float(input_scale), stream))


def oidnx_filter_sync_status(f):
    _check(_lib.oidnx_filter_sync_status(f))


def oidnx_debug_wait_probe(f, limit_us, stream=0):
    _check(_lib.oidnx_debug_wait_probe(f, int(limit_us), stream))


def oidnx_profile_next(f):
    _check(_lib.oidnx_profile_next(f))


def oidnx_get_profile(f):
    buf = ctypes.create_string_buffer(1 << 16)
    _check(_lib.oidnx_get_profile(f, buf, len(buf)))
    return json.loads(buf.value.decode())


def oidnx_get_resource_info(f):
    buf = ctypes.create_string_buffer(4096)
    _check(_lib.oidnx_get_resource_info(f, buf, len(buf)))
    return json.loads(buf.value.decode())


def oidnx_debug_read_activation(f, layer):
    """Flat float32 array of the stored activation (logical channels)."""
    need = _sz()
    _check(_lib.oidnx_debug_read_activation(f, layer, None, 0, ctypes.byref(need)))
    out = np.empty(need.value // 4, np.float32)
    _check(_lib.oidnx_debug_read_activation(f, layer, out.ctypes.data, out.nbytes,
                                            ctypes.byref(need)))
    return out


def oidnx_filter_release(f):
    _lib.oidnx_filter_release(f)


def oidnx_conv_create(weight, bias, precision=PRECISION_FP16):
    w = np.ascontiguousarray(weight, np.float32)
    b = np.ascontiguousarray(bias, np.float32)
    cout, cin = w.shape[:2]
    handle = _vp()
    _check(_lib.oidnx_conv_create(w.ctypes.data, b.ctypes.data, cout, cin, precision,
                                  ctypes.byref(handle)))
    return handle.value


def oidnx_conv_execute(c, in_ptr, out_ptr, w, h, relu=1, stream=0):
    _check(_lib.oidnx_conv_execute(c, in_ptr, out_ptr, w, h, relu, stream))


def oidnx_conv_release(c):
    _lib.oidnx_conv_release(c)


def oidnx_plan_tiles(width, height, max_tile_size=0, overlap=-1):
    """List of ((in_x, in_y, in_w, in_h), (out_x, out_y, out_w, out_h))."""
    count = _i()
    _check(_lib.oidnx_plan_tiles(width, height, max_tile_size, overlap, None, 0,
                                 ctypes.byref(count)))
    rects = (_i * (8 * max(count.value, 1)))()
    _check(_lib.oidnx_plan_tiles(width, height, max_tile_size, overlap, rects,
                                 count.value, ctypes.byref(count)))
    vals = list(rects)
    return [(tuple(vals[8 * i:8 * i + 4]), tuple(vals[8 * i + 4:8 * i + 8]))
            for i in range(count.value)]


def write_weight_blob(weights, dtype="f32"):
    """Serialise {layer: (OIHW weight, bias)} as an OXW1 blob (see oidnx.h)."""
    code = {"f32": 0, "f16": 1}[dtype]
    npdt = np.float32 if code == 0 else np.float16
    out = [b"OXW1", struct.pack("<II", 1, 2 * len(weights))]
    for name, (w, b) in weights.items():
        for suffix, arr in ((".weight", w), (".bias", b)):
            arr = np.ascontiguousarray(arr, npdt)
            nm = (name + suffix).encode()
            out.append(struct.pack("<I", len(nm)) + nm + b"\0" * ((4 - len(nm) % 4) % 4))
            out.append(struct.pack("<I", arr.ndim) + struct.pack(f"<{arr.ndim}I", *arr.shape))
            data = arr.tobytes()
            out.append(struct.pack("<I", code) + data + b"\0" * ((4 - len(data) % 4) % 4))
    return b"".join(out)

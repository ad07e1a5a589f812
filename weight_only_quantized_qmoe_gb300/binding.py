"""ctypes binding of libqmoe.so (include/qmoe.h).

Argument marshalling only: every function here has the C name and calls the
C entry point of the same name; pointers are passed as integers (device
addresses from ``tensor.data_ptr()``, host addresses from numpy / pinned
tensors) and streams as ``cudaStream_t`` integers.  Every step of the forward
runs in the library's CUDA kernels; there is no Python or CPU fallback, and
loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmoe.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "qmoe.h")

QMOE_OK, QMOE_ERR_INVALID_ARG, QMOE_ERR_UNSUPPORTED, QMOE_ERR_CUDA = 0, 1, 2, 3
QMOE_ERR_OOM, QMOE_ERR_STATE, QMOE_ERR_TIMEOUT = 4, 5, 6
QMOE_ZP_SYMMETRIC, QMOE_ZP_UINT8, QMOE_ZP_OFFSET = 0, 1, 2
QMOE_ACT_SWIGLU, QMOE_ACT_GEGLU_TANH = 0, 1
QMOE_ACT_RELU, QMOE_ACT_GELU_TANH, QMOE_ACT_SILU, QMOE_ACT_IDENTITY = 2, 3, 4, 5
QMOE_FC1_CONCAT, QMOE_FC1_INTERLEAVED, QMOE_FC1_SEPARATE_FC3 = 0, 1, 2
QMOE_F32, QMOE_F16, QMOE_BF16 = 0, 1, 2
QMOE_TRACE_NUM_EVENTS = 5
QMOE_PATH_NONE, QMOE_PATH_SEPARATE, QMOE_PATH_FUSED = 0, 1, 2
QMOE_FUSED_OFF, QMOE_FUSED_ON, QMOE_FUSED_AUTO = 0, 1, 2
QMOE_COMBINE_REDUCE, QMOE_COMBINE_ORDERED, QMOE_COMBINE_AUTO = 0, 1, 2

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_SIGS = {
    "qmoe_create": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_p)]),
    "qmoe_set_routing": (_i, [_p, _i]),
    "qmoe_set_zero_point_offset": (_i, [_p, ctypes.c_float]),
    "qmoe_set_gemm_min_rows": (_i, [_p, _i]),
    "qmoe_set_fused_decode": (_i, [_p, _i]),
    "qmoe_last_forward_path": (_i, [_p]),
    "qmoe_set_deterministic": (_i, [_p, _i]),
    "qmoe_set_swiglu_params": (_i, [_p, ctypes.c_float, ctypes.c_float, ctypes.c_float]),
    "qmoe_set_fc1_layout": (_i, [_p, _i]),
    "qmoe_set_bias": (_i, [_p, _i, _p, _p]),
    "qmoe_reserve": (_i, [_p, _i64]),
    "qmoe_prepack": (_i, [_p, _i, _p, _p, _p, _p]),
    "qmoe_forward": (_i, [_p, _p, _p, _p, _i64, _p]),
    "qmoe_forward_host": (_i, [_p, _p, _p, _p, _i64, _p]),
    "qmoe_get_routing": (_i, [_p, _p, _p, _p, _p, _p]),
    "qmoe_get_worklist": (_i, [_p, _i, _p, _p, _i64, ctypes.POINTER(_i), _p]),
    "qmoe_worklist_capacity": (_i64, [_p, _i, _i64]),
    "qmoe_set_trace_events": (_i, [_p, ctypes.POINTER(_p), _i]),
    "qmoe_poll_device_status": (_i, [_p]),
    "qmoe_set_wait_limit": (_i, [_p, _i64]),
    "qmoe_debug_inject_stall": (_i, [_p, _i]),
    "qmoe_forward_noalloc": (_i, [_p, _p, _p, _p, _i64, _p]),
    "qmoe_last_error": (ctypes.c_char_p, [_p]),
    "qmoe_status_string": (ctypes.c_char_p, [_i]),
    "qmoe_destroy": (None, [_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libqmoe.so (raises if it is missing: no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with weight_only_quantized_qmoe_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def header_functions() -> list:
    """Names of the functions declared in include/qmoe.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmoe_[a-z_0-9]+)\s*\(", text)))


# --- same-name wrappers -----------------------------------------------------
def qmoe_create(hidden, inter, experts, top_k, bits_fc1, bits_fc2, block_size, zp_mode,
                activation, dtype):
    """Returns (status, layer_handle)."""
    h = _p()
    st = load().qmoe_create(hidden, inter, experts, top_k, bits_fc1, bits_fc2, block_size,
                            zp_mode, activation, dtype, ctypes.byref(h))
    return st, h.value


def qmoe_set_routing(layer, normalize):
    return load().qmoe_set_routing(layer, int(normalize))


def qmoe_set_zero_point_offset(layer, offset):
    return load().qmoe_set_zero_point_offset(layer, float(offset))


def qmoe_set_gemm_min_rows(layer, min_rows):
    return load().qmoe_set_gemm_min_rows(layer, int(min_rows))


def qmoe_set_fused_decode(layer, mode):
    return load().qmoe_set_fused_decode(layer, int(mode))


def qmoe_set_deterministic(layer, mode):
    return load().qmoe_set_deterministic(layer, int(mode))


def qmoe_last_forward_path(layer):
    return load().qmoe_last_forward_path(layer)


def qmoe_set_swiglu_params(layer, alpha, beta, limit):
    return load().qmoe_set_swiglu_params(layer, float(alpha), float(beta), float(limit))


def qmoe_set_fc1_layout(layer, layout):
    return load().qmoe_set_fc1_layout(layer, int(layout))


def qmoe_set_bias(layer, fc, bias_dev, stream=None):
    return load().qmoe_set_bias(layer, int(fc), bias_dev, stream)


def qmoe_reserve(layer, max_tokens):
    return load().qmoe_reserve(layer, int(max_tokens))


def qmoe_prepack(layer, fc, codes, scales, zero_points, stream):
    return load().qmoe_prepack(layer, fc, codes, scales, zero_points or None, stream or None)


def qmoe_forward(layer, x, logits, out, num_tokens, stream):
    return load().qmoe_forward(layer, x, logits, out, int(num_tokens), stream or None)


def qmoe_forward_host(layer, x_host, logits_host, out_host, num_tokens, stream):
    return load().qmoe_forward_host(layer, x_host, logits_host, out_host, int(num_tokens),
                                    stream or None)


def qmoe_forward_noalloc(layer, x, logits, out, num_tokens, stream):
    """The forward for callers that may not allocate device memory: its
    workspace is the library's static scratch array (see include/qmoe.h)."""
    return load().qmoe_forward_noalloc(layer, x, logits, out, int(num_tokens), stream or None)


def qmoe_get_routing(layer, ids, weights, perm, offsets, stream):
    return load().qmoe_get_routing(layer, ids or None, weights or None, perm or None,
                                   offsets or None, stream or None)


def qmoe_get_worklist(layer, which, items, count, capacity, stream):
    """Returns (status, m_tile)."""
    m = _i(0)
    st = load().qmoe_get_worklist(layer, which, items or None, count or None, int(capacity),
                                  ctypes.byref(m), stream or None)
    return st, m.value


def qmoe_worklist_capacity(layer, which, num_tokens):
    return load().qmoe_worklist_capacity(layer, which, int(num_tokens))


def qmoe_set_trace_events(layer, events):
    """events: list of QMOE_TRACE_NUM_EVENTS cudaEvent_t handles, or None."""
    if events is None:
        return load().qmoe_set_trace_events(layer, None, 0)
    arr = (_p * len(events))(*events)
    return load().qmoe_set_trace_events(layer, arr, len(events))


def qmoe_poll_device_status(layer):
    return load().qmoe_poll_device_status(layer)


def qmoe_set_wait_limit(layer, iterations):
    return load().qmoe_set_wait_limit(layer, int(iterations))


def qmoe_debug_inject_stall(layer, enable):
    return load().qmoe_debug_inject_stall(layer, int(enable))


def qmoe_last_error(layer):
    return load().qmoe_last_error(layer).decode()


def qmoe_status_string(status):
    return load().qmoe_status_string(status).decode()


def qmoe_destroy(layer):
    load().qmoe_destroy(layer)

"""Python binding of the GB300 MXFP8 DSV3-style MoE layer library (libmoe_gb300.so).

Argument marshalling only: every function forwards to the C entry point of
the same name in ``include/moe.h``. Device buffers are passed as integer
device addresses (e.g. ``tensor.data_ptr()``), streams as integer
``cudaStream_t`` handles (0 = legacy default stream). Every step of the layer
runs in the library's CUDA kernels; there is no fallback path. Importing
this package fails loudly if the library has not been built
(``python -m moe_layer_dsv3_gb300.build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libmoe_gb300.so is not built (%s). Build it with `python -m moe_layer_dsv3_gb300.build`." % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_ARCH = 2
MOE_ERR_CUDA = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_BOUNDS = 6
MOE_ERR_SCRATCH = 7

WS_NAMES = ["STATUS", "META", "COUNTS", "OFFSETS", "POFF", "RANK", "POS", "INV", "ROWSRC", "LAPTILES", "HIST",
            "BASE", "LOGITS", "SSEL", "XQ", "XQ_SF", "RING_X", "RING_X_SF", "GU", "HQ", "HQ_SF", "HTOK", "HTOK_SF",
            "O", "DW", "DL", "RING_DO", "RING_DO_SF", "DOS", "DOS_SF", "DOTOK", "DOTOK_SF", "DGU", "DGU_SF",
            "DGUTOK", "DGUTOK_SF", "XTOK", "XTOK_SF", "DXE", "DWR_PART", "ORDER",
            "LAPBASE", "MOVED", "CONSUMED", "DH", "LAPORDER", "LAPKEY", "XQ_SFC", "DOS_SFC",
            "RINGINFO", "PUSHINFO", "WGINFO"]
WS = {n: i for i, n in enumerate(WS_NAMES)}
WQ_NAMES = ["W1F", "W1F_SF", "W2F", "W2F_SF", "W2B", "W2B_SF", "W1B", "W1B_SF"]
WQ = {n: i for i, n in enumerate(WQ_NAMES)}


class MoeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("T", "d", "E", "k", "n_groups", "topk_groups", "I", "n_shared", "capacity", "flags",
                 "n_mover_warps")]


class MoeError(RuntimeError):
    def __init__(self, name: str, code: int):
        super().__init__("%s failed with MOE error %d" % (name, code))
        self.code = code


_P = ctypes.c_void_p
_I = ctypes.c_int
_CFG = ctypes.POINTER(MoeConfig)
_SZ = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "moe_workspace_size": [_CFG, _SZ],
    "moe_weights_size": [_CFG, _SZ],
    "moe_quantize_mxfp8": [_P, _I, _I, _I, _P, _P, _P],
    "moe_quantize_weights": [_CFG, _P, _P, _P, _P, _P, _P],
    "moe_route": [_CFG, _P, _P, _P, _P, _P, _P, _P],
    "moe_route_noalloc": [_CFG, _P, _P, _P, _P, _P, _P],
    "moe_schedule": [_CFG, _P, _P, _P],
    "moe_forward": [_CFG, _P, _P, _P, _P, _P, _P],
    "moe_dispatch": [_CFG, _P, _P, _P],
    "moe_backward": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_status": [_CFG, _P, ctypes.POINTER(_I), ctypes.POINTER(_I), _I, _P],
    "moe_ws_view": [_CFG, _P, _I, ctypes.POINTER(_P), _SZ],
    "moe_wq_view": [_CFG, _P, _I, ctypes.POINTER(_P), _SZ],
    "moe_gemm_mxfp8": [_I, _I, _I, _P, _P, _P, _P, _P, _P],
    "moe_gemm_mxfp8_pair": [_I, _I, _I, _P, _P, _P, _P, _P, _P],
    "moe_quantize_nvfp4": [_P, _I, _I, ctypes.c_float, _P, _P, _I, _P],
    "moe_gemm_nvfp4": [_I, _I, _I, _P, _P, _P, _P, ctypes.c_float, _P, _P],
    "moe_expert_gemm_nvfp4": [_CFG, _I, _I, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P],
    "moe_expert_gemm_nvfp4_push": [_CFG, _I, _I, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P],
    "moe_scales_to_tiled": [_P, _I, _I, _P, _P],
    "moe_profile_enable": [_I],
    "moe_profile_read": [ctypes.c_void_p, _I, ctypes.POINTER(_I)],
    "moe_profile_trace": [ctypes.c_void_p, _I, ctypes.POINTER(_I)],
    "moe_launch_count": [],
    "moe_selftest_wait_timeout": [_P, ctypes.c_ulonglong, _P],
    "moe_debug_fail_tensor_maps": [_I],
}
for _name, _args in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_longlong if _name == "moe_launch_count" else ctypes.c_int


class MoeKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("ms", ctypes.c_double)]


def exported_symbols():
    return list(_SIGS)


def _check(name: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(name, rc)


def _p(x):
    return None if x is None or x == 0 else ctypes.c_void_p(int(x))


MOE_FLAG_LAP_LAUNCHES = 1   # one mover launch + one GEMM launch per ring lap instead of one launch for all laps
MOE_FLAG_WGRAD_PAIR = 2     # weight gradients on CTA pairs (256-row tiles) instead of single-CTA 128 x 256 tiles


def config(T, d, E, k, n_groups=1, topk_groups=1, I=128, n_shared=0, capacity=0, flags=0,
           n_mover_warps=0) -> MoeConfig:
    return MoeConfig(T, d, E, k, n_groups, topk_groups, I, n_shared, capacity, flags, n_mover_warps)


def moe_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size", _lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_weights_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t()
    _check("moe_weights_size", _lib.moe_weights_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_quantize_mxfp8(src, rows, K, axis, codes, scales, stream=0):
    _check("moe_quantize_mxfp8", _lib.moe_quantize_mxfp8(_p(src), rows, K, axis, _p(codes), _p(scales), _p(stream)))


def moe_quantize_weights(cfg, w_gu, w_d, ws_gu, ws_d, wq, stream=0):
    _check("moe_quantize_weights",
           _lib.moe_quantize_weights(ctypes.byref(cfg), _p(w_gu), _p(w_d), _p(ws_gu), _p(ws_d), _p(wq), _p(stream)))


def moe_route(cfg, x, w_router, bias, topk_idx, topk_w, ws, stream=0):
    _check("moe_route", _lib.moe_route(ctypes.byref(cfg), _p(x), _p(w_router), _p(bias), _p(topk_idx), _p(topk_w),
                                       _p(ws), _p(stream)))


def moe_route_noalloc(cfg, x, w_router, bias, topk_idx, topk_w, stream=0):
    """moe_route with its logits in the library's fixed device scratch (no workspace, no allocation)."""
    _check("moe_route_noalloc", _lib.moe_route_noalloc(ctypes.byref(cfg), _p(x), _p(w_router), _p(bias),
                                                       _p(topk_idx), _p(topk_w), _p(stream)))


def moe_schedule(cfg, topk_idx, ws, stream=0):
    _check("moe_schedule", _lib.moe_schedule(ctypes.byref(cfg), _p(topk_idx), _p(ws), _p(stream)))


def moe_forward(cfg, x, wq, topk_w, y, ws, stream=0):
    _check("moe_forward", _lib.moe_forward(ctypes.byref(cfg), _p(x), _p(wq), _p(topk_w), _p(y), _p(ws), _p(stream)))


def moe_dispatch(cfg, x, ws, stream=0):
    _check("moe_dispatch", _lib.moe_dispatch(ctypes.byref(cfg), _p(x), _p(ws), _p(stream)))


def moe_backward(cfg, x, w_router, topk_idx, topk_w, dy, wq, dx, dw_router, dw_gu, dw_d, dws_gu, dws_d, ws, stream=0):
    _check("moe_backward",
           _lib.moe_backward(ctypes.byref(cfg), _p(x), _p(w_router), _p(topk_idx), _p(topk_w), _p(dy), _p(wq), _p(dx),
                             _p(dw_router), _p(dw_gu), _p(dw_d), _p(dws_gu), _p(dws_d), _p(ws), _p(stream)))


def moe_status(cfg, ws, clear=True, stream=0):
    code, site = ctypes.c_int(), ctypes.c_int()
    _check("moe_status", _lib.moe_status(ctypes.byref(cfg), _p(ws), ctypes.byref(code), ctypes.byref(site),
                                         1 if clear else 0, _p(stream)))
    return code.value, site.value


def moe_ws_view(cfg, ws, which):
    ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
    w = WS[which] if isinstance(which, str) else which
    _check("moe_ws_view", _lib.moe_ws_view(ctypes.byref(cfg), _p(ws), w, ctypes.byref(ptr), ctypes.byref(n)))
    return ptr.value or 0, n.value


def moe_wq_view(cfg, wq, which):
    ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
    w = WQ[which] if isinstance(which, str) else which
    _check("moe_wq_view", _lib.moe_wq_view(ctypes.byref(cfg), _p(wq), w, ctypes.byref(ptr), ctypes.byref(n)))
    return ptr.value or 0, n.value


def moe_gemm_mxfp8(M, N, K, a, a_sf, b, b_sf, c, stream=0):
    _check("moe_gemm_mxfp8", _lib.moe_gemm_mxfp8(M, N, K, _p(a), _p(a_sf), _p(b), _p(b_sf), _p(c), _p(stream)))


def moe_gemm_mxfp8_pair(M, N, K, a, a_sf, b, b_sf, c, stream=0):
    _check("moe_gemm_mxfp8_pair",
           _lib.moe_gemm_mxfp8_pair(M, N, K, _p(a), _p(a_sf), _p(b), _p(b_sf), _p(c), _p(stream)))


def moe_quantize_nvfp4(src, rows, K, g, codes, scales, tiled=True, stream=0):
    _check("moe_quantize_nvfp4",
           _lib.moe_quantize_nvfp4(_p(src), rows, K, float(g), _p(codes), _p(scales), int(bool(tiled)), _p(stream)))


def moe_expert_gemm_nvfp4(cfg, N, K, a, a_sf, w, w_sf, alpha, out, ws, stream=0):
    _check("moe_expert_gemm_nvfp4",
           _lib.moe_expert_gemm_nvfp4(ctypes.byref(cfg), N, K, _p(a), _p(a_sf), _p(w), _p(w_sf), float(alpha),
                                      _p(out), _p(ws), _p(stream)))


def moe_expert_gemm_nvfp4_push(cfg, N, K, a, a_sf, w, w_sf, alpha, out, ws, stream=0):
    _check("moe_expert_gemm_nvfp4_push",
           _lib.moe_expert_gemm_nvfp4_push(ctypes.byref(cfg), N, K, _p(a), _p(a_sf), _p(w), _p(w_sf), float(alpha),
                                           _p(out), _p(ws), _p(stream)))


def moe_gemm_nvfp4(M, N, K, a, a_sf, b, b_sf, alpha, c, stream=0):
    _check("moe_gemm_nvfp4",
           _lib.moe_gemm_nvfp4(M, N, K, _p(a), _p(a_sf), _p(b), _p(b_sf), float(alpha), _p(c), _p(stream)))


def moe_scales_to_tiled(canon, rows, K, tiled, stream=0):
    _check("moe_scales_to_tiled", _lib.moe_scales_to_tiled(_p(canon), rows, K, _p(tiled), _p(stream)))


def moe_profile_enable(enable=True):
    _check("moe_profile_enable", _lib.moe_profile_enable(1 if enable else 0))


def moe_profile_read(max_entries=64):
    """{kernel name: (launches, total ms)} of the launches recorded since the last read."""
    buf = (MoeKernelTime * max_entries)()
    n = ctypes.c_int()
    _check("moe_profile_read", _lib.moe_profile_read(ctypes.cast(buf, ctypes.c_void_p), max_entries, ctypes.byref(n)))
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms) for i in range(min(n.value, max_entries))}


class MoeKernelSpan(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("start_ms", ctypes.c_double), ("end_ms", ctypes.c_double)]


def moe_profile_trace(max_entries=4096):
    """[(kernel name, start ms, end ms)] of the launches recorded since the last read, in issue order."""
    buf = (MoeKernelSpan * max_entries)()
    n = ctypes.c_int()
    _check("moe_profile_trace", _lib.moe_profile_trace(ctypes.cast(buf, ctypes.c_void_p), max_entries,
                                                       ctypes.byref(n)))
    return [(buf[i].name.decode(), buf[i].start_ms, buf[i].end_ms) for i in range(min(n.value, max_entries))]


def moe_selftest_wait_timeout(status, limit_ns, stream=0):
    _check("moe_selftest_wait_timeout", _lib.moe_selftest_wait_timeout(_p(status), limit_ns, _p(stream)))


def moe_debug_fail_tensor_maps(count):
    """Make the next `count` tensor-map encodings fail on the host (0 clears); tests only."""
    _check("moe_debug_fail_tensor_maps", _lib.moe_debug_fail_tensor_maps(int(count)))


def moe_launch_count():
    return int(_lib.moe_launch_count())

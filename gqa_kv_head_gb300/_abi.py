"""ctypes declarations of the C ABI in include/fr_kernels.h.

Loading fails loudly when the shared library has not been built: there is no
fallback implementation anywhere in this package.
"""
import ctypes
import os

from . import build as _build

FR_OK = 0
STATUS_NAMES = {0: "FR_OK", 1: "FR_ERR_INVALID_ARG", 2: "FR_ERR_UNSUPPORTED",
                3: "FR_ERR_WORKSPACE", 4: "FR_ERR_CUDA", 5: "FR_ERR_DEVICE_TIMEOUT"}


class FrError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


FR_ROPE_EXACT = 0
FR_ROPE_GGML_F32 = 1


class FrRopeParams(ctypes.Structure):
    _fields_ = [("n_dims", ctypes.c_int), ("freq_base", ctypes.c_float),
                ("freq_scale", ctypes.c_float), ("ext_factor", ctypes.c_float),
                ("attn_factor", ctypes.c_float), ("beta_fast", ctypes.c_float),
                ("beta_slow", ctypes.c_float), ("n_ctx_orig", ctypes.c_int),
                ("mode", ctypes.c_int), ("freq_factors", ctypes.POINTER(ctypes.c_float))]


class FrAttnOpts(ctypes.Structure):
    _fields_ = [("engine", ctypes.c_int), ("force_splits", ctypes.c_int),
                ("force_cluster", ctypes.c_int), ("wait_probe_iters", ctypes.c_int),
                ("merge_mode", ctypes.c_int), ("layout", ctypes.c_int), ("slice_rows", ctypes.c_int)]


class FrAttnPlan(ctypes.Structure):
    _fields_ = [("engine", ctypes.c_int), ("row_tiles", ctypes.c_int), ("splits", ctypes.c_int),
                ("cluster", ctypes.c_int), ("merge_kernel", ctypes.c_int), ("launches", ctypes.c_int),
                ("keys_on_m", ctypes.c_int), ("layout", ctypes.c_int), ("row_slices", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_RP = ctypes.POINTER(FrRopeParams)

_ATTN_ARGS = [_P, _P, _I64, _P, _RP, _F, _P, _I64, _P, _I64, _P, _I64,
              _I, _I, _I, _I, _F, _P, _P, _SZ]

SIGNATURES = {
    "fr_status_string": (ctypes.c_char_p, [_I]),
    "fr_abi_version": (_I, []),
    "fr_qkv_post": (_I, [_P, _I64, _P, _I, _I, _I, _RP, _F, _P, _P, _P]),
    "fr_decode_attn_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "fr_workspace_init": (_I, [_P, _SZ, _P]),
    "fr_workspace_check": (_I, [_P, _P]),
    "fr_decode_attn": (_I, _ATTN_ARGS + [_P]),
    "fr_decode_attn_ex": (_I, _ATTN_ARGS + [ctypes.POINTER(FrAttnOpts), _P]),
    "fr_decode_attn_noalloc": (_I, _ATTN_ARGS[:18] + [_P]),
    "fr_decode_attn_noalloc_check": (_I, [_P]),
    "fr_kv_append": (_I, [_P, _I64, _P, _I64, _P, _I, _I, _RP, _P, _I64, _P, _I64, _I64, _I64, _I64, _I64,
                          _P, _P, _P]),
    "fr_decode_attn_plan": (_I, [_I, _I, _I, _I, _I, _SZ, ctypes.POINTER(FrAttnOpts),
                                 ctypes.POINTER(FrAttnPlan)]),
}

_lib = None


def library_path(trace=False):
    return _build.library_path(trace)


def load(trace=False):
    """The loaded library (ctypes.CDLL) with argument types declared. The first
    call decides which build the process uses: trace=True loads the
    timeline-instrumented variant (gqa_kv_head_gb300.trace)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path(trace)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with gqa_kv_head_gb300.build.build() "
                           "(needs nvcc); this package has no non-CUDA fallback")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status, where):
    if status != FR_OK:
        raise FrError(status, where)

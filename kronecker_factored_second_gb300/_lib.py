"""ctypes binding of libokls.so (argument marshalling only).

Every function here forwards to the C ABI declared in include/okls.h under
the same name.  There is no fallback: if the shared library is missing the
import of this module's `lib()` raises.
"""

from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libokls.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "okls.h")

OKLS_OK = 0
OKLS_ERR_INVALID_ARG = 1
OKLS_ERR_UNSUPPORTED = 2
OKLS_ERR_CUDA = 3
OKLS_ERR_NONFINITE = 4
OKLS_ERR_TIMEOUT = 5
OKLS_ERR_NO_DEVICE = 6

OKLS_F32 = 0
OKLS_BF16 = 1

METHOD_OKLS = 0
METHOD_SHAMPOO = 1
METHOD_SOAP = 2
METHOD_CLEAN = 3

STATE_M, STATE_SA, STATE_SB, STATE_PA, STATE_PB, STATE_V = range(6)
STATE_MA, STATE_MB, STATE_VA, STATE_VB, STATE_VC = range(6, 11)

DEV_NONFINITE_INPUT = 0x1
DEV_NONFINITE_ITER = 0x2
DEV_NONFINITE_UPDATE = 0x4
DEV_TIMEOUT = 0x8


class okls_config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("m", ctypes.c_int64),
        ("n", ctypes.c_int64),
        ("param_dtype", ctypes.c_int32),
        ("grad_dtype", ctypes.c_int32),
        ("lr_peak", ctypes.c_float),
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("weight_decay", ctypes.c_float),
        ("ns_iters", ctypes.c_int32),
        ("ns_split_iters", ctypes.c_int32),
        ("ns_lo", ctypes.c_float),
        ("ridge", ctypes.c_float),
        ("variance_correction", ctypes.c_int32),
        ("eps_every_update", ctypes.c_int32),
        ("root_every", ctypes.c_int32),
        ("method", ctypes.c_int32),
        ("rank", ctypes.c_int32),
        ("oversample", ctypes.c_int32),
        ("power_iters", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 3),
    ]


class okls_profile(ctypes.Structure):
    _fields_ = [
        ("kernel_launches", ctypes.c_int64),
        ("gemm_launches", ctypes.c_int64),
        ("gemm_flops", ctypes.c_double),
        ("gemm_ms", ctypes.c_double),
        ("timed_launches", ctypes.c_int64),
        ("ns_launches", ctypes.c_int64),
        ("ns_flops", ctypes.c_double),
        ("ns_ms", ctypes.c_double),
        ("bw_launches", ctypes.c_int64),
        ("bw_bytes", ctypes.c_double),
        ("bw_ms", ctypes.c_double),
        ("bw_timed_launches", ctypes.c_int64),
    ]


class OklsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"okls error {code}: {msg}")
        self.code = code


_LIB = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGS = {
    "okls_abi_version": (_I32, []),
    "okls_last_error": (ctypes.c_char_p, []),
    "okls_config_default": (_I32, [ctypes.POINTER(okls_config), _I64, _I64, _I64]),
    "okls_state_bytes": (_I32, [ctypes.POINTER(okls_config), ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "okls_create": (_I32, [ctypes.POINTER(okls_config), _P, _SZ, _P, _SZ, ctypes.POINTER(_P)]),
    "okls_reset_state": (_I32, [_P, _P]),
    "okls_step": (_I32, [_P, _P, _P, _F, _P]),
    "okls_step_noise": (_I32, [_P, _P, _P, _F, _P, _P]),
    "okls_query_status": (_I32, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "okls_get_state": (_I32, [_P, _I32, _P, _P]),
    "okls_set_state": (_I32, [_P, _I32, _P, _P]),
    "okls_get_step": (_I32, [_P, ctypes.POINTER(_I64)]),
    "okls_set_step": (_I32, [_P, _I64]),
    "okls_destroy": (_I32, [_P]),
    "okls_profile_enable": (_I32, [_P, _I32]),
    "okls_set_wait_limit": (_I32, [_P, _I64, _I64]),
    "okls_profile_read": (_I32, [_P, ctypes.POINTER(okls_profile)]),
    "okls_ns_schedule": (_I32, [_I32, ctypes.c_double, ctypes.POINTER(ctypes.c_double),
                                ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I32)]),
    "okls_inv_root_workspace_bytes": (_I32, [_I64, _I64, _I32, _I32, ctypes.POINTER(_SZ)]),
    "okls_inv_root": (_I32, [_P, _P, _P, _P, _I64, _I64, _I32, _I32, _F, _F, _P, _SZ, _P]),
    "okls_inv_root_noalloc_capacity": (_SZ, []),
    "okls_inv_root_noalloc": (_I32, [_P, _P, _I64, _I64, _I32, _I32, _F, _F, _P]),
}


def header_functions() -> list[str]:
    """Names of the functions include/okls.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(okls_[a-z0-9_]+)\s*\(", text)))


def lib():
    """The loaded library (raises ImportError when it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing; build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def last_error() -> str:
    return lib().okls_last_error().decode(errors="replace")


def check(code: int) -> None:
    if code != OKLS_OK:
        raise OklsError(code, last_error())


def config_default(batch: int, m: int, n: int) -> okls_config:
    c = okls_config()
    check(lib().okls_config_default(ctypes.byref(c), batch, m, n))
    return c


def state_bytes(cfg: okls_config) -> tuple[int, int]:
    s, w = _SZ(0), _SZ(0)
    check(lib().okls_state_bytes(ctypes.byref(cfg), ctypes.byref(s), ctypes.byref(w)))
    return s.value, w.value


def ns_schedule(iters: int, lo: float):
    a = (ctypes.c_double * iters)()
    b = (ctypes.c_double * iters)()
    z = (_I32 * (iters + 1))()
    check(lib().okls_ns_schedule(iters, lo, a, b, z))
    return list(a), list(b), list(z)

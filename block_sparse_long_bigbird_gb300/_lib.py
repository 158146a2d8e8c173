"""ctypes binding of ``libsparse_attn.so`` (the C ABI in include/sparse_attn.h).

Argument marshalling only: every step of the attention forward and backward runs in the
library's CUDA kernels. There is no fallback: if the compiled library is
missing, every call raises.
"""

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsparse_attn.so")

SA_OK = 0
SA_ERR_INVALID_ARG = 1
SA_ERR_UNSUPPORTED = 2
SA_ERR_CUDA = 3
SA_ERR_TIMEOUT = 4
SA_ERR_BAD_INDEX = 5
STATUS_NAMES = {
    0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_CUDA",
    4: "SA_ERR_TIMEOUT", 5: "SA_ERR_BAD_INDEX",
}

SA_BF16 = 0
SA_FP32 = 1

SA_OPT_FORCE_SIMT = 1
SA_OPT_WAIT_LIMIT = 2
SA_OPT_MAX_SPLITS = 3
SA_OPT_GRID_CTAS = 4
SA_OPT_CHUNK_KEYS = 5

# Exported symbol -> (restype, argtypes).
_VP = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "build_bigbird_pattern": (_I, [ctypes.c_uint64, _I, _I, _I, _I, _I, _I, _VP]),
    "bigbird_attn_fwd": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _I, _VP, _VP, _I, _VP]),
    "longformer_attn_fwd": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP]),
    "longformer_attn_fwd_ex": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP, _I, _VP]),
    "longformer_attn_fwd_gproj": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP,
                                       _I, _VP]),
    "bigbird_attn_fwd_host": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _I, _VP, _VP, _I, _VP]),
    "longformer_attn_fwd_host": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP, _I, _VP]),
    "bigbird_attn_bwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _I, _VP, _VP, _I,
                              _VP]),
    "longformer_attn_bwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP, _I,
                                 _VP]),
    "longformer_attn_bwd_gproj": (_I, [_VP] * 13 + [_I, _I, _I, _I, _I, _VP, _I, _VP, _I, _VP, _I, _VP]),
    "sa_attn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "sa_bigbird_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "sa_longformer_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "sa_set_workspace": (_I, [_VP, ctypes.c_size_t]),
    "sa_get_last_device_status": (_I, [_VP]),
    "sa_status_string": (ctypes.c_char_p, [_I]),
    "sa_set_option": (_I, [_I, ctypes.c_int64]),
    "sa_last_launch_count": (_I, []),
    "bigbird_attn_fwd_noalloc": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _I, _VP, _VP, _VP]),
    "sa_check_wait_expiry": (_I, [ctypes.c_int64, _VP]),
}
NOALLOC_SCRATCH_BYTES = 16 << 20

_lock = threading.Lock()
_lib = None


class SparseAttnError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)}")


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -c 'import __graft_entry__ as g; g.build()'`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def check(status, what):
    if status != SA_OK:
        raise SparseAttnError(status, what)
    return status

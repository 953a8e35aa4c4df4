"""ctypes declarations of the C ABI in include/mla.h (no logic of the method here)."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_gb300.so")

MLA_F32, MLA_BF16 = 0, 1
STATUS = {0: "MLA_OK", 1: "MLA_ERR_NULL", 2: "MLA_ERR_SHAPE", 3: "MLA_ERR_DTYPE",
          4: "MLA_ERR_ALIGN", 5: "MLA_ERR_WORKSPACE", 6: "MLA_ERR_CUDA", 7: "MLA_ERR_TIMEOUT",
          8: "MLA_ERR_UNSUPPORTED"}
OPT_ATTN_PATH, OPT_KV_SPLITS, OPT_PREFILL_FUSED, OPT_NUM_SMS, OPT_PERSISTENT = 0, 1, 2, 3, 4

_lock = threading.Lock()
_lib = None

_vp, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

SIGNATURES = {
    "mla_kv_latent_project": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i, _i, _i, _i, _i, _vp]),
    "mla_latent_attention_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "mla_latent_attention_kv_splits": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "mla_latent_attention": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _i,
                                  _vp, _sz, _vp]),
    "mla_latent_attention_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f,
                                          _i, _i, _i, _vp]),
    "mla_latent_attention_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                         _i, _i, _f, _i, _i, _i, _vp]),
    "mla_explicit_attention": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp]),
    "mla_merge_partials": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "mla_get_device_error": (_i, [ctypes.POINTER(ctypes.c_uint), _i]),
    "mla_set_option": (_i, [_i, _i64]),
    "mla_status_string": (ctypes.c_char_p, [_i]),
    "mla_set_stage_events": (_i, [ctypes.POINTER(ctypes.c_void_p), _i]),
    "mla_launch_count": (ctypes.c_uint64, []),
    "mla_check_wait_timeout": (_i, [ctypes.c_uint, _vp]),
}


class MLAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the built library; raises if it has not been built (there is no
    fallback implementation)."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; build it with "
                "`python -m latent_causal_attention_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path == LIB_PATH:
            _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != 0:
        raise MLAError(fn, status)

"""ctypes view of libttt_mlp.so (the C ABI in include/ttt_mlp.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Loading fails loudly when the shared library has not been built;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libttt_mlp.so")

TTT_OK, TTT_EINVAL, TTT_EUNSUPPORTED, TTT_ECUDA, TTT_ETIMEOUT, TTT_EFAULT_INJECTED = range(6)
STATUS_NAMES = {0: "TTT_OK", 1: "TTT_EINVAL", 2: "TTT_EUNSUPPORTED", 3: "TTT_ECUDA",
                4: "TTT_ETIMEOUT", 5: "TTT_EFAULT_INJECTED"}
TTT_F32, TTT_BF16 = 0, 1
TTT_TARGET_NEXT, TTT_TARGET_CURRENT, TTT_TARGET_CAUSAL = 0, 1, 2
NOALLOC_SCRATCH_BYTES = 32 << 20  # TTT_NOALLOC_SCRATCH_BYTES in the header


class Config(C.Structure):
    _fields_ = [("d", C.c_int32), ("f", C.c_int32), ("chunk", C.c_int32), ("conv_k", C.c_int32),
                ("n_docs", C.c_int32), ("eta", C.c_float), ("act_dtype", C.c_int32),
                ("max_tokens", C.c_int64), ("target_mode", C.c_int32), ("clip_tau", C.c_float)]


_vp = C.c_void_p
_i32 = C.c_int32
_i64 = C.c_int64
_st = C.c_int

# name -> (restype, argtypes); the full exported surface of the header
SIGNATURES = {
    "ttt_mlp_workspace_bytes": (C.c_size_t, [C.POINTER(Config)]),
    "ttt_mlp_create": (_st, [C.POINTER(Config), _vp, _vp, _vp, _vp, _vp, _vp, C.c_size_t, _vp,
                             C.POINTER(_vp)]),
    "ttt_mlp_state_bytes": (C.c_size_t, [C.POINTER(Config)]),
    "ttt_mlp_scratch_bytes": (C.c_size_t, [C.POINTER(Config)]),
    "ttt_mlp_create_split": (_st, [C.POINTER(Config), _vp, _vp, _vp, _vp, _vp, _vp, C.c_size_t, _vp,
                                   C.c_size_t, _vp, C.POINTER(_vp)]),
    "ttt_mlp_forward_chunks": (_st, [_vp, _i32, _vp, _vp, _i64, C.POINTER(_i64), _i32, _vp, _vp]),
    "ttt_mlp_forward_static": (_st, [_vp, _vp, _i64, _vp, _vp]),
    "ttt_mlp_forward_chunks_host": (_st, [_vp, _i32, _vp, _vp, _i64, C.POINTER(_i64), _i32, _vp,
                                          _vp]),
    "ttt_mlp_reset": (_st, [_vp, _i32, _vp]),
    "ttt_mlp_get_fast_weight": (_st, [_vp, _i32, _vp, _vp]),
    "ttt_mlp_set_fast_weight": (_st, [_vp, _i32, _vp, _vp]),
    "ttt_mlp_check": (_st, [_vp, _vp]),
    "ttt_mlp_destroy": (_st, [_vp]),
    "ttt_mlp_last_error": (C.c_char_p, [_vp]),
    "ttt_mlp_path": (C.c_char_p, [_vp]),
    "ttt_mlp_profile_enable": (_st, [_vp, _i32]),
    "ttt_mlp_profile_read": (_st, [_vp, C.POINTER(C.c_float), C.POINTER(_i64)]),
    "ttt_mlp_intermediates": (_st, [_vp, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_i32)]),
    "ttt_target_noalloc": (_st, [_vp, _vp, _vp, _i64, _i32, _i32, _i32, C.POINTER(_i64), _i32,
                                 C.c_float, _vp, _vp, _vp]),
    "ttt_rmsnorm": (_st, [_vp, _vp, _i64, _i32, C.c_float, _i32, _vp]),
    "ttt_residual_add": (_st, [_vp, _vp, _i64, _i32, _i32, _vp]),
    "ttt_residual_rmsnorm": (_st, [_vp, _vp, _vp, _i64, _i32, C.c_float, _i32, _i32, _vp]),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load the library (once) and declare every exported signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m chunk_wise_weight_ttt_b300.build` "
            "(the layer has no non-CUDA implementation)")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class TTTError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status

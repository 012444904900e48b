"""ctypes view of libgbattn.so: the structures and entry points of include/gbattn.h.

Argument marshalling only.  Loading fails loudly if the library cannot be
built or found; there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_WORKSPACE = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_DEVICE_TIMEOUT = 5
ATTN_ERR_DEVICE_BOUNDS = 6

ATTN_F32 = 0
ATTN_BF16 = 1

ATTN_MASK_NONE = 0
ATTN_MASK_CAUSAL = 1
ATTN_MASK_BLOCK = 2

SIZE_MAX = ctypes.c_size_t(-1).value
NOALLOC_SCRATCH_BYTES = 32 << 20  # ATTN_NOALLOC_SCRATCH_BYTES in include/gbattn.h

I32P = ctypes.POINTER(ctypes.c_int32)


class BlockMaskC(ctypes.Structure):
    _fields_ = [
        ("row_ptr", ctypes.c_void_p),
        ("col_idx", ctypes.c_void_p),
        ("row_ptr_host", ctypes.c_void_p),
        ("col_idx_host", ctypes.c_void_p),
        ("block_q", ctypes.c_int32),
        ("block_k", ctypes.c_int32),
        ("n_row_blocks", ctypes.c_int32),
        ("n_col_blocks", ctypes.c_int32),
        ("nnz", ctypes.c_int32),
        ("causal_in_block", ctypes.c_int32),
    ]


class ParamsC(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("heads_q", ctypes.c_int32),
        ("heads_kv", ctypes.c_int32),
        ("seqlen", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("cu_seqlens_host", ctypes.c_void_p),
        ("n_seqs", ctypes.c_int32),
        ("q_stride_b", ctypes.c_int64),
        ("q_stride_h", ctypes.c_int64),
        ("q_stride_s", ctypes.c_int64),
        ("kv_stride_b", ctypes.c_int64),
        ("kv_stride_h", ctypes.c_int64),
        ("kv_stride_s", ctypes.c_int64),
        ("scale", ctypes.c_float),
        ("dtype", ctypes.c_int32),
        ("mask", ctypes.c_int32),
        ("block_mask", ctypes.POINTER(BlockMaskC)),
    ]


class LnParamsC(ctypes.Structure):
    """ln_params_t of include/gbln.h."""
    _fields_ = [
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("x_stride", ctypes.c_int64),
        ("r_stride", ctypes.c_int64),
        ("y_stride", ctypes.c_int64),
        ("h_stride", ctypes.c_int64),
        ("eps", ctypes.c_float),
        ("dtype", ctypes.c_int32),
    ]


# Every symbol include/gbattn.h and include/gbln.h declare, with its ctypes signature.
_VP = ctypes.c_void_p
_PP = ctypes.POINTER(ParamsC)
SIGNATURES = {
    "attn_fwd_workspace_size": (ctypes.c_size_t, [_PP]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_PP]),
    "attn_fwd": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "attn_bwd": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "attn_bwd_deterministic": (ctypes.c_int,
                               [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "attn_bwd_noalloc": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "attn_quantize_fp8": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "attn_fwd_fp8": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "attn_get_status": (ctypes.c_int, [_VP]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_set_timing_events": (ctypes.c_int, [ctypes.c_int, _VP, _VP]),
    "attn_version": (ctypes.c_char_p, []),
    "attn_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint, _VP]),
    "ln_residual_fwd": (ctypes.c_int, [ctypes.POINTER(LnParamsC), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
}

_lock = threading.Lock()
_lib = None


def checked_mode() -> bool:
    """GBATTN_CHECKED=1 in the environment selects the checked library: every
    device-computed index is compared with its tensor's extent before the access
    (a failure records ATTN_ERR_DEVICE_BOUNDS and skips the access)."""
    return os.environ.get("GBATTN_CHECKED", "0") == "1"


def library_path() -> str:
    return _build.LIB_CHECKED if checked_mode() else _build.LIB


def load(build_if_missing: bool = True):
    """Load libgbattn.so, or libgbattn_checked.so under GBATTN_CHECKED=1 (building
    both first if needed), and set up signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} not found at {path}; "
                               "build it with bwd_flashattention_fwd_sm_gb300.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        name = load().attn_status_string(code).decode()
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


def check(code: int, where: str) -> None:
    if code != ATTN_OK:
        raise AttnError(code, where, load().attn_last_error().decode())

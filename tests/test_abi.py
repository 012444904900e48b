"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/gbattn.h and include/gbln.h declare, and host-side validation rejects bad calls before
any device work.  Valid calls on a machine with no GPU must fail with
ATTN_ERR_CUDA: there is no CPU path behind the ABI."""

import ctypes
import os
import re

import numpy as np
import pytest

from bwd_flashattention_fwd_sm_gb300 import _lib
from bwd_flashattention_fwd_sm_gb300._lib import ParamsC, BlockMaskC

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = [os.path.join(INCLUDE, n) for n in sorted(os.listdir(INCLUDE)) if n.endswith(".h")]

FAKE = 1 << 20  # an aligned non-NULL address; never dereferenced by host validation


def declared_functions():
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:attn|ln)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def params(B=2, Hq=4, Hkv=2, S=256, D=128, dtype=_lib.ATTN_BF16, mask=_lib.ATTN_MASK_CAUSAL):
    p = ParamsC()
    p.batch, p.heads_q, p.heads_kv, p.seqlen, p.head_dim = B, Hq, Hkv, S, D
    p.q_stride_b, p.q_stride_h, p.q_stride_s = Hq * S * D, S * D, D
    p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = Hkv * S * D, S * D, D
    p.scale = 1.0 / np.sqrt(D)
    p.dtype, p.mask = dtype, mask
    return p


def fwd(lib, p, ws=FAKE, ws_bytes=1 << 40, q=FAKE, lse=FAKE):
    return lib.attn_fwd(ctypes.byref(p), q, FAKE, FAKE, FAKE, lse, ws, ws_bytes, None)


def bwd(lib, p, ws=FAKE, ws_bytes=1 << 40):
    return lib.attn_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, None)


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.SIGNATURES), names
    for n in names:
        assert hasattr(lib, n), n
    assert b"sm_103a" in lib.attn_version()


def test_status_strings(lib):
    for code, name in [(0, b"ATTN_OK"), (1, b"ATTN_ERR_INVALID_ARG"), (2, b"ATTN_ERR_UNSUPPORTED"),
                       (3, b"ATTN_ERR_WORKSPACE"), (4, b"ATTN_ERR_CUDA"), (5, b"ATTN_ERR_DEVICE_TIMEOUT"),
                       (6, b"ATTN_ERR_DEVICE_BOUNDS")]:
        assert lib.attn_status_string(code) == name


def test_valid_call_without_gpu_fails_with_cuda_error(lib):
    p = params()
    assert fwd(lib, p) == _lib.ATTN_ERR_CUDA
    assert bwd(lib, p) == _lib.ATTN_ERR_CUDA
    assert lib.attn_get_status(None) == _lib.ATTN_ERR_CUDA


@pytest.mark.parametrize("mutate, code", [
    (lambda p: setattr(p, "heads_kv", 3), _lib.ATTN_ERR_INVALID_ARG),
    (lambda p: setattr(p, "heads_q", 0), _lib.ATTN_ERR_INVALID_ARG),
    (lambda p: setattr(p, "head_dim", 96), _lib.ATTN_ERR_UNSUPPORTED),
    (lambda p: setattr(p, "dtype", 7), _lib.ATTN_ERR_INVALID_ARG),
    (lambda p: setattr(p, "mask", 9), _lib.ATTN_ERR_INVALID_ARG),
    (lambda p: setattr(p, "q_stride_s", 100), _lib.ATTN_ERR_INVALID_ARG),  # not a multiple of 8
    (lambda p: setattr(p, "kv_stride_s", 64), _lib.ATTN_ERR_INVALID_ARG),  # smaller than D
    (lambda p: setattr(p, "scale", float("nan")), _lib.ATTN_ERR_INVALID_ARG),
    (lambda p: setattr(p, "seqlen", -1), _lib.ATTN_ERR_INVALID_ARG),
    (lambda p: setattr(p, "mask", _lib.ATTN_MASK_BLOCK), _lib.ATTN_ERR_INVALID_ARG),  # no block_mask
])
def test_invalid_params_rejected(lib, mutate, code):
    p = params()
    mutate(p)
    assert fwd(lib, p) == code
    assert bwd(lib, p) == code
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == _lib.SIZE_MAX
    assert lib.attn_last_error() != b""


def test_pointer_and_workspace_checks(lib):
    p = params()
    assert fwd(lib, p, q=0) == _lib.ATTN_ERR_INVALID_ARG
    assert fwd(lib, p, q=FAKE + 2) == _lib.ATTN_ERR_INVALID_ARG  # misaligned
    need = lib.attn_fwd_workspace_size(ctypes.byref(p))
    assert 0 < need < _lib.SIZE_MAX
    assert fwd(lib, p, ws=0) == _lib.ATTN_ERR_WORKSPACE
    assert fwd(lib, p, ws_bytes=need - 1) == _lib.ATTN_ERR_WORKSPACE
    assert fwd(lib, p, ws=FAKE + 16) == _lib.ATTN_ERR_WORKSPACE  # not 256-byte aligned
    bneed = lib.attn_bwd_workspace_size(ctypes.byref(p))
    # the dQ accumulator alone is rows * D * 4 bytes
    assert bneed >= 2 * 4 * 256 * 128 * 4
    assert bwd(lib, p, ws_bytes=bneed - 1) == _lib.ATTN_ERR_WORKSPACE


def test_empty_problem_is_a_no_op(lib):
    p = params(B=0)
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 0
    assert lib.attn_fwd(ctypes.byref(p), None, None, None, None, None, None, 0, None) == _lib.ATTN_OK
    p = params(S=0)
    assert lib.attn_bwd(ctypes.byref(p), *([None] * 10), 0, None) == _lib.ATTN_OK


def varlen_params(cu, host=True):
    p = params(B=0)
    cu = np.asarray(cu, dtype=np.int32)
    p.cu_seqlens = FAKE
    p.cu_seqlens_host = cu.ctypes.data if host else None
    p.n_seqs = len(cu) - 1
    T, Hq, Hkv, D = int(cu[-1]), 4, 2, 128
    p.seqlen = int(np.max(np.diff(cu))) if len(cu) > 1 else 0
    p.q_stride_h, p.q_stride_s = D, Hq * D
    p.kv_stride_h, p.kv_stride_s = D, Hkv * D
    return p, cu


def test_varlen_validation(lib):
    p, cu = varlen_params([0, 5, 300, 301])
    assert fwd(lib, p) == _lib.ATTN_ERR_CUDA  # valid: reaches the device step
    p, cu = varlen_params([0, 5, 3, 301])
    assert fwd(lib, p) == _lib.ATTN_ERR_INVALID_ARG  # decreasing
    p, cu = varlen_params([1, 5, 300])
    assert fwd(lib, p) == _lib.ATTN_ERR_INVALID_ARG  # does not start at 0
    p, cu = varlen_params([0, 5, 300], host=False)
    assert fwd(lib, p) == _lib.ATTN_ERR_INVALID_ARG  # host copy missing
    p, cu = varlen_params([0, 5, 300])
    p.seqlen = 200
    assert fwd(lib, p) == _lib.ATTN_ERR_INVALID_ARG  # a sequence longer than seqlen


def block_mask_struct(row_ptr, col_idx, nb, keep):
    rp = np.asarray(row_ptr, dtype=np.int32)
    ci = np.asarray(col_idx if len(col_idx) else [0], dtype=np.int32)
    keep += [rp, ci]
    bm = BlockMaskC()
    bm.row_ptr, bm.col_idx = FAKE, FAKE
    bm.row_ptr_host, bm.col_idx_host = rp.ctypes.data, ci.ctypes.data
    bm.block_q = bm.block_k = 64
    bm.n_row_blocks = bm.n_col_blocks = nb
    bm.nnz = int(rp[-1])
    bm.causal_in_block = 1
    return bm


@pytest.mark.parametrize("row_ptr, col_idx, code", [
    ([0, 1, 3, 4, 6], [0, 0, 1, 2, 1, 3], _lib.ATTN_ERR_CUDA),          # valid
    ([0, 1, 3, 4, 6], [0, 1, 0, 2, 1, 3], _lib.ATTN_ERR_INVALID_ARG),   # unsorted row
    ([0, 1, 3, 4, 6], [0, 0, 0, 2, 1, 3], _lib.ATTN_ERR_INVALID_ARG),   # duplicate column
    ([0, 1, 3, 4, 6], [0, 0, 1, 2, 1, 4], _lib.ATTN_ERR_INVALID_ARG),   # column out of range
    ([0, 1, 3, 2, 6], [0, 0, 1, 2, 1, 3], _lib.ATTN_ERR_INVALID_ARG),   # row_ptr decreases
    ([1, 1, 3, 4, 6], [0, 0, 1, 2, 1, 3], _lib.ATTN_ERR_INVALID_ARG),   # row_ptr[0] != 0
])
def test_block_mask_validation(lib, row_ptr, col_idx, code):
    keep = []
    p = params(S=256, mask=_lib.ATTN_MASK_BLOCK)
    bm = block_mask_struct(row_ptr, col_idx, 4, keep)
    p.block_mask = ctypes.pointer(bm)
    assert fwd(lib, p) == code
    assert bwd(lib, p) == code


def test_block_mask_shape_checked(lib):
    keep = []
    p = params(S=256, mask=_lib.ATTN_MASK_BLOCK)
    bm = block_mask_struct([0, 1, 2, 3], [0, 1, 2], 3, keep)  # 3 blocks, seqlen 256 needs 4
    p.block_mask = ctypes.pointer(bm)
    assert fwd(lib, p) == _lib.ATTN_ERR_INVALID_ARG
    bm = block_mask_struct([0, 1, 2, 3, 4], [0, 1, 2, 3], 4, keep)
    bm.block_q = 128
    p.block_mask = ctypes.pointer(bm)
    assert fwd(lib, p) == _lib.ATTN_ERR_UNSUPPORTED


def test_fp32_head_dim_64_accepted(lib):
    p = params(D=64, dtype=_lib.ATTN_F32)
    p.q_stride_b, p.q_stride_h, p.q_stride_s = 4 * 256 * 64, 256 * 64, 64
    p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = 2 * 256 * 64, 256 * 64, 64
    assert fwd(lib, p) == _lib.ATTN_ERR_CUDA


def test_deterministic_backward_dispatch(lib):
    """attn_bwd_deterministic: float32 I/O is refused before anything is queued;
    a valid bf16 call without a GPU fails with the CUDA error like attn_bwd."""
    p = params(D=64, dtype=_lib.ATTN_F32)
    p.q_stride_b, p.q_stride_h, p.q_stride_s = 4 * 256 * 64, 256 * 64, 64
    p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = 2 * 256 * 64, 256 * 64, 64
    det = lambda q: lib.attn_bwd_deterministic(ctypes.byref(q), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                               FAKE, FAKE, 1 << 40, None)
    assert det(p) == _lib.ATTN_ERR_UNSUPPORTED
    assert b"deterministic" in lib.attn_last_error()
    assert det(params()) == _lib.ATTN_ERR_CUDA


def test_bf16_head_dim_64_accepted(lib):
    """bf16 with head_dim 64 runs on the tensor-core kernels: a valid call fails only for want of a GPU."""
    p = params(D=64)
    p.q_stride_b, p.q_stride_h, p.q_stride_s = 4 * 256 * 64, 256 * 64, 64
    p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = 2 * 256 * 64, 256 * 64, 64
    assert fwd(lib, p) == _lib.ATTN_ERR_CUDA
    assert bwd(lib, p) == _lib.ATTN_ERR_CUDA


def test_selftest_bounded_wait_limit_validated(lib):
    """The timeout self-test refuses a limit outside [1 us, 1 s] before touching a device."""
    assert lib.attn_selftest_bounded_wait(0, None) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_bounded_wait(2_000_000, None) == _lib.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_bounded_wait(1000, None) == _lib.ATTN_ERR_CUDA  # valid, but no GPU here


def test_row_count_limit(lib):
    """Query rows over all heads are indexed in 32 bits on the device: more are refused."""
    p = params(B=1 << 12, Hq=1 << 10, Hkv=1 << 10, S=1 << 10)
    assert fwd(lib, p) == _lib.ATTN_ERR_UNSUPPORTED
    assert b"2^31" in lib.attn_last_error()


def fp8_fwd(lib, p, scales=FAKE, ws_bytes=1 << 40):
    return lib.attn_fwd_fp8(ctypes.byref(p), FAKE, FAKE, FAKE, scales, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes, None)


def fp8_quant(lib, p, scales=FAKE):
    return lib.attn_quantize_fp8(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, scales, FAKE, FAKE, None)


def test_fp8_validation(lib):
    """The FP8 entry points: bf16, head_dim 128, fixed length; checked before any device work."""
    for mask in (_lib.ATTN_MASK_NONE, _lib.ATTN_MASK_CAUSAL):
        assert fp8_fwd(lib, params(mask=mask)) == _lib.ATTN_ERR_CUDA  # valid: fails only for want of a GPU
        assert fp8_quant(lib, params(mask=mask)) == _lib.ATTN_ERR_CUDA
    p = params(D=64)
    p.q_stride_b, p.q_stride_h, p.q_stride_s = 4 * 256 * 64, 256 * 64, 64
    p.kv_stride_b, p.kv_stride_h, p.kv_stride_s = 2 * 256 * 64, 256 * 64, 64
    assert fp8_fwd(lib, p) == _lib.ATTN_ERR_UNSUPPORTED and b"head_dim" in lib.attn_last_error()
    assert fp8_quant(lib, p) == _lib.ATTN_ERR_UNSUPPORTED
    assert fp8_fwd(lib, params(dtype=_lib.ATTN_F32)) == _lib.ATTN_ERR_UNSUPPORTED
    cu = np.array([0, 100, 256], dtype=np.int32)
    pv = params(S=256)
    pv.cu_seqlens = FAKE
    pv.cu_seqlens_host = cu.ctypes.data
    pv.n_seqs = 2
    assert fp8_fwd(lib, pv) == _lib.ATTN_ERR_UNSUPPORTED and b"fixed-length" in lib.attn_last_error()
    assert fp8_fwd(lib, params(), scales=FAKE + 2) == _lib.ATTN_ERR_INVALID_ARG
    assert fp8_quant(lib, params(), scales=0) == _lib.ATTN_ERR_INVALID_ARG
    assert fp8_fwd(lib, params(), ws_bytes=16) == _lib.ATTN_ERR_WORKSPACE
    assert fp8_fwd(lib, params(B=0)) == _lib.ATTN_OK and fp8_quant(lib, params(S=0)) == _lib.ATTN_OK


def test_head_dim_256_accepted(lib):
    """head_dim 256: forward and backward accepted (both dtypes); the deterministic
    backward is refused (its query-stationary dQ pass covers head dims 64 and
    128 only)."""
    for dtype in (_lib.ATTN_BF16, _lib.ATTN_F32):
        p = params(D=256, dtype=dtype)
        assert fwd(lib, p) == _lib.ATTN_ERR_CUDA
        assert bwd(lib, p) == _lib.ATTN_ERR_CUDA
    det = lib.attn_bwd_deterministic(ctypes.byref(params(D=256)), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, FAKE, 1 << 40, None)
    assert det == _lib.ATTN_ERR_UNSUPPORTED
    p = params(D=512)
    assert fwd(lib, p) == _lib.ATTN_ERR_UNSUPPORTED and b"256" in lib.attn_last_error()


def test_workspace_sizes_cover_the_float32_buffers(lib):
    """The workspace queries are host arithmetic and need no GPU.  The backward's
    workspace holds at least the float32 dQ accumulator (one float per element
    of Q) and D (one float per query row).  With few forward units the forward
    splits each unit's key range; every part then keeps float32 O and its row
    max and sum per query row, so the forward's workspace holds at least two
    parts of them."""
    def sizes(**kw):
        p = params(**kw)
        return lib.attn_fwd_workspace_size(ctypes.byref(p)), lib.attn_bwd_workspace_size(ctypes.byref(p))

    for mask in (_lib.ATTN_MASK_NONE, _lib.ATTN_MASK_CAUSAL):
        rows = 2 * 16 * 8192
        nf, nb = sizes(B=2, Hq=16, Hkv=16, S=8192, D=128, mask=mask)
        assert nb >= rows * 128 * 4 + rows * 4
        assert 0 < nf < nb  # 1024 units: no split, only the work list
    # 64 two-tile units over 64 key tiles: the key range is split in two
    rows = 2 * 8192
    nf, nb = sizes(B=1, Hq=2, Hkv=2, S=8192, D=128, mask=_lib.ATTN_MASK_NONE)
    assert nf >= 2 * rows * (128 + 2) * 4
    assert nb >= rows * 128 * 4 + rows * 4
    # float32 I/O at head dim 64 keeps the same accumulator
    rows = 1 * 4 * 1000
    nf, nb = sizes(B=1, Hq=4, Hkv=4, S=1000, D=64, dtype=_lib.ATTN_F32, mask=_lib.ATTN_MASK_NONE)
    assert nb >= rows * 64 * 4 + rows * 4
    # more positions never need less
    small = sizes(B=1, Hq=4, Hkv=2, S=2048, D=128)
    large = sizes(B=1, Hq=4, Hkv=2, S=4096, D=128)
    assert large[1] > small[1]

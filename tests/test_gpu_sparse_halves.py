"""GPU parity of the block-sparse forward on every listing pattern of a tile.

The forward computes S for 128 x 128 tiles (two 64-row blocks x two 64-key
blocks).  In each 64-row block, a 64-key half the block mask does not list is
neither read nor exponentiated: its P is written as zeros.  The mask built here
gives every query tile, across its key tiles, each of the 16 patterns of the
four 64 x 64 blocks.  Those include one row block with no listed half beside a
row block with one or two, and the lower or upper half alone.  The cases run
with and without causal masking inside blocks, at a positive and a negative
scale (the negative one flips the sign of S before the row max), at head dims
64, 128 and 256, and on the FP8 forward.  Tolerances are those of every other
test (parity_util; FP8: the P-rounding bound of test_gpu_fp8).
"""

import numpy as np
import pytest
import torch

import oracle
from bwd_flashattention_fwd_sm_gb300 import BlockMask, attn_fwd, attn_fwd_fp8, get_status, quantize_fp8
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, compare, gpu_run, oracle_run

DEV = torch.device("cuda", 0)
S = 1024  # 16 blocks of 64: 8 query tiles x 8 key tiles of 128


def pattern_csr(causal_in_block):
    """Query tile t and key tile u list the four blocks given by the bits of (5t + u) mod 16
    (bit 2r + c: row block r, key half c).  Every query tile then meets eight
    distinct patterns, and the 64 tiles hold all 16."""
    nb = S // 64
    keep = np.zeros((nb, nb), bool)
    for t in range(nb // 2):
        for u in range(nb // 2):
            bits = (5 * t + u) % 16
            for r in range(2):
                for c in range(2):
                    keep[2 * t + r, 2 * u + c] = bool((bits >> (2 * r + c)) & 1)
    if causal_in_block:
        keep &= np.tril(np.ones((nb, nb), bool))
    return W.csr_from_dense_blocks(keep, causal_in_block=causal_in_block)


def test_pattern_covers_every_case():
    """(CPU) Host check of the mask itself: all 16 patterns appear, including the
    half-listed ones, and no row block is left empty without causal masking."""
    csr = pattern_csr(0)
    rp, ci = np.asarray(csr["row_ptr"]), np.asarray(csr["col_idx"])
    nb = S // 64
    keep = np.zeros((nb, nb), bool)
    for i in range(nb):
        keep[i, ci[rp[i]:rp[i + 1]]] = True
    tiles = keep.reshape(nb // 2, 2, nb // 2, 2).transpose(0, 2, 1, 3).reshape(-1, 4)
    seen = {int(sum(int(b) << j for j, b in enumerate(t))) for t in tiles}
    assert seen == set(range(16))
    assert keep.any(axis=1).all()


@pytest.mark.gpu
@pytest.mark.parametrize("causal_in_block", [0, 1])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_sparse_halves_fwd_bwd(D, causal_in_block):
    wl = W.Workload(f"halves_{D}_{causal_in_block}", 1, 4, 2, S, D, "bf16", "block", seed=120 + D)
    inp = W.make_inputs(wl.with_(mask="none"))
    inp["block_mask"] = pattern_csr(causal_in_block)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))


@pytest.mark.gpu
@pytest.mark.parametrize("causal_in_block", [0, 1])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_sparse_halves_negative_scale(D, causal_in_block):
    scale = -0.7 / np.sqrt(D)
    wl = W.Workload(f"halves_neg_{D}_{causal_in_block}", 1, 4, 2, S, D, "bf16", "block", seed=130 + D)
    inp = W.make_inputs(wl.with_(mask="none"))
    csr = pattern_csr(causal_in_block)
    q, k, v = (inp[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = attn_fwd(q, k, v, block_mask=BlockMask.from_csr(csr, device=DEV), scale=scale)
    torch.cuda.synchronize()
    assert get_status() == 0
    ro, rl = oracle.attn_fwd(*(inp[n].double().numpy() for n in ("q", "k", "v")), scale=scale, block_mask=csr)
    compare(f"o[{wl.name}]", o.double().cpu().numpy(), ro, "bf16")
    compare(f"lse[{wl.name}]", lse.double().cpu().numpy(), rl, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("scale_sign", [1.0, -1.0])
@pytest.mark.parametrize("causal_in_block", [0, 1])
def test_sparse_halves_fp8(causal_in_block, scale_sign):
    from test_gpu_fp8 import _check_fwd, _inputs
    q, k, v = _inputs(1, 4, 2, S, seed=140 + causal_in_block)
    csr = pattern_csr(causal_in_block)
    scale = scale_sign / np.sqrt(128)
    f = quantize_fp8(q.to(DEV), k.to(DEV), v.to(DEV))
    o, lse = attn_fwd_fp8(f, block_mask=BlockMask.from_csr(csr, device=DEV), scale=scale)
    torch.cuda.synchronize()
    assert get_status() == 0
    _check_fwd(o, lse, q, k, v, scale=scale, csr=csr)

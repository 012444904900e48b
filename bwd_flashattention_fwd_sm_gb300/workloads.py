"""Seeded synthetic workloads: shapes, masks, sequence lengths and input tensors.

This module only draws inputs.  It holds none of the attention arithmetic, so the
GPU tests, the benchmark and the oracle checks can all take their inputs from it
without sharing any computation.

Workload shapes follow the attention operator the pages describe: Q, K, V of
shape [batch, head, seq_len, head_dim] (zwxr.cn CANN ops-nn fused-attention
article, section 3.1), sequence lengths of 2048 and up (same article, section
1.2), its measured case B=1, H=8, S=2048, D=128 (section 5.1), causal and
block-sparse masks (smzdm contest article, section 03, on skipping blocks that
need no computation) and batches of long and short sequences (same article,
section 02, on uneven work).

Inputs: Q, K, V, dO are iid N(0, 1) drawn in float32 from ``torch.Generator``
seeded with the workload's seed, in that order, then rounded to bfloat16
(round-to-nearest-even) where the workload is bf16.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads_q: int
    heads_kv: int
    seqlen: int          # S for fixed length; the maximum length for variable length
    head_dim: int
    dtype: str           # "f32" or "bf16"
    mask: str            # "none", "causal" or "block"
    varlen: bool = False
    n_seqs: int = 0      # variable length: number of sequences
    min_len: int = 0     # variable length: lengths uniform in [min_len, seqlen]
    seed: int = 0
    passes: str = "fwd+bwd"
    window_blocks: int = 16   # block mask: sliding window, in 64-token blocks
    random_blocks: int = 64   # block mask: random key blocks drawn per query block
    block: int = 64           # block mask tile size (query and key)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five configurations the method is checked on, plus the S=8192 headline shape
# and the pages' own measured shape.
WORKLOADS = {
    "c1_dense_f32": Workload("c1_dense_f32", 1, 2, 2, 64, 64, "f32", "none", seed=1),
    "c2_causal_fwd": Workload("c2_causal_fwd", 2, 16, 16, 2048, 128, "bf16", "causal", seed=2, passes="fwd"),
    "c3_causal_gqa": Workload("c3_causal_gqa", 4, 32, 8, 4096, 128, "bf16", "causal", seed=3),
    "c4_block_sparse": Workload("c4_block_sparse", 1, 16, 16, 8192, 128, "bf16", "block", seed=4, passes="bwd"),
    "c5_varlen_causal": Workload("c5_varlen_causal", 1, 32, 32, 8192, 128, "bf16", "causal", varlen=True,
                                 n_seqs=16, min_len=128, seed=5),
    "h0_dense_s8192": Workload("h0_dense_s8192", 2, 16, 16, 8192, 128, "bf16", "none", seed=6),
    "h0_causal_s8192": Workload("h0_causal_s8192", 2, 16, 16, 8192, 128, "bf16", "causal", seed=6),
    "p2_dense_s2048": Workload("p2_dense_s2048", 1, 8, 8, 2048, 128, "bf16", "none", seed=7),
    # half of the headline batch: the same kernels at a size a profiler replays quickly
    "h1_dense_s8192": Workload("h1_dense_s8192", 1, 16, 16, 8192, 128, "bf16", "none", seed=6),
    # head dim 64 at the headline length (bf16 on the tensor cores)
    "h2_dense_s8192_d64": Workload("h2_dense_s8192_d64", 2, 16, 16, 8192, 64, "bf16", "none", seed=8),
    "h2_causal_s8192_d64": Workload("h2_causal_s8192_d64", 2, 16, 16, 8192, 64, "bf16", "causal", seed=8),
    # head dim 256 at the headline length, forward and backward
    "d256_dense_s8192": Workload("d256_dense_s8192", 2, 16, 16, 8192, 256, "bf16", "none", seed=10),
}


def torch_dtype(wl: Workload) -> torch.dtype:
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def seq_lengths(wl: Workload) -> np.ndarray:
    """Sequence lengths (int32).  Fixed length: ``batch`` copies of ``seqlen``."""
    if not wl.varlen:
        return np.full(wl.batch, wl.seqlen, dtype=np.int32)
    g = torch.Generator().manual_seed(wl.seed)
    lens = torch.randint(wl.min_len, wl.seqlen + 1, (wl.n_seqs,), generator=g)
    return lens.numpy().astype(np.int32)


def cu_seqlens(wl: Workload) -> np.ndarray:
    lens = seq_lengths(wl)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def block_mask_csr(wl: Workload, seqlen: int | None = None) -> dict:
    """Block-sparse mask over (block x block) tiles as CSR lists, columns ascending.

    Row block i keeps key blocks (sliding window of ``window_blocks`` ending at i)
    united with ``random_blocks`` distinct key blocks drawn uniformly from all key
    blocks (``torch.randperm`` of a generator seeded with the workload's seed, row
    by row), then intersected with the causal rule at block level (j <= i).
    Inside the kept tiles the causal rule also applies token by token
    (``causal_in_block`` = 1).  One mask serves every batch entry and head.
    """
    S = seqlen if seqlen is not None else wl.seqlen
    nb = (S + wl.block - 1) // wl.block
    g = torch.Generator().manual_seed(wl.seed)
    rows, row_ptr = [], [0]
    for i in range(nb):
        window = set(range(max(0, i - wl.window_blocks + 1), i + 1))
        rand = set(torch.randperm(nb, generator=g)[: min(wl.random_blocks, nb)].tolist())
        cols = sorted(c for c in (window | rand) if c <= i)
        rows.extend(cols)
        row_ptr.append(len(rows))
    return {
        "row_ptr": np.asarray(row_ptr, dtype=np.int32),
        "col_idx": np.asarray(rows, dtype=np.int32),
        "n_row_blocks": nb,
        "n_col_blocks": nb,
        "block_q": wl.block,
        "block_k": wl.block,
        "causal_in_block": 1,
    }


def csr_from_dense_blocks(keep: np.ndarray, block: int = 64, causal_in_block: int = 0) -> dict:
    """CSR lists from a boolean [n_row_blocks, n_col_blocks] tile map."""
    keep = np.asarray(keep, dtype=bool)
    row_ptr, cols = [0], []
    for r in range(keep.shape[0]):
        c = np.nonzero(keep[r])[0].tolist()
        cols.extend(c)
        row_ptr.append(len(cols))
    return {
        "row_ptr": np.asarray(row_ptr, dtype=np.int32),
        "col_idx": np.asarray(cols, dtype=np.int32),
        "n_row_blocks": keep.shape[0],
        "n_col_blocks": keep.shape[1],
        "block_q": block,
        "block_k": block,
        "causal_in_block": int(causal_in_block),
    }


def tensor_shapes(wl: Workload):
    """(q-like shape, kv-like shape) in the layouts the library and oracle use."""
    if wl.varlen:
        T = int(cu_seqlens(wl)[-1])
        return (T, wl.heads_q, wl.head_dim), (T, wl.heads_kv, wl.head_dim)
    return ((wl.batch, wl.heads_q, wl.seqlen, wl.head_dim),
            (wl.batch, wl.heads_kv, wl.seqlen, wl.head_dim))


def make_inputs(wl: Workload) -> dict:
    """Seeded CPU tensors q, k, v, do in the workload's dtype (plus metadata)."""
    qs, ks = tensor_shapes(wl)
    g = torch.Generator().manual_seed(wl.seed)
    dt = torch_dtype(wl)
    out = {}
    for name, shape in (("q", qs), ("k", ks), ("v", ks), ("do", qs)):
        out[name] = torch.randn(shape, generator=g, dtype=torch.float32).to(dt)
    if wl.varlen:
        out["cu_seqlens"] = cu_seqlens(wl)
    if wl.mask == "block":
        out["block_mask"] = block_mask_csr(wl)
    return out


def tile_spread(x: torch.Tensor, seed: int, spread: int = 3, tile: int = 128) -> torch.Tensor:
    """x [..., S, D] with each `tile`-row block along S multiplied by 2^U{-spread..spread}
    (seeded), rounded back to x's dtype: inputs whose per-tile magnitudes differ, so
    that per-tile scales differ too."""
    g = torch.Generator().manual_seed(seed)
    S = x.shape[-2]
    nt = (S + tile - 1) // tile
    e = torch.randint(-spread, spread + 1, tuple(x.shape[:-2]) + (nt,), generator=g).float()
    f = torch.pow(2.0, e).repeat_interleave(tile, dim=-1)[..., :S, None]
    return (x.float() * f).to(x.dtype)


def unmasked_pairs(wl: Workload, block_mask: dict | None = None) -> int:
    """Number of allowed (query, key) pairs summed over batch entries, for ONE head.

    Used to count algorithmic FLOPs: forward 4*D*pairs*Hq, backward 10*D*pairs*Hq.
    """
    lens = seq_lengths(wl)
    if wl.mask == "none":
        return int(sum(int(L) * int(L) for L in lens))
    if wl.mask == "causal":
        return int(sum(int(L) * (int(L) + 1) // 2 for L in lens))
    bm = block_mask if block_mask is not None else block_mask_csr(wl)
    total = 0
    for L in lens:
        L = int(L)
        for rb in range(bm["n_row_blocks"]):
            i0, i1 = rb * bm["block_q"], min((rb + 1) * bm["block_q"], L)
            if i0 >= L:
                break
            for e in range(bm["row_ptr"][rb], bm["row_ptr"][rb + 1]):
                cb = int(bm["col_idx"][e])
                j0, j1 = cb * bm["block_k"], min((cb + 1) * bm["block_k"], L)
                if j0 >= L:
                    continue
                ii = np.arange(i0, i1)[:, None]
                jj = np.arange(j0, j1)[None, :]
                ok = np.ones((i1 - i0, j1 - j0), dtype=bool)
                if bm["causal_in_block"]:
                    ok &= jj <= ii
                total += int(ok.sum())
    return total

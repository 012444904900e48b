"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding, run the oracle on the same seeded inputs, compare element by element.

Tolerances (written here, used by every GPU test):
  float32 I/O : max |gpu - oracle| <= 1e-3 on O, LSE, dQ, dK, dV (the 1e-3
                alignment bar of the zwxr.cn CANN ops-nn article, section 3.4,
                read as an absolute bound).
  bfloat16 I/O: |gpu - oracle| <= 2e-2 + half_ulp(oracle) element-wise, and
                ||gpu - oracle||_2 / ||oracle||_2 <= 1e-2 per tensor; LSE
                (float32) max-abs <= 2e-2.  half_ulp(x) is half the spacing of
                bfloat16 numbers at |x| (2^(e-8) for |x| in [2^e, 2^(e+1))): the
                distance by which rounding the exact value to a bf16 output can
                move it by itself.  Below |x| = 8 that is under 2^-6 < 2e-2, so
                the term matters only for outputs the 2e-2 bar alone could not
                hold even when rounded correctly.
  GQA groups  : dK and dV of a KV head sum the contributions of its G query
                heads, each product taking its own bf16 rounding of P (dV) or
                dS (dK) with float32 accumulation, the arithmetic the method
                prescribes.  Independent roundings add in quadrature, so the
                error of a group sum grows like sqrt(G).  The 2e-2 term is the
                stated bar at the largest group of the configurations (G = 4,
                the causal GQA one) and scales by sqrt(G / 4) above it; G <= 4
                keeps 2e-2.  tests/test_tolerance.py replays that rounding in
                float64 for G = 1, 4, 16: its RMS error doubles with each
                fourfold G, at G = 16 the replay itself breaks the unscaled bar,
                and the scaled bar holds it with room to spare.

Margins: with GBATTN_PARITY_LOG set to a file path, every comparison appends one
JSON line (name, dtype, max-abs, rel-L2, the largest ratio of error to its
bound, element count) to that file before asserting.
"""

from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from bwd_flashattention_fwd_sm_gb300 import BlockMask, SeqLens, attn_bwd, attn_fwd, get_status
from bwd_flashattention_fwd_sm_gb300 import workloads as W

TOL_F32 = 1e-3
TOL_BF16_ABS = 2e-2
TOL_BF16_REL = 1e-2


def half_ulp_bf16(x):
    """Half the spacing of bfloat16 numbers at |x| (8 significant bits): for |x|
    in [2^e, 2^(e+1)) the spacing is 2^(e-7); 0 where x is 0."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, ex = np.frexp(x)  # x = m 2^ex with m in [0.5, 1), so e = ex - 1
    return np.where(x > 0, np.ldexp(1.0, ex - 9), 0.0)


def _log_margin(name, dtype, max_abs, rel, ratio, n):
    path = os.environ.get("GBATTN_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"name": name, "dtype": dtype, "max_abs": max_abs, "rel_l2": rel,
                            "worst_err_over_bound": ratio, "n": int(n)}) + "\n")


def group_scale(group: int) -> float:
    """Factor on the 2e-2 term for dK and dV of a KV head shared by `group` query heads."""
    return max(1.0, (group / 4.0) ** 0.5)


def compare(name, got, ref, dtype, abs_scale=1.0):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{name}: -inf positions differ"
    fin = ~inf_ref
    g, r = got[fin], ref[fin]
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    if g.size == 0:
        return 0.0, 0.0
    err = np.abs(g - r)
    max_abs = float(err.max())
    nrm = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / nrm) if nrm > 0 else float(np.linalg.norm(g - r))
    if dtype == "f32":
        bound = np.full_like(r, TOL_F32)
    elif name.startswith("lse"):
        bound = np.full_like(r, TOL_BF16_ABS)
    else:
        bound = TOL_BF16_ABS * abs_scale + half_ulp_bf16(r)
    ratio = err / bound
    worst = int(np.argmax(ratio))
    _log_margin(name, dtype, max_abs, rel, float(ratio[worst]), g.size)
    assert np.all(err <= bound), (f"{name}: |err| {err[worst]:.3e} > {bound[worst]:.3e} at value "
                                  f"{r[worst]:.4f} (max-abs {max_abs:.3e})")
    if dtype != "f32" and not name.startswith("lse"):
        assert rel <= TOL_BF16_REL, f"{name}: rel-L2 {rel:.3e} > {TOL_BF16_REL}"
    return max_abs, rel


def gpu_run(wl: W.Workload, inputs: dict, passes="fwd+bwd", deterministic=False):
    """Run the CUDA path on `inputs` (CPU tensors); returns CPU float64 numpy results.

    deterministic: the backward through attn_bwd_deterministic."""
    dev = torch.device("cuda")
    q, k, v, do = (inputs[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = {"scale": wl.scale}
    if wl.mask == "causal":
        kw["causal"] = True
    if wl.mask == "block":
        kw["block_mask"] = BlockMask.from_csr(inputs["block_mask"], device=dev)
    if wl.varlen:
        kw["seqlens"] = SeqLens(inputs["cu_seqlens"], device=dev)
        kw["seqlen"] = wl.seqlen
    o, lse = attn_fwd(q, k, v, **kw)
    out = {"o": o, "lse": lse}
    if "bwd" in passes:
        dq, dk, dv = attn_bwd(q, k, v, o, do, lse, deterministic=deterministic, **kw)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert get_status() == 0, "device status word set"
    return {n: t.double().cpu().numpy() for n, t in out.items()}


def oracle_kw(wl: W.Workload, inputs: dict):
    kw = {"scale": wl.scale}
    if wl.mask == "causal":
        kw["causal"] = True
    if wl.mask == "block":
        kw["block_mask"] = inputs["block_mask"]
    return kw


def oracle_run(wl, inputs, passes="fwd+bwd", cu=None):
    q, k, v, do = (inputs[n].double().numpy() for n in ("q", "k", "v", "do"))
    kw = oracle_kw(wl, inputs)
    if cu is not None:
        kw["cu_seqlens"] = cu
    o, lse = oracle.attn_fwd(q, k, v, **kw)
    ref = {"o": o, "lse": lse}
    if "bwd" in passes:
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, **kw)
        ref.update(dq=dq, dk=dk, dv=dv)
    return ref


def check_all(wl, got, ref, names=("o", "lse", "dq", "dk", "dv")):
    report = {}
    group = wl.heads_q // wl.heads_kv
    for n in names:
        if n in ref:
            scale = group_scale(group) if n in ("dk", "dv") else 1.0
            report[n] = compare(f"{n}[{wl.name}]", got[n], ref[n], wl.dtype, abs_scale=scale)
    return report

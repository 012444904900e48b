"""The checked library on the GPU, with valid inputs only.

A process started with GBATTN_CHECKED=1 loads libgbattn_checked.so, whose
kernels compare every device-computed index (work-list entries, block-mask
entries, the rows behind each tile load, reduce-add, row read and row store)
with its tensor's extent before the access.  With valid arguments no check may
fail: after every call the device status word must still read ATTN_OK, and the
results must match the oracle at the usual parity bound.  No test here feeds a
kernel a bad index.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from bwd_flashattention_fwd_sm_gb300 import _lib, get_status, quantize_fp8, attn_fwd_fp8
from bwd_flashattention_fwd_sm_gb300 import workloads as W
from parity_util import check_all, gpu_run, oracle_run
import test_gpu_parity as T

lib = _lib.load()
assert lib.attn_version().endswith(b" checked"), lib.attn_version()
cases = [
    (W.Workload("chk_causal_gqa", 1, 8, 2, 300, 128, "bf16", "causal", seed=71), None, False),
    (W.Workload("chk_dense_d64", 2, 4, 4, 257, 64, "bf16", "none", seed=72), None, False),
    (W.Workload("chk_block", 1, 4, 2, 520, 128, "bf16", "block", seed=73), T.tiles_csr(520, seed=5), False),
    (W.Workload("chk_block_d64", 1, 2, 1, 333, 64, "bf16", "block", seed=74), T.tiles_csr(333, seed=6), False),
    (W.Workload("chk_det", 1, 4, 2, 300, 128, "bf16", "causal", seed=75), None, True),
    (W.Workload("chk_d256", 1, 2, 1, 200, 256, "bf16", "causal", seed=76), None, False),
    (W.Workload("chk_f32", 1, 2, 2, 130, 64, "f32", "causal", seed=77), None, False),
    (W.Workload("chk_f32_block", 1, 2, 1, 200, 128, "f32", "block", seed=78), T.tiles_csr(200, seed=7), False),
    (W.Workload("chk_split", 1, 1, 1, 4096, 128, "bf16", "causal", seed=79), None, False),
]
for wl, csr, det in cases:
    inp = W.make_inputs(wl.with_(mask="none") if csr is not None else wl)
    if csr is not None:
        inp["block_mask"] = csr
    got = gpu_run(wl, inp, deterministic=det)
    assert get_status() == 0, wl.name
    check_all(wl, got, oracle_run(wl, inp))
    print("ok", wl.name, flush=True)

# packed variable length (the causal GQA and the float32 path)
lens = [5, 0, 128, 1, 200, 64, 129]
cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
for dtype, D in (("bf16", 128), ("bf16", 64), ("f32", 128)):
    wl = W.Workload("chk_varlen", 1, 4, 2, max(lens), D, dtype, "causal", varlen=True, n_seqs=len(lens), seed=80)
    T_ = int(cu[-1])
    g = torch.Generator().manual_seed(80)
    dt = W.torch_dtype(wl)
    inp = {{n: torch.randn(s, generator=g).to(dt) for n, s in
           (("q", (T_, 4, D)), ("k", (T_, 2, D)), ("v", (T_, 2, D)), ("do", (T_, 4, D)))}}
    inp["cu_seqlens"] = cu
    got = gpu_run(wl, inp)
    assert get_status() == 0
    check_all(wl, got, oracle_run(wl, inp, cu=cu))
    print("ok varlen", dtype, D, flush=True)

# the FP8 forward (quantisation and the e4m3 form of the forward kernel)
wl = W.Workload("chk_fp8", 1, 2, 1, 300, 128, "bf16", "causal", seed=81)
inp = W.make_inputs(wl)
q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
o, lse = attn_fwd_fp8(quantize_fp8(q, k, v), causal=True, scale=wl.scale)
torch.cuda.synchronize()
assert get_status() == 0
assert torch.isfinite(o.float()).all()
print("ok fp8", flush=True)
print("CHECKED-OK")
"""


def test_checked_library_keeps_status_ok_and_parity():
    env = dict(os.environ, GBATTN_CHECKED="1")
    script = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "CHECKED-OK" in r.stdout, (r.stdout[-3000:], r.stderr[-3000:])

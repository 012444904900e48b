"""The device-side timeout path, exercised without faulting or hanging a GPU: a
warp waits (through the kernels' bounded mbarrier wait) on a barrier nothing
completes, gives up after the limit, and records ATTN_ERR_DEVICE_TIMEOUT in
the status word; the host reads it, the word clears, and attention calls on
the same context still give correct results."""

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_sm_gb300 import _lib, get_status
from bwd_flashattention_fwd_sm_gb300 import workloads as W

from parity_util import check_all, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = _lib.load()
    torch.cuda.synchronize()
    assert get_status() == _lib.ATTN_OK
    stream = torch.cuda.current_stream()
    assert lib.attn_selftest_bounded_wait(2000, stream.cuda_stream) == _lib.ATTN_OK  # 2 ms
    assert get_status() == _lib.ATTN_ERR_DEVICE_TIMEOUT
    assert get_status() == _lib.ATTN_OK  # read once, then cleared
    # the context is intact: a small problem still matches the oracle
    wl = W.Workload("after_timeout", 1, 2, 2, 200, 128, "bf16", "causal", seed=41)
    inp = W.make_inputs(wl)
    check_all(wl, gpu_run(wl, inp), oracle_run(wl, inp))

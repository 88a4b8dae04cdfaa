"""The failure path of the on-chip pipeline waits, exercised without a GPU
fault: a wait on a barrier that nothing completes runs out after the
library's limit (2 s), the kernel reports MM3IDX_DEV_TIMEOUT through the
device status word and returns, and the context keeps working (a decode right
after it matches the oracle)."""

import time

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("warps", [1, 5])
def test_wait_limit_reports_timeout_and_context_survives(cuda_device, warps):
    import torch
    import sparse_attention_block_paged_gb300 as mm
    torch.cuda.synchronize()
    assert mm.get_device_error() == 0
    t0 = time.perf_counter()
    mm.check_wait_timeout(warps)
    assert mm.get_device_error() == mm.DEV_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 1.5 < elapsed < 30.0, elapsed
    assert mm.get_device_error() == 0          # reading clears the word

    wl = W.make("tiny")
    d = to_device(wl)
    got = mm.decode(d["q"], d["cache"], d["table"], d["lens"], query_len=wl.query_len,
                    max_seq_len=wl.max_seq_len, topk=wl.topk, init_blocks=wl.init_blocks,
                    local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    np.testing.assert_array_equal(got.cpu().numpy(), oracle.problem(wl, want_scores=False)[1])
    assert mm.get_device_error() == 0

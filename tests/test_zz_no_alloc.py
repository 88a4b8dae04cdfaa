"""mm3idx_decode_static: the decode entry point for callers that cannot give
the library any device memory (no allocator at hand, or allocation not
allowed where they call from).  It uses the library's own fixed device array
instead of a workspace.  Checked through the C ABI against mm3idx_decode on
the same inputs, on two calls in a row (the array keeps the previous call's
contents, which must not matter).

This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest

import workloads as W
from helpers import to_device

pytestmark = pytest.mark.gpu


def _static_call(mm, p, topk, init_blocks, local_blocks, out, stream):
    return mm.lib.mm3idx_decode_static(ctypes.byref(p), topk, init_blocks, local_blocks,
                                       out.data_ptr(), out.stride(0), out.stride(1),
                                       ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("case", ["spec_like", "tiny"])
def test_static_scratch_decode_matches_workspace_decode(cuda_device, case):
    import torch
    import sparse_attention_block_paged_gb300 as mm
    if case == "tiny":
        wl = W.make("tiny")
    else:
        # requests long enough to be split across CTAs, so the scratch holds
        # partial candidate lists between the two kernels
        wl = W.random_case(77, num_reqs=12, query_len=4, heads=2, topk=16, init_blocks=1,
                           local_blocks=2, min_len=4096, max_len=32768)
    d = to_device(wl)
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    want = mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw).cpu().numpy()

    p = mm._problem(d["q"], d["cache"], d["table"], d["lens"], wl.query_len, wl.max_seq_len,
                    wl.sm_scale)
    stream = torch.cuda.current_stream()
    for call in range(2):
        out = torch.full((wl.heads, wl.rows, wl.topk), -7, dtype=torch.int32, device="cuda")
        rc = _static_call(mm, p, wl.topk, wl.init_blocks, wl.local_blocks, out, stream)
        assert rc == 0, mm.status_string(rc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), want, err_msg=f"call {call}")
    assert mm.get_device_error() == 0


def test_static_scratch_rejects_too_large_problems(cuda_device):
    import torch
    import sparse_attention_block_paged_gb300 as mm
    # 40000 requests of partial lists need more than the static array holds
    n = 40000
    q = torch.zeros((n, 1, 128), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((n, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones((n,), dtype=torch.int32, device="cuda")
    p = mm._problem(q, cache, table, lens, 1, 128, 0.1)
    out = torch.empty((1, n, 32), dtype=torch.int32, device="cuda")
    rc = _static_call(mm, p, 32, 1, 1, out, torch.cuda.current_stream())
    assert rc == -12
    assert "static" in mm.status_string(rc)

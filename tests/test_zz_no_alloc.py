"""mm3idx_decode_static: the decode entry point for callers that cannot give
the library any device memory (no allocator at hand, or allocation not
allowed where they call from).  It uses the library's own fixed device array
instead of a workspace.  Checked through the C ABI against the CPU oracle and
against mm3idx_decode on the same inputs, on two calls in a row (the array
keeps the previous call's contents, which must not matter), and checked to
leave the device's free memory unchanged.

This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, to_device

pytestmark = pytest.mark.gpu


def _static_call(mm, p, topk, init_blocks, local_blocks, out, stream):
    return mm.lib.mm3idx_decode_static(ctypes.byref(p), topk, init_blocks, local_blocks,
                                       out.data_ptr(), out.stride(0), out.stride(1),
                                       ctypes.c_void_p(stream.cuda_stream))


def _largest_batch_under_cap(mm, heads, query_len, max_seq_len, topk):
    """The most requests whose decode workspace still fits the static array."""
    lo, hi = 1, 1 << 16
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if mm.workspace_bytes(mm.OP_DECODE, heads, mid, query_len, max_seq_len,
                              topk) <= mm.STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _case(mm, name):
    if name == "tiny":
        return W.make("tiny")
    if name == "spec_like":
        # requests long enough to be split across CTAs, so the array holds
        # partial candidate lists between the CTAs of a request
        return W.random_case(77, num_reqs=12, query_len=4, heads=2, topk=16, init_blocks=1,
                             local_blocks=2, min_len=4096, max_len=32768)
    # topk 32 doubles the partial lists; as many requests as the array holds
    n = _largest_batch_under_cap(mm, 1, 2, 3000, 32)
    return W.random_case(78, num_reqs=n, query_len=2, heads=1, topk=32, init_blocks=2,
                         local_blocks=3, min_len=2, max_len=3000, max_seq_len=3000)


@pytest.mark.parametrize("case", ["spec_like", "tiny", "topk32_at_cap"])
def test_static_scratch_decode_matches_oracle_and_workspace_decode(cuda_device, case):
    import torch
    import sparse_attention_block_paged_gb300 as mm
    wl = _case(mm, case)
    if case == "topk32_at_cap":
        need = mm.workspace_bytes(mm.OP_DECODE, wl.heads, wl.num_reqs, wl.query_len,
                                  wl.max_seq_len, wl.topk)
        more = mm.workspace_bytes(mm.OP_DECODE, wl.heads, wl.num_reqs + 1, wl.query_len,
                                  wl.max_seq_len, wl.topk)
        assert need <= mm.STATIC_SCRATCH_BYTES < more
    s, want = oracle.problem(wl)
    d = to_device(wl)
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    with_ws = mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw).cpu().numpy()
    check_ids(with_ws, want, s, wl, where=f"{case} workspace decode")

    p = mm._problem(d["q"], d["cache"], d["table"], d["lens"], wl.query_len, wl.max_seq_len,
                    wl.sm_scale)
    stream = torch.cuda.current_stream()
    outs = [torch.full((wl.heads, wl.rows, wl.topk), -7, dtype=torch.int32, device="cuda")
            for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for call in range(2):
        rc = _static_call(mm, p, wl.topk, wl.init_blocks, wl.local_blocks, outs[call], stream)
        assert rc == 0, mm.status_string(rc)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, f"call {call} changed free memory"
    for call in range(2):
        got = outs[call].cpu().numpy()
        check_ids(got, want, s, wl, where=f"{case} static call {call}")
        np.testing.assert_array_equal(got, with_ws, err_msg=f"{case} call {call}")
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
    # a rejected argument comes back as its own code, not as a scratch error
    q2 = torch.zeros((n, 33, 128), dtype=torch.bfloat16, device="cuda")
    p2 = mm._problem(q2, cache, table, lens, 1, 128, 0.1)
    out2 = torch.empty((33, n, 32), dtype=torch.int32, device="cuda")
    assert _static_call(mm, p2, 32, 1, 1, out2, torch.cuda.current_stream()) == -10

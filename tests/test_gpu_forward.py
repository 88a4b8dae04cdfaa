"""mm3idx_forward: one batch of decode requests followed by prefill requests
(the indexer_nvfp4 page's forward splits a batch the same way: decode rows
first, through the decode scorer, the rest through the prefill scorer, into
one output).  The whole batch is a ragged batch for the oracle
(oracle.problem_ragged); every row is compared with it."""

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mm(cuda_device):
    import sparse_attention_block_paged_gb300 as m
    return m


def mixed_case(seed, *, num_decodes, decode_qlen, decode_lens, prefill_rows, prefill_prefix,
               heads=1, topk=16, init_blocks=1, local_blocks=2, kv_format="bf16",
               max_seq_len=None):
    ql = [decode_qlen] * num_decodes + list(prefill_rows)
    pre = [max(0, n - decode_qlen) for n in decode_lens] + list(prefill_prefix)
    return W.ragged_case(seed, query_lens=ql, prefix_lens=pre, heads=heads, topk=topk,
                         init_blocks=init_blocks, local_blocks=local_blocks,
                         max_seq_len=max_seq_len, kv_format=kv_format)


def run_forward(mm, wl, num_decodes, decode_qlen, **kw):
    import torch
    d = to_device(wl)
    cu = wl.cu_seqlens
    start = int(cu[num_decodes])
    pcu = torch.from_numpy((cu[num_decodes:] - start).astype(np.int32)).cuda()
    prefill_rows = np.diff(cu[num_decodes:])
    pmax = int(prefill_rows.max()) if len(prefill_rows) else 1
    cache = d["cache"] if wl.kv_format == "bf16" else d["codes"]
    ids = mm.forward(d["q"], cache, d["table"], d["lens"], pcu, num_decodes=num_decodes,
                     decode_query_len=decode_qlen, prefill_max_query_len=max(pmax, 1),
                     max_seq_len=wl.max_seq_len, topk=wl.topk, init_blocks=wl.init_blocks,
                     local_blocks=wl.local_blocks, sm_scale=wl.sm_scale,
                     index_scales=d.get("scales"), **kw)
    return ids.cpu().numpy()


CASES = [
    # seed, decodes, decode qlen, prefill rows, prefill prefixes, heads, topk, format
    (1, 6, 4, [300, 700], [1000, 0], 1, 16, "bf16"),
    (2, 5, 2, [257], [3000], 2, 8, "bf16"),
    (3, 4, 4, [400, 129], [6000, 9000], 1, 32, "bf16"),    # 32-key lists
    (4, 6, 4, [300, 700], [1000, 0], 1, 16, "nvfp4"),
    (5, 0, 4, [600], [900], 1, 16, "bf16"),                 # prefill only
    (6, 7, 4, [], [], 1, 16, "bf16"),                       # decode only
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_forward_matches_oracle(mm, case):
    seed, nd, dq, prows, ppre, heads, topk, fmt = case
    rng = np.random.default_rng(seed)
    lens = rng.integers(500, 9000, size=nd)
    wl = mixed_case(seed, num_decodes=nd, decode_qlen=dq, decode_lens=lens, prefill_rows=prows,
                    prefill_prefix=ppre, heads=heads, topk=topk, kv_format=fmt)
    s, want = oracle.problem_ragged(wl)
    got = run_forward(mm, wl, nd, dq)
    assert mm.get_device_error() == 0
    check_ids(got, want, s, wl, where=f"forward seed{seed}")


def test_forward_spec_decode_batch_with_chunked_prefills(mm):
    """64 decode requests of 4 rows (4K-32K tokens) and two chunked prefills
    in one call, twice on the same workspace; every row against the oracle."""
    import torch
    rng = np.random.default_rng(7)
    lens = rng.integers(4096, 32768, size=64, endpoint=True)
    wl = mixed_case(7, num_decodes=64, decode_qlen=4, decode_lens=lens,
                    prefill_rows=[1000, 900], prefill_prefix=[3000, 1200], max_seq_len=32768)
    s, want = oracle.problem_ragged(wl)
    pmax = 1000
    n = mm.forward_workspace_bytes(1, 64, 4, 2, pmax, wl.max_seq_len, wl.topk)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for call in range(2):
        got = run_forward(mm, wl, 64, 4, workspace=ws)
        assert mm.get_device_error() == 0
        check_ids(got, want, s, wl, where=f"mixed batch call {call}")

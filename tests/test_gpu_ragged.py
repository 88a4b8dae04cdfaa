"""GPU parity of the ragged-batch calls (mm3idx_score_ragged, mm3idx_topk_ragged,
mm3idx_prefill_ragged) against the oracle's ragged composition: scores and
ids element by element on small batches (requests with no new rows,
one-row requests, rows spanning several 128-row tiles with ragged tails,
chunked prefixes), NVFP4, a ragged batch of equal counts against the uniform
call, malformed offsets, and a larger chunked-prefill batch on sampled rows."""

import copy

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, check_ids_row, check_scores, row_request, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mm(cuda_device):
    import sparse_attention_block_paged_gb300 as m
    return m


def dev(wl):
    import torch
    d = to_device(wl)
    d["cu"] = torch.from_numpy(wl.cu_seqlens).cuda()
    return d


def run_prefill(mm, wl, **kw):
    d = dev(wl)
    cache = d["cache"] if wl.kv_format == "bf16" else d["codes"]
    ids = mm.prefill_ragged(d["q"], cache, d["table"], d["lens"], d["cu"],
                            max_query_len=wl.query_len, max_seq_len=wl.max_seq_len,
                            topk=wl.topk, init_blocks=wl.init_blocks,
                            local_blocks=wl.local_blocks, sm_scale=wl.sm_scale,
                            index_scales=d.get("scales"), **kw)
    return ids.cpu().numpy()


CASES = [
    # seed, query lens, prefix lens, heads, topk, init, local
    (1, [5, 0, 130, 1], [0, 40, 300, 1000], 1, 4, 1, 1),
    (2, [300, 129, 1, 257], [0, 2000, 127, 128], 2, 16, 1, 2),
    (3, [1000, 0, 0, 700], [0, 5, 9, 3000], 1, 8, 2, 2),
    (4, [128, 128, 128], [128, 0, 383], 4, 32, 2, 3),
    (5, [2000, 31, 500, 1, 64, 900], [6000, 0, 2500, 10000, 64, 12], 2, 16, 1, 2),
    # 32-key lists (batched offers) over CTA shares that start and end
    # inside tiles of several requests
    (6, [500, 3, 900, 257], [9000, 12000, 4000, 6000], 1, 27, 1, 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_ragged_prefill_and_scores_match_oracle(mm, case):
    seed, ql, pre, heads, topk, init, local = case
    wl = W.ragged_case(seed, query_lens=ql, prefix_lens=pre, heads=heads, topk=topk,
                       init_blocks=init, local_blocks=local)
    s, want = oracle.problem_ragged(wl)
    got = run_prefill(mm, wl)
    check_ids(got, want, s, wl, where=f"ragged prefill seed{seed}")
    d = dev(wl)
    sc = mm.score_ragged(d["q"], d["cache"], d["table"], d["lens"], d["cu"],
                         max_query_len=wl.query_len, max_seq_len=wl.max_seq_len,
                         sm_scale=wl.sm_scale)
    check_scores(sc.cpu().numpy(), s, f"ragged scores seed{seed}")
    assert mm.get_device_error() == 0


def test_ragged_topk_on_given_scores_is_exact(mm):
    """The selector alone on the oracle's scores (rounded to fp32, as the
    kernel reads them) against the oracle's selection on those same values."""
    import torch
    wl = W.ragged_case(6, query_lens=[40, 0, 7, 300], prefix_lens=[900, 3, 2000, 0], heads=2,
                       topk=16, init_blocks=1, local_blocks=2)
    s, _ = oracle.problem_ragged(wl)
    s32 = s.astype(np.float32)
    want = np.empty((wl.heads, wl.rows, wl.topk), dtype=np.int32)
    for h in range(wl.heads):
        for r in range(wl.rows):
            i, j, ql = row_request(wl, r)
            nb = (int(wl.seq_lens[i]) - ql + j) // 128 + 1
            want[h, r] = oracle.select(s32[h, r, :nb].astype(np.float64), wl.topk,
                                       wl.init_blocks, wl.local_blocks)
    d = dev(wl)
    got = mm.topk_ragged(torch.from_numpy(s32).cuda(), d["lens"], d["cu"],
                         max_query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
                         init_blocks=wl.init_blocks, local_blocks=wl.local_blocks)
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    assert mm.get_device_error() == 0


def test_ragged_nvfp4_prefill_matches_oracle(mm):
    wl = W.ragged_case(7, query_lens=[600, 3, 0, 250], prefix_lens=[0, 4000, 10, 1500], heads=1,
                       topk=16, init_blocks=1, local_blocks=2, kv_format="nvfp4")
    s, want = oracle.problem_ragged(wl)
    check_ids(run_prefill(mm, wl), want, s, wl, where="ragged nvfp4")
    assert mm.get_device_error() == 0


def test_ragged_with_equal_counts_equals_uniform_call(mm):
    wl = W.ragged_case(8, query_lens=[200, 200, 200], prefix_lens=[0, 1000, 3000], heads=2,
                       topk=16, init_blocks=1, local_blocks=2)
    got_r = run_prefill(mm, wl)
    u = copy.copy(wl)
    u.cu_seqlens = None
    u.query_len = 200
    d = to_device(u)
    got_u = mm.prefill(d["q"], d["cache"], d["table"], d["lens"], query_len=200,
                       max_seq_len=u.max_seq_len, topk=u.topk, init_blocks=1, local_blocks=2,
                       sm_scale=u.sm_scale).cpu().numpy()
    np.testing.assert_array_equal(got_r, got_u)


def test_ragged_bad_offsets_are_flagged(mm):
    import torch
    wl = W.ragged_case(9, query_lens=[100, 100], prefix_lens=[0, 300], heads=1, topk=4,
                       init_blocks=1, local_blocks=1)
    d = dev(wl)
    d["cu"] = torch.tensor([0, 150, 120], dtype=torch.int32, device="cuda")   # decreasing
    mm.prefill_ragged(d["q"], d["cache"], d["table"], d["lens"], d["cu"], max_query_len=150,
                      max_seq_len=wl.max_seq_len, topk=4, init_blocks=1, local_blocks=1,
                      sm_scale=wl.sm_scale)
    assert mm.get_device_error() & mm.DEV_BAD_ROWS


def test_ragged_chunked_prefill_batch_sampled(mm):
    """Eight requests of 1000..8000 new rows after 0..24000 earlier tokens."""
    rng = np.random.default_rng(12)
    ql = rng.integers(1000, 8000, size=8, endpoint=True)
    pre = rng.integers(0, 24000, size=8, endpoint=True)
    wl = W.ragged_case(12, query_lens=ql, prefix_lens=pre, heads=1, topk=16, init_blocks=1,
                       local_blocks=2, max_seq_len=32768)
    got = run_prefill(mm, wl)
    assert mm.get_device_error() == 0
    cu = wl.cu_seqlens
    for i in range(wl.num_reqs):
        sub = copy.copy(wl)
        sub.cu_seqlens = None
        sub.query_len = int(cu[i + 1] - cu[i])
        sub.seq_lens = wl.seq_lens[i:i + 1].copy()
        sub.block_table = wl.block_table[i:i + 1].copy()
        sub.q = wl.q[cu[i]:cu[i + 1]].copy()
        for j in sorted({0, 1, 127, 128, sub.query_len - 1, sub.query_len // 2}):
            s, want = oracle.row(sub, j, 0)
            check_ids_row(got[0, int(cu[i]) + j], want, s, len(s) - 1, wl.topk, wl.init_blocks,
                          wl.local_blocks, where=f"chunked req {i} row {j}")

"""GPU parity of the sparse page table written by the decode kernel
(mm3idx_decode_sparse_table) against the oracle's table of the oracle's ids.

Rows whose ids equal the oracle's (all rows whose selection is decided by
more than the score tolerance) must give the oracle's table row and context
length exactly.  A row whose ids legitimately differ (a near-tie) is checked
for validity: its table row must describe its own ids.  The ids themselves
must be exactly those of the plain decode call."""

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, to_device

pytestmark = pytest.mark.gpu
BLOCK = 128


@pytest.fixture(scope="module")
def mm(cuda_device):
    import sparse_attention_block_paged_gb300 as m
    return m


def run(mm, wl, attn, ppb, stride):
    import torch
    d = to_device(wl)
    rows = wl.rows
    st = torch.full((rows, wl.topk * ppb), -5, dtype=torch.int32, device="cuda")
    ctx = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    cache = d["cache"] if wl.kv_format == "bf16" else d["codes"]
    ids = mm.decode_sparse_table(d["q"], cache, d["table"], d["lens"], **kw,
                                 attention_block_table=torch.from_numpy(attn).cuda(),
                                 sparse_block_table_out=st, sparse_context_lens_out=ctx,
                                 block_page_stride=stride, pages_per_block=ppb,
                                 index_scales=d.get("scales"))
    if wl.kv_format == "bf16":
        plain = mm.decode(d["q"], cache, d["table"], d["lens"], **kw)
    else:
        plain = mm.decode_nvfp4(d["q"], cache, d["scales"], d["table"], d["lens"], **kw)
    assert mm.get_device_error() == 0
    ids, plain = ids.cpu().numpy(), plain.cpu().numpy()
    np.testing.assert_array_equal(ids, plain)
    return ids, st.cpu().numpy(), ctx.cpu().numpy()


def check_table(wl, got_ids, got_st, got_ctx, want_ids, attn, ppb, stride, rows, where):
    """got_* are the GPU outputs of the listed batch rows; want_ids the
    oracle's ids of the same rows."""
    sub_attn = np.stack([attn[r // wl.query_len] for r in rows])
    # each row as its own one-query request at its own position
    pos_lens = np.array([wl.seq_lens[r // wl.query_len] - wl.query_len + r % wl.query_len + 1
                         for r in rows], dtype=np.int32)
    want_st, want_ctx = oracle.sparse_table(want_ids, pos_lens, 1, sub_attn, ppb, stride)
    for k, r in enumerate(rows):
        if np.array_equal(got_ids[k], want_ids[k]):
            assert got_st[k].tolist() == want_st[k].tolist(), f"{where} row {r} table"
            assert int(got_ctx[k]) == int(want_ctx[k]), f"{where} row {r} context"
            continue
        # near-tie: the row must describe its own ids
        pos = int(pos_lens[k]) - 1
        ctx = 0
        for s, b in enumerate(got_ids[k]):
            if b < 0:
                assert got_st[k][s * ppb:(s + 1) * ppb].tolist() == [-1] * ppb, where
                continue
            base = int(sub_attn[k][b]) * stride
            assert got_st[k][s * ppb:(s + 1) * ppb].tolist() == list(range(base, base + ppb)), where
            ctx += min(BLOCK, pos + 1 - BLOCK * int(b))
        assert int(got_ctx[k]) == ctx, f"{where} row {r} context (tie row)"


CASES = [
    # seed, reqs, qlen, topk, init, local, min_len, max_len, P, stride multiple, kv format
    (1, 3, 1, 4, 1, 1, 1, 2000, 1, 1, "bf16"),
    (2, 5, 4, 16, 1, 2, 100, 5000, 2, 1, "bf16"),
    (3, 4, 4, 16, 1, 2, 129, 3000, 2, 2, "bf16"),
    (4, 2, 3, 8, 2, 2, 3, 900, 4, 2, "bf16"),
    (5, 9, 1, 16, 1, 2, 16000, 40000, 8, 1, "bf16"),      # requests split across CTAs
    (6, 40, 4, 16, 1, 2, 4, 700, 1, 2, "bf16"),            # short requests: nb < topk, -1 slots
    (7, 3, 2, 16, 0, 0, 5000, 9000, 16, 2, "bf16"),        # no forced blocks
    (8, 6, 4, 16, 1, 2, 2000, 20000, 2, 2, "nvfp4"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}-{c[10]}-P{c[8]}")
def test_sparse_table_matches_oracle(mm, case):
    seed, reqs, qlen, topk, init, local, lo, hi, ppb, mul, fmt = case
    wl = W.random_case(seed, num_reqs=reqs, query_len=qlen, heads=1, topk=topk,
                       init_blocks=init, local_blocks=local, min_len=lo, max_len=hi,
                       kv_format=fmt)
    attn = W.attention_block_table(wl, seed)
    ids, st, ctx = run(mm, wl, attn, ppb, mul * ppb)
    s, want = oracle.problem(wl)
    check_ids(ids, want, s, wl, where=f"sparse seed{seed}")
    rows = list(range(wl.rows))
    check_table(wl, ids[0], st, ctx, want[0], attn, ppb, mul * ppb, rows, f"seed{seed}")


def test_sparse_table_full_size_spec_decode_sampled(mm):
    wl = W.make("spec_decode")
    attn = W.attention_block_table(wl, 1)
    ids, st, ctx = run(mm, wl, attn, 2, 4)
    rng = np.random.default_rng(0)
    order = np.argsort(wl.seq_lens)
    reqs = sorted(set([int(order[0]), int(order[-1])] +
                      [int(x) for x in rng.choice(wl.num_reqs, size=4, replace=False)]))
    sub = oracle.subset(wl, reqs)
    s, want = oracle.problem(sub)
    rows = [i * wl.query_len + j for i in reqs for j in range(wl.query_len)]
    check_ids(ids[:, rows], want, s, sub, where="spec sparse")
    check_table(wl, ids[0, rows], st[rows], ctx[rows], want[0], attn, 2, 4, rows, "spec sparse")


def test_sparse_table_empty_batch_and_graph_replay(mm):
    import torch
    wl = W.random_case(11, num_reqs=5, query_len=4, heads=1, topk=16, init_blocks=1,
                       local_blocks=2, min_len=3000, max_len=30000)
    attn = W.attention_block_table(wl, 11)
    d = to_device(wl)
    st = torch.full((wl.rows, 32), -5, dtype=torch.int32, device="cuda")
    ctx = torch.full((wl.rows,), -5, dtype=torch.int32, device="cuda")
    out = torch.empty((1, wl.rows, 16), dtype=torch.int32, device="cuda")
    ws = mm.new_workspace(mm.OP_DECODE, 1, wl.num_reqs, 4, wl.max_seq_len, 16)
    at = torch.from_numpy(attn).cuda()
    kw = dict(query_len=4, max_seq_len=wl.max_seq_len, topk=16, init_blocks=1, local_blocks=2,
              sm_scale=wl.sm_scale, attention_block_table=at, sparse_block_table_out=st,
              sparse_context_lens_out=ctx, block_page_stride=2, pages_per_block=2, out=out,
              workspace=ws)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()        # inputs were copied on the default stream
    with torch.cuda.stream(stream):
        mm.decode_sparse_table(d["q"], d["cache"], d["table"], d["lens"], **kw, stream=stream)
        torch.cuda.synchronize()
        first = (st.clone(), ctx.clone())
        st.fill_(-5)
        ctx.fill_(-5)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            mm.decode_sparse_table(d["q"], d["cache"], d["table"], d["lens"], **kw,
                                   stream=torch.cuda.current_stream())
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st, first[0]) and torch.equal(ctx, first[1])
    assert mm.get_device_error() == 0
    s, want = oracle.problem(wl)
    check_ids(out.cpu().numpy(), want, s, wl, where="graph sparse")
    check_table(wl, out.cpu().numpy()[0], st.cpu().numpy(), ctx.cpu().numpy(), want[0], attn, 2, 2,
                list(range(wl.rows)), "graph sparse")
    # an empty batch writes nothing
    e = wl.seq_lens[:0]
    mm.decode_sparse_table(d["q"][:0], d["cache"], d["table"][:0], torch.from_numpy(e).cuda(),
                           **{**kw, "attention_block_table": at[:0], "out": None,
                              "workspace": None})
    torch.cuda.synchronize()

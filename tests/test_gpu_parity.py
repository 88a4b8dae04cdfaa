"""GPU parity: every CUDA entry point against the CPU oracle on the same seeded
inputs.  Small cases span several tiles, CTA splits and ragged tails and are
compared element by element; the named full-size workloads are compared on
sampled rows the oracle computes one by one."""

import math

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, check_scores, decode_sample, prefill_sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mm(cuda_device):
    import sparse_attention_block_paged_gb300 as m
    return m


def run_decode(mm, wl, **kw):
    d = to_device(wl)
    args = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
                init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    args.update(kw)
    if wl.kv_format == "bf16":
        ids = mm.decode(d["q"], d["cache"], d["table"], d["lens"], **args)
    else:
        ids = mm.decode_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"], **args)
    return ids.cpu().numpy()


def run_scores(mm, wl):
    d = to_device(wl)
    s = mm.score(d["q"], d["cache"], d["table"], d["lens"], query_len=wl.query_len,
                 max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale)
    return s.cpu().numpy()


def run_prefill(mm, wl):
    d = to_device(wl)
    ids = mm.prefill(d["q"], d["cache"], d["table"], d["lens"], query_len=wl.query_len,
                     max_seq_len=wl.max_seq_len, topk=wl.topk, init_blocks=wl.init_blocks,
                     local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)
    return ids.cpu().numpy()


# ------------------------------------------------------------ tiny workload

def test_tiny_decode_exact(mm):
    wl = W.make("tiny")
    s, want = oracle.problem(wl)
    got = run_decode(mm, wl)
    np.testing.assert_array_equal(got, want)
    check_scores(run_scores(mm, wl), s, "tiny scores")
    assert mm.get_device_error() == 0


# --------------------------------------------------- small decode sweeps

DECODE_CASES = [
    # seed, reqs, qlen, heads, topk, init, local, min_len, max_len
    (1, 3, 1, 1, 4, 1, 1, 1, 2000),
    (2, 5, 4, 1, 16, 1, 2, 100, 5000),
    (3, 4, 4, 4, 16, 1, 2, 129, 3000),
    (4, 2, 3, 2, 8, 2, 2, 3, 900),
    (5, 6, 2, 8, 32, 2, 3, 128, 4096),
    (6, 1, 8, 4, 16, 0, 0, 5000, 9000),
    (7, 9, 1, 1, 16, 1, 2, 16000, 40000),
    (8, 2, 4, 1, 5, 1, 2, 128, 130),
    (9, 3, 16, 2, 12, 3, 1, 200, 2600),
    (10, 40, 4, 1, 16, 1, 2, 1, 700),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"seed{c[0]}")
def test_decode_matches_oracle(mm, case):
    seed, reqs, qlen, heads, topk, init, local, lo, hi = case
    wl = W.random_case(seed, num_reqs=reqs, query_len=qlen, heads=heads, topk=topk,
                       init_blocks=init, local_blocks=local, min_len=lo, max_len=hi)
    s, want = oracle.problem(wl)
    got = run_decode(mm, wl)
    check_ids(got, want, s, wl, where=f"decode seed{seed}")
    check_scores(run_scores(mm, wl), s, f"scores seed{seed}")
    assert mm.get_device_error() == 0


def test_decode_reused_workspace_and_graph_replay(mm):
    import torch
    wl = W.random_case(31, num_reqs=6, query_len=4, heads=2, topk=16, init_blocks=1,
                       local_blocks=2, min_len=3000, max_len=30000)
    s, want = oracle.problem(wl)
    d = to_device(wl)
    ws = mm.new_workspace(mm.OP_DECODE, wl.heads, wl.num_reqs, wl.query_len, wl.max_seq_len, wl.topk)
    out = torch.full((wl.heads, wl.rows, wl.topk), -7, dtype=torch.int32, device="cuda")
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
              init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale,
              out=out, workspace=ws)
    for _ in range(3):
        out.fill_(-7)
        mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw)
        check_ids(out.cpu().numpy(), want, s, wl, where="reuse")
    # stale partial lists do not matter, only the tickets (the first bytes,
    # returned to zero by every completed call) must be zero
    n_tickets = (wl.num_reqs * 4 + 255) // 256 * 256
    assert int(ws[:n_tickets].sum()) == 0
    ws[n_tickets:].fill_(0xA5)
    out.fill_(-7)
    mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw)
    check_ids(out.cpu().numpy(), want, s, wl, where="dirty workspace")
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw)   # warm up on this stream
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            mm.decode(d["q"], d["cache"], d["table"], d["lens"], **kw)
    for _ in range(3):
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        check_ids(out.cpu().numpy(), want, s, wl, where="graph")


# ---------------------------------------------------------- prefill

PREFILL_CASES = [
    # seed, seq_lens, query_len, heads, topk, init, local
    (1, [700], 700, 1, 4, 1, 1),
    (2, [300, 1000], 300, 2, 8, 1, 2),          # prefix 700 on request 1: unaligned tiles
    (3, [1280], 1280, 1, 16, 1, 2),
    (4, [2000, 2000, 777], 257, 1, 16, 2, 2),   # ragged last tile, different prefixes
    (5, [4096], 1500, 4, 32, 1, 3),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: f"seed{c[0]}")
def test_prefill_matches_oracle(mm, case):
    seed, seq, qlen, heads, topk, init, local = case
    wl = W.build(f"prefill-{seed}", seed=seed, seq_lens=seq, query_len=qlen, heads=heads,
                 topk=topk, init_blocks=init, local_blocks=local, max_seq_len=max(seq) + 64)
    s, want = oracle.problem(wl)
    check_scores(run_scores(mm, wl), s, f"prefill scores seed{seed}")
    check_ids(run_prefill(mm, wl), want, s, wl, where=f"prefill seed{seed}")
    assert mm.get_device_error() == 0


@pytest.mark.parametrize("topk,init,local", [(16, 1, 2), (4, 0, 0), (9, 3, 2), (32, 1, 2),
                                             (17, 0, 0), (25, 4, 3),
                                             # 16-key lists keeping 8, 12, 14, 15, 16 slots
                                             (12, 2, 2), (16, 2, 2), (16, 1, 1), (16, 0, 1),
                                             (16, 0, 0)])
def test_fused_prefill_selection_equals_two_kernels(mm, topk, init, local):
    """The prefill kernel selects as it scores (16-key lists for topk <= 16,
    else 32; of a 16-key list only the topk - init - local slots a row can
    need are kept).  Its ids must be those of the score kernel followed by the
    selector, bit for bit (the same fp32 scores and the same keys)."""
    wl = W.random_case(70 + topk, num_reqs=3, query_len=700, heads=2, topk=topk,
                       init_blocks=init, local_blocks=local, min_len=700,
                       max_len=5000 if topk <= 16 else 12000)
    d = to_device(wl)
    fused = run_prefill(mm, wl)
    sc = mm.score(d["q"], d["cache"], d["table"], d["lens"], query_len=wl.query_len,
                  max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale)
    two = mm.topk(sc, d["lens"], query_len=wl.query_len, max_seq_len=wl.max_seq_len,
                  topk=topk, init_blocks=init, local_blocks=local).cpu().numpy()
    np.testing.assert_array_equal(fused, two)
    s, want = oracle.problem(wl)
    check_ids(fused, want, s, wl, where=f"fused topk{topk}")
    assert mm.get_device_error() == 0


@pytest.mark.parametrize("topk,ties", [(16, "some"), (4, "some"), (24, "some"), (32, "some"),
                                       (32, "none"), (20, "many"), (32, "all")])
def test_topk_selector_bit_exact_on_same_scores(mm, topk, ties):
    """Given the same fp32 scores, selection must agree bit for bit.  The
    selector thresholds each 256-block chunk on the lane maxima (topk - forced
    <= 16) or on the lanes' best four (above); "many" and "all" put more than
    32 scores at the threshold, which takes its one-at-a-time path."""
    import torch
    rng = np.random.default_rng(5 + topk)
    seq = rng.integers(1, 20000 if topk > 16 else 9000, size=37).astype(np.int32)
    qlen, heads = 3, 2
    seq = np.maximum(seq, qlen)
    msl = int(seq.max())
    W_ = -(-msl // 128)
    sc = rng.standard_normal((heads, len(seq) * qlen, W_)).astype(np.float32)
    if ties == "some":
        sc[:, :, ::7] = sc[:, :, 3:4]          # plenty of exact ties
    elif ties == "many":
        sc[:, :, ::3] = np.float32(2.5)        # a third of the blocks tie near the top
    elif ties == "all":
        sc[:] = np.float32(0.75)               # the lowest ids win
    want = oracle.select_problem(sc.astype(np.float64), seq, qlen, topk, 1, 2)
    got = mm.topk(torch.from_numpy(sc).cuda(), torch.from_numpy(seq).cuda(), query_len=qlen,
                  max_seq_len=msl, topk=topk, init_blocks=1, local_blocks=2)
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    assert mm.get_device_error() == 0


# ------------------------------------------------------------------ NVFP4

NVFP4_DECODE_CASES = [
    # seed, query_len, heads, topk, init, local: rows per request 1..32 cover
    # one, two and four 8-row query tiles of the kernel, 16- and 32-key lists
    (1, 4, 1, 16, 1, 2),
    (2, 4, 1, 16, 1, 2),
    (3, 4, 1, 16, 1, 2),
    (4, 1, 1, 4, 1, 1),
    (5, 3, 4, 16, 1, 2),     # 12 rows
    (6, 8, 2, 32, 2, 3),     # 16 rows, 32-key lists
    (7, 4, 8, 24, 1, 2),     # 32 rows, 32-key lists
]


@pytest.mark.parametrize("case", NVFP4_DECODE_CASES, ids=lambda c: f"seed{c[0]}")
def test_nvfp4_decode_matches_oracle(mm, case):
    seed, qlen, heads, topk, init, local = case
    wl = W.random_case(seed, num_reqs=5, query_len=qlen, heads=heads, topk=topk,
                       init_blocks=init, local_blocks=local, min_len=500, max_len=20000,
                       kv_format="nvfp4")
    s, want = oracle.problem(wl)
    got = run_decode(mm, wl)
    check_ids(got, want, s, wl, where=f"nvfp4 seed{seed}")
    assert mm.get_device_error() == 0


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"seed{c[0]}")
def test_nvfp4_decode_sweep_matches_oracle(mm, case):
    """The bf16 decode sweep (tiny and single-block requests, fewer blocks
    than CTAs, 1-16 rows per request, topk 4-32) over NVFP4 pages: ids and
    the score call's scores against the oracle."""
    seed, reqs, qlen, heads, topk, init, local, lo, hi = case
    wl = W.random_case(100 + seed, num_reqs=reqs, query_len=qlen, heads=heads, topk=topk,
                       init_blocks=init, local_blocks=local, min_len=lo, max_len=hi,
                       kv_format="nvfp4")
    s, want = oracle.problem(wl)
    check_ids(run_decode(mm, wl), want, s, wl, where=f"nvfp4 sweep seed{seed}")
    d = to_device(wl)
    sc = mm.score_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"],
                        query_len=wl.query_len, max_seq_len=wl.max_seq_len,
                        sm_scale=wl.sm_scale).cpu().numpy()
    check_scores(sc, s, f"nvfp4 sweep scores seed{seed}")
    assert mm.get_device_error() == 0


def test_nvfp4_equals_bf16_path_on_dequantised_cache(mm):
    """The NVFP4 kernel's dequantised keys are exact bf16 values, so scoring the
    oracle-dequantised cache on the bf16 path must give the same ids."""
    wl = W.random_case(9, num_reqs=4, query_len=4, heads=1, topk=16, init_blocks=1,
                       local_blocks=2, min_len=2000, max_len=9000, kv_format="nvfp4")
    got4 = run_decode(mm, wl)
    import copy
    bf = copy.copy(wl)
    bf.kv_format = "bf16"
    bf.cache = oracle.nvfp4_dequant_bf16(wl.codes, wl.scales)
    got16 = run_decode(mm, bf)
    np.testing.assert_array_equal(got4, got16)


def test_nvfp4_extreme_scales(mm):
    """Scales near the subnormal floor and near saturation (6 * 448)."""
    wl = W.random_case(12, num_reqs=3, query_len=2, heads=1, topk=8, init_blocks=1,
                       local_blocks=1, min_len=300, max_len=3000, kv_format="nvfp4")
    rng = np.random.default_rng(3)
    choices = np.array([0x01, 0x02, 0x07, 0x08, 0x09, 0x7E, 0x7D, 0x77, 0x38, 0xB8], dtype=np.uint8)
    wl.scales[:] = rng.choice(choices, size=wl.scales.shape)
    s, want = oracle.problem(wl)
    got = run_decode(mm, wl)
    check_ids(got, want, s, wl, where="nvfp4 extremes")


# ------------------------------------------------------------ edge cases

def test_padding_and_no_forced_blocks(mm):
    wl = W.random_case(40, num_reqs=4, query_len=2, heads=2, topk=32, init_blocks=0,
                       local_blocks=0, min_len=2, max_len=3000)
    s, want = oracle.problem(wl)
    check_ids(run_decode(mm, wl), want, s, wl, where="pad")


def test_empty_batch_is_noop(mm):
    import torch
    q = torch.zeros((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    lens = torch.zeros((0,), dtype=torch.int32, device="cuda")
    ids = mm.decode(q, cache, table, lens, query_len=1, max_seq_len=512, topk=4, init_blocks=1,
                    local_blocks=1, sm_scale=0.1)
    assert ids.shape == (1, 0, 4)


def test_device_status_for_bad_lengths_and_pages(mm):
    wl = W.random_case(41, num_reqs=3, query_len=2, heads=1, topk=4, init_blocks=1,
                       local_blocks=1, min_len=300, max_len=900)
    wl.seq_lens[1] = 1                       # shorter than query_len
    s, want = oracle.problem(wl)
    got = run_decode(mm, wl)
    assert mm.get_device_error() & mm.DEV_SEQ_TOO_SHORT
    check_ids(got, want, s, wl, where="short")
    bad = W.random_case(42, num_reqs=2, query_len=1, heads=1, topk=4, init_blocks=1,
                        local_blocks=1, min_len=600, max_len=900)
    bad.block_table[0, 1] = bad.num_pages + 3   # out of range page
    run_decode(mm, bad)
    assert mm.get_device_error() & mm.DEV_BAD_PAGE
    assert mm.get_device_error() == 0           # read-and-clear


# ------------------------------------------------- full-size named workloads

def _sample_rows(wl, reqs):
    return [i * wl.query_len + j for i in reqs for j in range(wl.query_len)]


@pytest.mark.parametrize("key", ["spec_decode", "high_batch", "nvfp4_decode"])
def test_full_size_decode_sampled(mm, key):
    """The named decode batches in the bench's launch configuration: ids of
    the whole batch in one call, checked on at least 16 requests (the
    shortest, the longest, requests split across CTAs, random others); for
    the bf16 batches also the score call's scores on the same rows."""
    import torch
    wl = W.make(key)
    got = run_decode(mm, wl)
    assert mm.get_device_error() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    reqs, split = decode_sample(wl, sms)
    assert len(reqs) >= 16 and any(r in split for r in reqs)
    sub = oracle.subset(wl, reqs)
    s, want = oracle.problem(sub)
    rows = _sample_rows(wl, reqs)
    check_ids(got[:, rows], want, s, sub, where=key)
    if wl.kv_format == "bf16":
        sc = run_scores(mm, wl)
        assert mm.get_device_error() == 0
        check_scores(sc[:, rows], s, f"{key} scores")


def _prefill_rows_check(wl, rows, ids, scores=None, where=""):
    from helpers import check_ids_row
    for r in rows:
        s, want = oracle.row(wl, r, 0)
        c = len(s) - 1
        check_ids_row(ids[0, r], want, s, c, wl.topk, wl.init_blocks, wl.local_blocks,
                      where=f"{where} row {r}")
        if scores is not None:
            full = np.full(scores.shape[2], -np.inf)
            full[:len(s)] = s
            check_scores(scores[0, r][None], full[None], f"{where} scores row {r}")


def test_full_size_prefill_sampled(mm):
    """The 32768-token causal prefill: the fused ids (scorer with selection)
    and the score call (the score-mode kernel the prefill roofline is timed
    on), checked on every 61st row and the first and last 256 rows."""
    wl = W.make("prefill")
    ids = run_prefill(mm, wl)
    assert mm.get_device_error() == 0
    sc = run_scores(mm, wl)
    assert mm.get_device_error() == 0
    _prefill_rows_check(wl, prefill_sample_rows(wl.rows), ids, sc, where="prefill")


def test_full_size_prefill_topk32_sampled(mm):
    """The 32768-token causal prefill at topk 32 (32-key lists in the
    scorer), ids checked on the bf16 prefill's sample rows."""
    wl = W.make("prefill_topk32")
    ids = run_prefill(mm, wl)
    assert mm.get_device_error() == 0
    _prefill_rows_check(wl, prefill_sample_rows(wl.rows), ids, where="prefill topk32")
    # Every row: the score call followed by the standalone selector (its
    # lanes' best-four threshold at topk 32) picks the same ids bit for bit.
    d = to_device(wl)
    sc = mm.score(d["q"], d["cache"], d["table"], d["lens"], query_len=wl.query_len,
                  max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale)
    two = mm.topk(sc, d["lens"], query_len=wl.query_len, max_seq_len=wl.max_seq_len,
                  topk=wl.topk, init_blocks=wl.init_blocks,
                  local_blocks=wl.local_blocks).cpu().numpy()
    assert mm.get_device_error() == 0
    np.testing.assert_array_equal(ids, two)


def test_full_size_nvfp4_prefill_sampled(mm):
    """The 32768-token NVFP4 causal prefill (dequantised copy, then the fused
    scorer), ids and scores checked on the same rows as the bf16 prefill."""
    wl = W.make("nvfp4_prefill")
    d = to_device(wl)
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale)
    ids = mm.prefill_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"], topk=wl.topk,
                           init_blocks=wl.init_blocks, local_blocks=wl.local_blocks,
                           **kw).cpu().numpy()
    sc = mm.score_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"],
                        **kw).cpu().numpy()
    assert mm.get_device_error() == 0
    _prefill_rows_check(wl, prefill_sample_rows(wl.rows), ids, sc, where="nvfp4 prefill")


def test_fused_prefill_workspace_reuse_and_graph_replay(mm):
    """The fused selection keeps tile records and candidate lists in the workspace.
    A larger batch, then a smaller one, then a graph replay of the smaller
    one on the same workspace: each must match the oracle (records and
    lists of the earlier call must not leak into the later one)."""
    import torch
    big = W.random_case(81, num_reqs=3, query_len=900, heads=2, topk=16, init_blocks=1,
                        local_blocks=2, min_len=900, max_len=6000, max_seq_len=6000)
    small = W.random_case(82, num_reqs=2, query_len=300, heads=2, topk=16, init_blocks=1,
                          local_blocks=2, min_len=300, max_len=2000, max_seq_len=6000)
    ws = torch.full((mm.workspace_bytes(mm.OP_PREFILL, 2, 3, 900, 6000, 16),), 0xA5,
                    dtype=torch.uint8, device="cuda")
    kw = lambda wl: dict(query_len=wl.query_len, max_seq_len=6000, topk=16,  # noqa: E731
                         init_blocks=1, local_blocks=2, sm_scale=wl.sm_scale, workspace=ws)
    for wl in (big, small):
        d = to_device(wl)
        got = mm.prefill(d["q"], d["cache"], d["table"], d["lens"], **kw(wl)).cpu().numpy()
        s, want = oracle.problem(wl)
        check_ids(got, want, s, wl, where=f"reuse {wl.name}")
    d = to_device(small)
    out = torch.full((2, small.rows, 16), -9, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        mm.prefill(d["q"], d["cache"], d["table"], d["lens"], **kw(small), out=out, stream=stream)
        torch.cuda.synchronize()
        out.fill_(-9)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            mm.prefill(d["q"], d["cache"], d["table"], d["lens"], **kw(small), out=out,
                       stream=torch.cuda.current_stream())
        g.replay()
    torch.cuda.synchronize()
    s, want = oracle.problem(small)
    check_ids(out.cpu().numpy(), want, s, small, where="graph fused prefill")
    assert mm.get_device_error() == 0

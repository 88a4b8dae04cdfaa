"""Pins for the CPU oracle: each test checks it against something other than
itself -- brute force written independently in numpy, closed forms, invariants,
special cases that reduce to a library routine, and library fp8 conversions.
No test here needs a GPU.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

BLOCK = 128


# --------------------------------------------------------------- brute force

def brute_force(wl, scale=None):
    """Score every visible token of every row into a dense matrix, take block
    maxima by reshaping, fully sort all blocks, then apply the forced rule.

    Independent of the oracle's code: numpy matmul in float64 over the
    request's logical key sequence, built by gathering whole pages."""
    scale = wl.sm_scale if scale is None else scale
    H, R = wl.heads, wl.rows
    scores = np.full((H, R, wl.width), -np.inf)
    ids = np.full((H, R, wl.topk), -1, dtype=np.int32)
    # query rows of request i: cu[i] .. cu[i+1]-1 (ragged) or query_len each
    cu = (wl.cu_seqlens if wl.cu_seqlens is not None
          else np.arange(wl.num_reqs + 1) * wl.query_len)
    for i in range(wl.num_reqs):
        nbmax = -(-int(wl.seq_lens[i]) // BLOCK)
        if nbmax == 0:
            continue
        if wl.kv_format == "bf16":
            pages = wl.cache[wl.block_table[i, :nbmax]]
        else:
            pages = oracle.nvfp4_dequant_bf16(wl.codes[wl.block_table[i, :nbmax]],
                                              wl.scales[wl.block_table[i, :nbmax]])
        keys = W.bf16_to_f32(pages).astype(np.float64).reshape(nbmax * BLOCK, 128)
        ql = int(cu[i + 1] - cu[i])
        for j in range(ql):
            r = int(cu[i]) + j
            pos = int(wl.seq_lens[i]) - ql + j
            if pos < 0:
                continue
            q = W.bf16_to_f32(wl.q[r]).astype(np.float64)          # [H, 128]
            dense = q @ keys.T                                      # [H, tokens]
            dense[:, pos + 1:] = -np.inf
            nb = pos // BLOCK + 1
            bmax = dense[:, :nb * BLOCK].reshape(H, nb, BLOCK).max(axis=2) * scale
            scores[:, r, :nb] = bmax
            c = nb - 1
            forced = {b for b in range(nb)
                      if b < wl.init_blocks or b >= c - wl.local_blocks + 1}
            for h in range(H):
                order = sorted(range(nb), key=lambda b: (-bmax[h, b], b))
                picks = [b for b in order if b not in forced]
                picks = picks[:wl.topk - len(forced)]
                sel = sorted(forced | set(picks))
                ids[h, r, :len(sel)] = sel
    return scores, ids


def tiny_cases():
    rng = np.random.default_rng(7)
    cases = []
    for k in range(200):
        query_len = int(rng.integers(1, 5))
        heads = int(rng.choice([1, 2, 4]))
        topk = int(rng.choice([2, 3, 4, 6, 8]))
        init = int(rng.integers(0, 3))
        local = int(rng.integers(0, 3))
        while init + local > topk:
            local -= 1
            if local < 0:
                local, init = 0, init - 1
        # lengths cluster around multiples of 128 so partial blocks and
        # block-boundary queries are common
        base = int(rng.integers(0, 9)) * BLOCK
        seq = [max(query_len, base + int(rng.integers(-3, 4))) for _ in range(int(rng.integers(1, 4)))]
        cases.append(dict(seed=10_000 + k, seq_lens=seq, query_len=query_len,
                          heads=heads, topk=topk, init_blocks=init,
                          local_blocks=local, max_seq_len=max(seq) + int(rng.integers(0, 300))))
    return cases


@pytest.mark.parametrize("case", tiny_cases(), ids=lambda c: str(c["seed"]))
def test_oracle_matches_brute_force(case):
    wl = W.build("tiny-bf", **case)
    s_o, i_o = oracle.problem(wl)
    s_b, i_b = brute_force(wl)
    fin = np.isfinite(s_b)
    assert np.array_equal(np.isfinite(s_o), fin)
    np.testing.assert_allclose(s_o[fin], s_b[fin], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(i_o, i_b)


@pytest.mark.parametrize("seed", range(12))
def test_oracle_matches_brute_force_nvfp4(seed):
    rng = np.random.default_rng(seed)
    seq = [int(x) for x in rng.integers(1, 700, size=2)]
    wl = W.build("tiny-fp4", seed=seed, seq_lens=seq, query_len=int(rng.integers(1, 4)),
                 heads=1, topk=4, init_blocks=1, local_blocks=1,
                 max_seq_len=max(seq), kv_format="nvfp4")
    wl.seq_lens = np.maximum(wl.seq_lens, wl.query_len).astype(np.int32)
    s_o, i_o = oracle.problem(wl)
    s_b, i_b = brute_force(wl)
    fin = np.isfinite(s_b)
    np.testing.assert_allclose(s_o[fin], s_b[fin], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(i_o, i_b)


# -------------------------------------------------- library special case

def test_single_request_prefill_is_causal_matmul():
    """One request, identity block table, query_len = seq_len: the pre-max
    matrix is numpy.matmul(Q, K^T) under a causal mask."""
    seq = 3 * BLOCK + 17
    wl = W.build("ident", seed=3, seq_lens=[seq], query_len=seq, heads=1,
                 topk=4, init_blocks=1, local_blocks=1, max_seq_len=seq,
                 pool_pages=4, poison=False)
    nb = -(-seq // BLOCK)
    wl.block_table[0, :nb] = np.arange(nb)
    s_o, _ = oracle.problem(wl)
    Q = W.bf16_to_f32(wl.q[:, 0]).astype(np.float64)
    K = W.bf16_to_f32(wl.cache[:nb]).astype(np.float64).reshape(-1, 128)[:seq]
    S = np.matmul(Q, K.T)
    S[np.triu_indices(seq, 1)] = -np.inf
    Spad = np.full((seq, nb * BLOCK), -np.inf)
    Spad[:, :seq] = S
    expect = Spad.reshape(seq, nb, BLOCK).max(axis=2) * wl.sm_scale
    np.testing.assert_allclose(s_o[0], expect, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------- closed forms

def planted(alphas, seq, init=1, local=1, topk=4, ties=False):
    """Keys of chosen blocks are alpha*q (one token per block), everything
    else small noise; block b's score is then sm_scale*alpha_b*|q|^2."""
    wl = W.build("plant", seed=5, seq_lens=[seq], query_len=1, heads=1,
                 topk=topk, init_blocks=init, local_blocks=local,
                 max_seq_len=seq, poison=False)
    rng = np.random.default_rng(11)
    q = np.zeros(128, np.float32)
    q[:8] = 1.0                                   # |q|^2 = 8, exact in bf16
    wl.q[0, 0] = W.bf16_bits(q)
    nb = -(-seq // BLOCK)
    for b in range(nb):
        p = wl.block_table[0, b]
        wl.cache[p] = W.bf16_bits(rng.uniform(-1e-3, 1e-3, (BLOCK, 128)).astype(np.float32))
    for b, a in alphas.items():
        p = wl.block_table[0, b]
        wl.cache[p, 5] = W.bf16_bits(np.float32(a) * q)
    return wl


def test_planted_winners_and_scores():
    seq = 10 * BLOCK
    alphas = {3: 2.0, 7: 4.0, 5: 3.0, 2: 1.0}
    wl = planted(alphas, seq, init=1, local=1, topk=4)
    s, ids = oracle.row(wl, 0, 0)
    for b, a in alphas.items():
        assert s[b] == pytest.approx(wl.sm_scale * a * 8.0, rel=1e-12)
    # forced {0, 9}; the two best candidates are 7 (alpha 4) and 5 (alpha 3)
    assert list(ids) == [0, 5, 7, 9]


def test_planted_exact_tie_goes_to_lower_id():
    seq = 10 * BLOCK
    wl = planted({6: 3.0, 4: 3.0, 2: 3.0}, seq, init=1, local=1, topk=3)
    _, ids = oracle.row(wl, 0, 0)
    assert list(ids) == [0, 2, 9]


def test_select_ties_and_forced_rule():
    s = np.array([0.0, 5.0, 5.0, 1.0, 5.0, 2.0])
    # forced: init {0}, local 2 -> {4, 5}; candidates 1,2,3 ranked 1,2 (tie) then 3
    assert list(oracle.select(s, 4, 1, 2)) == [0, 1, 4, 5]
    assert list(oracle.select(s, 5, 1, 2)) == [0, 1, 2, 4, 5]
    # fewer visible blocks than topk: all visible, then -1
    assert list(oracle.select(s[:3], 5, 1, 1)) == [0, 1, 2, -1, -1]
    # no forced blocks at all
    assert list(oracle.select(s, 2, 0, 0)) == [1, 2]
    # init and local overlap on a short row
    assert list(oracle.select(s[:2], 4, 2, 2)) == [0, 1, -1, -1]
    # empty row
    assert list(oracle.select(s[:0], 3, 1, 1)) == [-1, -1, -1]


# ------------------------------------------------------ hand-checkable case

def test_tiny_decode_by_hand():
    wl = W.make("tiny")
    _, ids = oracle.problem(wl)
    # request 0: seq 300 -> blocks 0..2 visible, fewer than topk 4
    assert list(ids[0, 0]) == [0, 1, 2, -1]
    # request 1: seq 700 -> c = 5, forced {0, 5}, best 2 of {1..4}
    s = oracle.block_scores(wl, 1, 0)
    best = sorted(range(1, 5), key=lambda b: (-s[b], b))[:2]
    assert list(ids[0, 1]) == sorted([0, 5] + best)


def test_tiny_decode_golden():
    """Regression against tests/golden/tiny_decode.txt (written by
    tests/golden/make_golden.py from the oracle alone)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_decode.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    wl = W.make("tiny")
    s, ids = oracle.problem(wl)
    for r in rows:
        row, kind = int(r[0]), r[1]
        vals = r[2:]
        if kind == "ids":
            assert [int(v) for v in vals] == list(ids[0, row])
        else:
            got = s[0, row, :len(vals)]
            np.testing.assert_allclose(got, [float(v) for v in vals], rtol=1e-12)


# ----------------------------------------------------------------- invariants

def _small(seed, **kw):
    base = dict(num_reqs=3, query_len=3, heads=2, topk=5, init_blocks=1,
                local_blocks=2, min_len=200, max_len=1400)
    base.update(kw)
    return W.random_case(seed, **base)


@pytest.mark.parametrize("seed", range(6))
def test_invariants(seed):
    wl = _small(seed)
    s, ids = oracle.problem(wl)
    for h in range(wl.heads):
        for r in range(wl.rows):
            i, j = divmod(r, wl.query_len)
            pos = int(wl.seq_lens[i]) - wl.query_len + j
            c = pos // BLOCK
            nb = c + 1
            row = ids[h, r]
            valid = row[row >= 0]
            forced = {b for b in range(nb) if b < wl.init_blocks or b > c - wl.local_blocks}
            assert forced <= set(valid.tolist())                  # forced present
            assert valid.max() <= c                                # causal bound
            assert len(set(valid.tolist())) == len(valid)          # unique
            assert np.all(np.diff(valid) > 0)                      # ascending
            if (row < 0).any():                                    # -1 only if nb < topk
                assert nb < wl.topk and list(valid) == list(range(nb))
                assert np.all(row[len(valid):] == -1)


def test_page_permutation_invariance():
    wl = _small(21)
    _, ids = oracle.problem(wl)
    s, _ = oracle.problem(wl)
    rng = np.random.default_rng(1)
    perm = rng.permutation(wl.num_pages)
    inv = np.argsort(perm)
    wl2 = _small(21)
    wl2.cache = wl.cache[perm]                      # new page p holds old page perm[p]
    used = wl.block_table < wl.num_pages
    wl2.block_table = np.where(used, inv[np.minimum(wl.block_table, wl.num_pages - 1)],
                               wl.block_table).astype(np.int32)
    s2, ids2 = oracle.problem(wl2)
    np.testing.assert_array_equal(ids, ids2)
    np.testing.assert_array_equal(s, s2)


def test_positive_scale_invariance():
    wl = _small(22)
    _, ids = oracle.problem(wl)
    for sc in (1.0, 0.01, 37.5):
        wl.sm_scale = sc
        s2, ids2 = oracle.problem(wl)
        np.testing.assert_array_equal(ids, ids2)


def test_head_independence():
    wl = _small(23, heads=3)
    s, ids = oracle.problem(wl)
    one = _small(23, heads=3)
    one.q = np.ascontiguousarray(wl.q[:, 1:2])
    one.heads = 1
    s1, ids1 = oracle.problem(one)
    np.testing.assert_array_equal(s[1], s1[0])
    np.testing.assert_array_equal(ids[1], ids1[0])


def test_decode_row_is_last_prefill_row():
    seq = 5 * BLOCK + 40
    pre = W.build("pre", seed=9, seq_lens=[seq], query_len=seq, heads=1, topk=4,
                  init_blocks=1, local_blocks=1, max_seq_len=seq)
    dec = W.build("pre", seed=9, seq_lens=[seq], query_len=seq, heads=1, topk=4,
                  init_blocks=1, local_blocks=1, max_seq_len=seq)
    dec.query_len = 1
    dec.q = pre.q[-1:].copy()
    s_p, i_p = oracle.problem(pre)
    s_d, i_d = oracle.problem(dec)
    np.testing.assert_array_equal(s_p[0, -1], s_d[0, 0])
    np.testing.assert_array_equal(i_p[0, -1], i_d[0, 0])


# ------------------------------------------------------------------- NVFP4

def test_e2m1_values_from_the_spec():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert abs(v) == mags[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e4m3_decode_matches_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        v = oracle.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v)
        else:
            assert v == ref[b] and math.copysign(1, v) == math.copysign(1, ref[b])


def test_e4m3_rounding_matches_torch_in_range():
    """Every NVFP4 product and every midpoint between adjacent e4m3 values:
    the oracle's search-based rounding equals torch's fp32 -> e4m3fn cast
    (round to nearest even) wherever the value is within +-448."""
    vals = set()
    for s in range(256):
        if (s & 0x7F) == 0x7F:
            continue
        for c in range(16):
            vals.add(oracle.e2m1_value(c) * oracle.e4m3_value(s))
    grid = sorted({oracle.e4m3_value(b) for b in range(0x7F)})
    vals.update((a + b) / 2 for a, b in zip(grid, grid[1:]))
    vals.update(-v for v in list(vals))
    x = np.array(sorted(v for v in vals if abs(v) <= 448.0), dtype=np.float64)
    assert np.all(x.astype(np.float32).astype(np.float64) == x)   # exact in fp32
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rn_satfinite(float(v)) for v in x], dtype=np.uint8)
    # torch keeps the sign of zero results; so does the oracle
    np.testing.assert_array_equal(got, ref)


def test_e4m3_satfinite_clamps():
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 2688.0):
        assert oracle.e4m3_rn_satfinite(v) == 0x7E
        assert oracle.e4m3_rn_satfinite(-v) == 0xFE
    # largest NVFP4 product 6 * 448 saturates
    assert oracle.nvfp4_value(7, 0x7E) == 448.0
    assert oracle.nvfp4_value(15, 0x7E) == -448.0


def test_nvfp4_subnormal_results():
    # scale = smallest subnormal 2^-9: 0.5 * 2^-9 = 2^-10 is a tie between
    # 0 and 2^-9 and goes to the even code (0); 1.5 * 2^-9 ties to 2 * 2^-9
    tiny = 0x01
    assert oracle.e4m3_value(tiny) == 2.0 ** -9
    assert oracle.nvfp4_value(1, tiny) == 0.0
    assert oracle.nvfp4_value(3, tiny) == 2.0 ** -8
    assert oracle.nvfp4_value(2, tiny) == 2.0 ** -9
    assert oracle.nvfp4_value(7, tiny) == 6 * 2.0 ** -9


# ------------------------------------------------------- sparse page table

def test_sparse_table_by_hand():
    # seq 300, one query: pos 299, blocks 0..2 (the last holds tokens 256..299).
    # Attention blocks 7, 3, 9; two pages per block, four pages between blocks:
    # block 7 -> pages 28, 29; block 3 -> 12, 13; block 9 -> 36, 37.
    t, c = oracle.sparse_table(np.array([[0, 1, 2, -1]]), np.array([300]), 1,
                               np.array([[7, 3, 9]]), 2, 4)
    assert t.tolist() == [[28, 29, 12, 13, 36, 37, -1, -1]]
    assert c.tolist() == [128 + 128 + 44]
    # seq 700: pos 699 in block 5 (tokens 640..699, 60 of them); blocks 0, 2,
    # 4, 5 selected; one page per block, two pages between blocks.
    t, c = oracle.sparse_table(np.array([[0, 2, 4, 5]]), np.array([700]), 1,
                               np.array([[10, 11, 12, 13, 14, 15]]), 1, 2)
    assert t.tolist() == [[20, 24, 28, 30]]
    assert c.tolist() == [3 * 128 + 60]


def _walk_sparse_attention(table_row, ctx, pages_per_block, attn_row, block_page_stride):
    """(logical token) read by a paged attention that walks `ctx` tokens of the
    compacted table, inverted through the attention cache layout: page
    attn_row[b] * stride + p holds tokens 128 b + p * (128 / P) ...  of block b."""
    per_page = BLOCK // pages_per_block
    where = {}
    for b, blk in enumerate(attn_row):
        for p in range(pages_per_block):
            where[int(blk) * block_page_stride + p] = (b, p)
    out = []
    for u in range(ctx):
        b, p = where[int(table_row[u // per_page])]
        out.append(b * BLOCK + p * per_page + u % per_page)
    return out


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("pages_per_block,stride_mul", [(1, 1), (2, 1), (2, 2), (4, 2), (8, 1)])
def test_sparse_table_walk_reads_exactly_the_selected_visible_tokens(seed, pages_per_block,
                                                                      stride_mul):
    wl = _small(seed, heads=1, topk=6)
    _, ids = oracle.problem(wl)
    rng = np.random.default_rng(100 + seed)
    nblk = wl.block_table.shape[1]
    # distinct physical blocks per request, so the layout can be inverted
    attn = np.stack([rng.permutation(4 * nblk)[:nblk] for _ in range(wl.num_reqs)]).astype(np.int32)
    stride = stride_mul * pages_per_block
    table, ctx = oracle.sparse_table(ids[0], wl.seq_lens, wl.query_len, attn, pages_per_block,
                                     stride)
    for r in range(wl.rows):
        i, j = divmod(r, wl.query_len)
        pos = int(wl.seq_lens[i]) - wl.query_len + j
        sel = set(int(b) for b in ids[0, r] if b >= 0)
        want = [t for t in range(pos + 1) if t // BLOCK in sel]    # token-level enumeration
        assert _walk_sparse_attention(table[r], int(ctx[r]), pages_per_block, attn[i],
                                      stride) == want
        n = len(sel)
        assert np.all(table[r, n * pages_per_block:] == -1)


def test_sparse_table_full_selection_and_identity_layout():
    # every visible block kept (nb <= topk): the sparse context is the whole
    # causal context pos + 1; with one page per block and stride 1 the table
    # row is the attention table's entries for the ids
    wl = _small(3, heads=1, topk=16, min_len=130, max_len=1500)
    _, ids = oracle.problem(wl)
    table, ctx = oracle.sparse_table(ids[0], wl.seq_lens, wl.query_len, wl.block_table, 1, 1)
    for r in range(wl.rows):
        i, j = divmod(r, wl.query_len)
        pos = int(wl.seq_lens[i]) - wl.query_len + j
        assert pos // BLOCK + 1 <= wl.topk
        assert int(ctx[r]) == pos + 1
        valid = ids[0, r][ids[0, r] >= 0]
        assert table[r, :len(valid)].tolist() == wl.block_table[i, valid].tolist()


# ------------------------------------------------------------ ragged batches

def ragged_tiny_cases():
    rng = np.random.default_rng(11)
    cases = []
    for k in range(60):
        n = int(rng.integers(1, 5))
        ql = [int(rng.choice([0, 1, 2, 5, 130, 131])) for _ in range(n)]
        pre = [int(rng.integers(0, 4)) * BLOCK + int(rng.integers(-2, 3)) for _ in range(n)]
        pre = [max(0, p) for p in pre]
        if sum(ql) == 0:
            ql[0] = 3
        topk = int(rng.choice([2, 4, 6]))
        cases.append(dict(seed=20_000 + k, query_lens=ql, prefix_lens=pre,
                          heads=int(rng.choice([1, 2])), topk=topk, init_blocks=1,
                          local_blocks=int(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("case", ragged_tiny_cases(), ids=lambda c: str(c["seed"]))
def test_ragged_oracle_matches_brute_force(case):
    wl = W.ragged_case(**case)
    s_o, i_o = oracle.problem_ragged(wl)
    s_b, i_b = brute_force(wl)
    fin = np.isfinite(s_b)
    assert np.array_equal(np.isfinite(s_o), fin)
    np.testing.assert_allclose(s_o[fin], s_b[fin], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(i_o, i_b)


def test_ragged_with_equal_counts_is_the_uniform_batch():
    wl = W.ragged_case(5, query_lens=[3, 3, 3], prefix_lens=[200, 700, 1000], heads=2, topk=5,
                       init_blocks=1, local_blocks=2)
    s_r, i_r = oracle.problem_ragged(wl)
    import copy
    u = copy.copy(wl)
    u.cu_seqlens = None
    u.query_len = 3
    s_u, i_u = oracle.problem(u)
    np.testing.assert_array_equal(i_r, i_u)
    np.testing.assert_array_equal(s_r, s_u)

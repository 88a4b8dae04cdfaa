"""Comparison rules and device marshalling shared by the GPU tests."""

import numpy as np

SCORE_RTOL = 1e-3   # |d| <= 1e-3 * max(1, |s|)
BLOCK = 128


def to_device(wl, device="cuda"):
    import torch
    q = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).to(device)
    table = torch.from_numpy(np.ascontiguousarray(wl.block_table)).to(device)
    lens = torch.from_numpy(np.ascontiguousarray(wl.seq_lens)).to(device)
    if wl.kv_format == "bf16":
        cache = torch.from_numpy(wl.cache.view(np.int16)).view(torch.bfloat16).to(device)
        return dict(q=q, cache=cache, table=table, lens=lens)
    codes = torch.from_numpy(wl.codes).to(device)
    scales = torch.from_numpy(wl.scales).to(device)
    return dict(q=q, codes=codes, scales=scales, table=table, lens=lens)


def check_scores(got, want, where=""):
    """got fp32, want fp64, same shape; -inf exactly where the oracle has -inf."""
    got = np.asarray(got, dtype=np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{where}: -inf pattern differs"
    assert np.all(got[~fin] == want[~fin]), f"{where}: non-finite values differ"
    err = np.abs(got[fin] - want[fin])
    tol = SCORE_RTOL * np.maximum(1.0, np.abs(want[fin]))
    bad = err > tol
    assert not bad.any(), f"{where}: {bad.sum()} scores off, worst {err.max():.3g}"


def forced_set(c, init_blocks, local_blocks):
    if c < 0:
        return set()
    return {b for b in range(c + 1) if b < init_blocks or b > c - local_blocks}


def check_ids_row(got_row, want_row, scores, c, topk, init_blocks, local_blocks, where=""):
    """The comparison rule for one row.  scores: oracle fp64 scores of the
    visible blocks 0..c.  Exact when the selection is decided by more than the
    score tolerance, otherwise a validity check."""
    got_row = [int(x) for x in got_row]
    want_row = [int(x) for x in want_row]
    if got_row == want_row:
        return
    F = forced_set(c, init_blocks, local_blocks)
    cand = sorted((b for b in range(c + 1) if b not in F), key=lambda b: (-scores[b], b))
    m = topk - len(F)
    decided = len(cand) <= m or (scores[cand[m - 1]] - scores[cand[m]]
                                 > SCORE_RTOL * max(1.0, abs(scores[cand[m - 1]])))
    assert not decided, f"{where}: ids {got_row} != oracle {want_row}"
    valid = [x for x in got_row if x >= 0]
    n = len(F) + min(m, len(cand))
    assert len(valid) == n and got_row[n:] == [-1] * (topk - n), f"{where}: bad padding {got_row}"
    assert valid == sorted(set(valid)), f"{where}: not unique ascending {got_row}"
    assert F <= set(valid), f"{where}: forced blocks missing {got_row}"
    kth = scores[cand[m - 1]]
    tol = SCORE_RTOL * max(1.0, abs(kth))
    picks = set(valid) - F
    for b in cand:
        if scores[b] > kth + tol:
            assert b in picks, f"{where}: clear winner {b} missing {got_row}"
    for b in picks:
        assert b in cand and scores[b] >= kth - tol, f"{where}: pick {b} too weak {got_row}"


def row_request(wl, r):
    """(request, index in it, rows of it) of batch row r, uniform or ragged."""
    if wl.cu_seqlens is None:
        i, j = divmod(r, wl.query_len)
        return i, j, wl.query_len
    i = int(np.searchsorted(wl.cu_seqlens, r, side="right")) - 1
    return i, r - int(wl.cu_seqlens[i]), int(wl.cu_seqlens[i + 1] - wl.cu_seqlens[i])


def check_ids(got, want, scores, wl, rows=None, where=""):
    """got/want int32 [H, R, topk] (or the sampled rows), scores fp64 [H, R, W]."""
    H = got.shape[0]
    rows = range(got.shape[1]) if rows is None else rows
    for h in range(H):
        for k, r in enumerate(rows):
            i, j, ql = row_request(wl, r)
            pos = int(min(max(wl.seq_lens[i], 0), wl.max_seq_len)) - ql + j
            c = pos // BLOCK if pos >= 0 else -1
            check_ids_row(got[h, k], want[h, k], scores[h, k], c, wl.topk, wl.init_blocks,
                          wl.local_blocks, where=f"{where} h{h} row{r}")


def split_requests(wl, sms):
    """Requests of a decode batch whose blocks the streaming kernel spreads
    over more than one CTA.  The kernel gives each CTA an equal share of the
    request-major list of positions (each request counts six extra positions
    before its blocks); position x belongs to CTA ((x + 1) * G - 1) // total."""
    nb = (np.minimum(np.maximum(wl.seq_lens.astype(np.int64), 0), wl.max_seq_len) + 127) // 128
    slots = np.where(nb > 0, nb + 6, 0)
    total = int(slots.sum())
    grid = max(1, min(sms, wl.num_reqs * -(-wl.max_seq_len // 128)))
    first = np.concatenate([[0], np.cumsum(slots)[:-1]]) + 6   # each request's first block
    cta = lambda x: ((x + 1) * grid - 1) // total               # noqa: E731
    return [i for i in range(wl.num_reqs) if nb[i] > 0 and cta(first[i]) != cta(first[i] + nb[i] - 1)]


def decode_sample(wl, sms, n=16, seed=0):
    """At least n requests of a decode batch: the shortest, the longest, the
    first and last few split across CTAs, and random others."""
    rng = np.random.default_rng(seed)
    order = np.argsort(wl.seq_lens, kind="stable")
    split = split_requests(wl, sms)
    pick = {int(order[0]), int(order[1]), int(order[-1]), int(order[-2])}
    pick |= set(split[:4]) | set(split[-4:])
    rest = [i for i in range(wl.num_reqs) if i not in pick]
    need = max(0, n - len(pick))
    pick |= set(int(x) for x in rng.choice(rest, size=min(need, len(rest)), replace=False))
    return sorted(pick), split


def prefill_sample_rows(rows, every=61, edge=256):
    """Rows of a long prefill checked one by one: every `every`-th row plus the
    first and last `edge`."""
    return sorted(set(range(0, rows, every)) | set(range(min(edge, rows)))
                  | set(range(max(0, rows - edge), rows)))

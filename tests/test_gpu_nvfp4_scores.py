"""NVFP4 block scores (mm3idx_score_nvfp4) against the CPU oracle.

The NVFP4 element rule (indexer_nvfp4 page, module docstring) is
e4m3_rn_satfinite(e2m1 code * e4m3 scale).  Short query runs are scored by the
streaming decode kernel, which dequantises each page on chip; long ones by
the tensor-core scorer on a bf16 copy.  Both are compared element by element
with the oracle's fp64 scores at the score tolerance, and the decode kernel's
own dequantisation is checked bit for bit on every (code, scale) pair and at
every token position of a page."""

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, check_scores, decode_sample, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mm(cuda_device):
    import sparse_attention_block_paged_gb300 as m
    return m


def nvfp4_scores(mm, wl):
    d = to_device(wl)
    s = mm.score_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"],
                       query_len=wl.query_len, max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale)
    return s.cpu().numpy()


SCORE_CASES = [
    # seed, reqs, qlen, heads, min_len, max_len   (heads * qlen <= 32: streaming kernel)
    (1, 5, 4, 1, 500, 20000),
    (2, 3, 1, 1, 1, 900),
    (3, 4, 8, 4, 129, 5000),
    (4, 9, 2, 2, 16000, 40000),
    (5, 2, 16, 2, 3000, 9000),
    (8, 4, 3, 4, 700, 9000),        # 12 rows: two 8-row query tiles
    # heads * qlen > 32: bf16 copy + tensor-core scorer
    (6, 2, 300, 1, 300, 2000),
    (7, 3, 257, 2, 700, 3000),
]


@pytest.mark.parametrize("case", SCORE_CASES, ids=lambda c: f"seed{c[0]}")
def test_nvfp4_scores_match_oracle(mm, case):
    seed, reqs, qlen, heads, lo, hi = case
    wl = W.random_case(100 + seed, num_reqs=reqs, query_len=qlen, heads=heads, topk=16,
                       init_blocks=1, local_blocks=2, min_len=lo, max_len=hi, kv_format="nvfp4")
    s, _ = oracle.problem(wl)
    check_scores(nvfp4_scores(mm, wl), s, f"nvfp4 scores seed{seed}")
    assert mm.get_device_error() == 0


def test_full_size_nvfp4_decode_scores_sampled(mm):
    """The NVFP4 decode batch (128 requests x 4 rows, 32K-128K tokens): scores
    of the whole batch in one call, checked on sampled requests."""
    import torch
    wl = W.make("nvfp4_decode")
    got = nvfp4_scores(mm, wl)
    assert mm.get_device_error() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    reqs, split = decode_sample(wl, sms)
    assert any(r in split for r in reqs)
    sub = oracle.subset(wl, reqs)
    s, _ = oracle.problem(sub)
    rows = [i * wl.query_len + j for i in reqs for j in range(wl.query_len)]
    check_scores(got[:, rows], s, "nvfp4 decode full size")


def _exhaustive_pages():
    """128 pages; page p isolates token t = p.  Its 8 scale groups take the
    finite e4m3 scale bytes in turn (254 of them, 1024 slots: each scale at
    least 4 times), and group g's 16 elements hold the 16 e2m1 codes rotated
    by p + g.  Tokens before t hold -448 in every element (code -6 at scale
    448 saturates to -448, the smallest value), so the max over tokens 0..t
    is token t's element; tokens after t hold +448, which a row at position
    t must not see."""
    finite = [s for s in range(256) if s not in (0x7F, 0xFF)]
    pages = 128
    codes = np.empty((pages, 128, 64), dtype=np.uint8)
    scales = np.full((pages, 128, 8), 0x7E, dtype=np.uint8)
    nib = np.empty((pages, 128), dtype=np.uint8)        # token t's 128 codes, per page
    for p in range(pages):
        t = p
        codes[p, :t] = 0xFF                              # -6, -6
        codes[p, t + 1:] = 0x77                          # +6, +6
        for g in range(8):
            scales[p, t, g] = finite[(8 * p + g) % len(finite)]
            for i in range(16):
                nib[p, 16 * g + i] = (i + p + g) % 16
        codes[p, t] = nib[p, 0::2] | (nib[p, 1::2] << 4)
    return codes, scales, nib


def test_decode_kernel_dequant_bit_exact(mm):
    """Every (e2m1 code, finite e4m3 scale) pair at every token position of a
    page, through the streaming decode kernel's own dequantisation: request
    r = 4p + k sees token p of page p only (seq_len p + 1); its 32 heads are
    one-hot queries on elements 32k .. 32k+31 with sm_scale 1, so each score
    is one dequantised element, exact in fp32.  Compared bit for bit with the
    oracle's value of the element."""
    import torch
    codes, scales, nib = _exhaustive_pages()
    pages = codes.shape[0]
    reqs = 4 * pages
    heads = 32
    q = np.zeros((reqs, heads, 128), dtype=np.uint16)
    for r in range(reqs):
        k = r % 4
        for h in range(heads):
            q[r, h, 32 * k + h] = 0x3F80                 # bf16 1.0
    table = (np.arange(reqs, dtype=np.int32) // 4).reshape(reqs, 1)
    lens = (np.arange(reqs, dtype=np.int32) // 4) + 1
    dev = torch.device("cuda", 0)
    got = mm.score_nvfp4(
        torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(dev),
        torch.from_numpy(codes).to(dev), torch.from_numpy(scales).to(dev),
        torch.from_numpy(table).to(dev), torch.from_numpy(lens).to(dev),
        query_len=1, max_seq_len=128, sm_scale=1.0).cpu().numpy()
    assert mm.get_device_error() == 0
    value = np.array([[oracle.nvfp4_value(c, s) for c in range(16)] for s in range(256)])
    want = np.empty((heads, reqs), dtype=np.float64)
    for r in range(reqs):
        p, k = divmod(r, 4)
        for h in range(heads):
            e = 32 * k + h
            want[h, r] = value[scales[p, p, e // 16], nib[p, e]]
    assert np.array_equal(got[:, :, 0].astype(np.float64), want), np.argwhere(
        got[:, :, 0].astype(np.float64) != want)[:10]
    # every finite scale byte and every code was exercised
    seen = {(int(scales[p, p, e // 16]), int(nib[p, e])) for p in range(pages) for e in range(128)}
    assert len(seen) == 254 * 16


def _bad_page_case(kv_format, qlen):
    wl = W.random_case(61, num_reqs=3, query_len=qlen, heads=2, topk=8, init_blocks=1,
                       local_blocks=1, min_len=max(qlen, 700), max_len=3000, kv_format=kv_format)
    s, _ = oracle.problem(wl)
    # request 1's block 2 points past the cache: it holds no visible tokens,
    # so every row of the request that sees it scores it -inf
    wl.block_table[1, 2] = wl.num_pages + 5
    s[:, wl.query_len:2 * wl.query_len, 2] = -np.inf
    want = oracle.select_problem(np.where(np.isfinite(s), s, -1e300), wl.seq_lens, wl.query_len,
                                 wl.topk, wl.init_blocks, wl.local_blocks)
    return wl, s, want


@pytest.mark.parametrize("kv_format", ["bf16", "nvfp4"])
@pytest.mark.parametrize("qlen", [2, 300])
def test_bad_page_scores_minus_inf(mm, kv_format, qlen):
    """A block table entry outside the cache: its block gets no visible
    tokens (-inf) and MM3IDX_DEV_BAD_PAGE is set, on the streaming kernel
    (2 rows per request) and on the tensor-core scorer (300 rows), for bf16
    and NVFP4 pages alike; the ids then follow from those scores."""
    wl, s, want = _bad_page_case(kv_format, qlen)
    d = to_device(wl)
    kw = dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, sm_scale=wl.sm_scale)
    sel = dict(topk=wl.topk, init_blocks=wl.init_blocks, local_blocks=wl.local_blocks)
    if kv_format == "bf16":
        got = mm.score(d["q"], d["cache"], d["table"], d["lens"], **kw).cpu().numpy()
        ids = (mm.decode if qlen <= 16 else mm.prefill)(d["q"], d["cache"], d["table"], d["lens"],
                                                        **kw, **sel).cpu().numpy()
    else:
        got = mm.score_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"],
                             **kw).cpu().numpy()
        f = mm.decode_nvfp4 if qlen <= 16 else mm.prefill_nvfp4
        ids = f(d["q"], d["codes"], d["scales"], d["table"], d["lens"], **kw, **sel).cpu().numpy()
    assert mm.get_device_error() & mm.DEV_BAD_PAGE
    check_scores(got, s, f"bad page {kv_format} qlen{qlen}")
    check_ids(ids, want, np.where(np.isfinite(s), s, -1e300), wl,
              where=f"bad page ids {kv_format} qlen{qlen}")
    assert mm.get_device_error() == 0

"""GPU parity of the NVFP4 prefill (mm3idx_prefill_nvfp4) against the oracle:
small causal and chunked cases element by element, the full-size NVFP4
prefill on sampled rows, the equality with the bf16 prefill on the
oracle-dequantised cache, and the dequantised pages themselves, bit for bit,
over every (e2m1 code, e4m3 scale) pair."""

import copy

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import check_ids, check_ids_row, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mm(cuda_device):
    import sparse_attention_block_paged_gb300 as m
    return m


def kwargs(wl):
    return dict(query_len=wl.query_len, max_seq_len=wl.max_seq_len, topk=wl.topk,
                init_blocks=wl.init_blocks, local_blocks=wl.local_blocks, sm_scale=wl.sm_scale)


def run_prefill_nvfp4(mm, wl, workspace=None):
    d = to_device(wl)
    ids = mm.prefill_nvfp4(d["q"], d["codes"], d["scales"], d["table"], d["lens"], **kwargs(wl),
                           workspace=workspace)
    return ids.cpu().numpy()


CASES = [
    # seed, reqs, qlen, heads, topk, init, local, min_len, max_len
    (1, 1, 700, 1, 4, 1, 1, 700, 700),          # whole-request prefill, ragged tail
    (2, 2, 300, 2, 16, 1, 2, 300, 2000),        # chunked: prefix + 300 new tokens
    (3, 3, 129, 1, 8, 2, 2, 129, 5000),
    (4, 1, 1000, 4, 32, 2, 3, 9000, 9000),      # 63-71 blocks a row: 32-key lists
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_nvfp4_prefill_matches_oracle(mm, case):
    seed, reqs, qlen, heads, topk, init, local, lo, hi = case
    wl = W.random_case(seed, num_reqs=reqs, query_len=qlen, heads=heads, topk=topk,
                       init_blocks=init, local_blocks=local, min_len=lo, max_len=hi,
                       kv_format="nvfp4")
    s, want = oracle.problem(wl)
    got = run_prefill_nvfp4(mm, wl)
    check_ids(got, want, s, wl, where=f"nvfp4 prefill seed{seed}")
    assert mm.get_device_error() == 0


def test_nvfp4_prefill_equals_bf16_prefill_on_dequantised_cache(mm):
    wl = W.random_case(7, num_reqs=2, query_len=900, heads=2, topk=16, init_blocks=1,
                       local_blocks=2, min_len=900, max_len=4000, kv_format="nvfp4")
    got4 = run_prefill_nvfp4(mm, wl)
    bf = copy.copy(wl)
    bf.kv_format = "bf16"
    bf.cache = oracle.nvfp4_dequant_bf16(wl.codes, wl.scales)
    d = to_device(bf)
    got16 = mm.prefill(d["q"], d["cache"], d["table"], d["lens"], **kwargs(bf)).cpu().numpy()
    np.testing.assert_array_equal(got4, got16)
    assert mm.get_device_error() == 0


def test_nvfp4_dequantised_pages_bit_exact(mm):
    """Every (code, scale byte) pair except the two NaN scales, read back from
    the workspace's bf16 copy and compared with the oracle's value."""
    import torch
    wl = W.random_case(8, num_reqs=1, query_len=256, heads=1, topk=32, init_blocks=1,
                       local_blocks=1, min_len=256, max_len=256, kv_format="nvfp4")
    pages = wl.block_table[0, :2]
    scale_bytes = np.array([b if b not in (0x7F, 0xFF) else 0 for b in range(256)], dtype=np.uint8)
    for k, pg in enumerate(pages):
        # 128 tokens x 8 groups = 1024 groups per page: each scale byte 4 times
        wl.scales[pg] = np.tile(scale_bytes, 4).reshape(128, 8)
        nib = np.tile(np.arange(16, dtype=np.uint8), 128 * 8).reshape(128, 128)
        nib = np.roll(nib, k, axis=1)
        wl.codes[pg] = nib[:, 0::2] | (nib[:, 1::2] << 4)
    n = mm.workspace_bytes(mm.OP_PREFILL_NVFP4, 1, 1, 256, 256, 32)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    run_prefill_nvfp4(mm, wl, workspace=ws)
    assert mm.get_device_error() == 0
    # The workspace ends with the bf16 copy [1 * 2 pages, 128, 128] and its
    # int32 table [1, 2] (rounded up to 256 bytes).
    width = 2
    copy = n - (width * 128 * 128 * 2 + 256)
    got = ws[copy:copy + width * 128 * 128 * 2].cpu().numpy().view(np.uint16)
    got = got.reshape(width, 128, 128)
    want = oracle.nvfp4_dequant_bf16(wl.codes[pages], wl.scales[pages])
    np.testing.assert_array_equal(got, want)
    table = ws[copy + width * 32768:copy + width * 32768 + 8].cpu().numpy().view(np.int32)
    assert table.tolist() == [0, 1]


def test_nvfp4_prefill_full_size_sampled(mm):
    wl = W.make("nvfp4_prefill")
    got = run_prefill_nvfp4(mm, wl)
    assert mm.get_device_error() == 0
    rows = sorted(set([0, 1, 127, 128, 255, 256, 4095, 16384, wl.query_len - 129,
                       wl.query_len - 1] + list(range(5, wl.query_len, 2999))))
    for r in rows:
        s, want = oracle.row(wl, r, 0)
        check_ids_row(got[0, r], want, s, len(s) - 1, wl.topk, wl.init_blocks, wl.local_blocks,
                      where=f"nvfp4 prefill row {r}")


def test_nvfp4_prefill_flags_bad_pages(mm):
    wl = W.random_case(9, num_reqs=2, query_len=200, heads=1, topk=4, init_blocks=1,
                       local_blocks=1, min_len=400, max_len=900, kv_format="nvfp4")
    wl.block_table[1, 0] = wl.num_pages + 3
    run_prefill_nvfp4(mm, wl)
    assert mm.get_device_error() & mm.DEV_BAD_PAGE

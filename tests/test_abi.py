"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/mm3idx.h declares, and rejects bad arguments with
the documented status codes before touching the device."""

import ctypes
import os
import re

import numpy as np
import pytest

import sparse_attention_block_paged_gb300 as mm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mm3idx.h")


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mm3idx_\w+)\s*\(", src, re.M)))


def header_constants():
    src = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(MM3IDX_\w+)\s+\(?(-?\d+)\)?", src)}


def test_every_declared_symbol_is_exported():
    names = declared()
    assert len(names) >= 9
    lib = ctypes.CDLL(mm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(mm.SYMBOLS) == set(names)


def test_constants_match_binding():
    c = header_constants()
    assert c["MM3IDX_OK"] == mm.OK
    assert c["MM3IDX_OP_DECODE"] == mm.OP_DECODE and c["MM3IDX_OP_PREFILL"] == mm.OP_PREFILL
    assert c["MM3IDX_OP_PREFILL_NVFP4"] == mm.OP_PREFILL_NVFP4
    assert c["MM3IDX_MAX_TOPK"] == mm.MAX_TOPK
    assert c["MM3IDX_MAX_DECODE_ROWS"] == mm.MAX_DECODE_ROWS
    assert (c["MM3IDX_DEV_BAD_PAGE"], c["MM3IDX_DEV_SEQ_TOO_LONG"], c["MM3IDX_DEV_SEQ_TOO_SHORT"],
            c["MM3IDX_DEV_TIMEOUT"], c["MM3IDX_DEV_BAD_ROWS"]) == (
                mm.DEV_BAD_PAGE, mm.DEV_SEQ_TOO_LONG, mm.DEV_SEQ_TOO_SHORT, mm.DEV_TIMEOUT,
                mm.DEV_BAD_ROWS)
    assert mm.Problem.sm_scale.offset > mm.Problem.max_seq_len.offset
    for k, v in c.items():
        if k.startswith("MM3IDX_ERR_"):
            assert mm.status_string(v) not in ("", "unknown status")


# Fake, 256-byte aligned addresses: validation must reject the arguments
# before any pointer is dereferenced or any CUDA call is made.
FAKE = 0x7f0000000000


def problem(**kw):
    p = mm.Problem()
    vals = dict(idx_q=FAKE, q_token_stride=128, q_head_stride=128, heads=1, index_cache=FAKE,
                index_scales=None, num_pages=16, block_table=FAKE, table_stride=8, table_width=8,
                seq_lens=FAKE, num_reqs=2, query_len=1, max_seq_len=1000, sm_scale=0.088)
    vals.update(kw)
    for k, v in vals.items():
        setattr(p, k, v)
    return p


def decode_status(p, topk=4, init=1, local=1, out=FAKE, ohs=1024, ors=4, ws=FAKE, wsb=1 << 20):
    return mm.lib.mm3idx_decode(ctypes.byref(p), topk, init, local, out, ohs, ors, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(query_len=0), -6),
    (dict(max_seq_len=0, query_len=1), -6),
    (dict(heads=0), -1),
    (dict(sm_scale=0.0), -1),
    (dict(sm_scale=-1.0), -1),
    (dict(sm_scale=float("inf")), -1),
    (dict(max_seq_len=0xFFFF * 128), -5),
    (dict(idx_q=FAKE + 8), -2),
    (dict(q_token_stride=100), -2),
    (dict(index_cache=FAKE + 4), -3),
    (dict(num_pages=0), -3),
    (dict(index_scales=FAKE), -3),
    (dict(table_width=7), -4),
    (dict(table_stride=6, table_width=8), -4),
])
def test_decode_rejects_bad_problems(kw, code):
    assert decode_status(problem(**kw)) == code


@pytest.mark.parametrize("topk,init,local,code", [
    (0, 0, 0, -7), (33, 1, 1, -7), (4, 3, 2, -7), (4, -1, 1, -7), (4, 1, -1, -7)])
def test_decode_rejects_bad_topk(topk, init, local, code):
    assert decode_status(problem(), topk=topk, init=init, local=local) == code


def test_decode_rejects_wide_rows_and_bad_outputs():
    assert decode_status(problem(heads=8, query_len=5, q_token_stride=1024)) == -10
    assert decode_status(problem(), ors=3) == -8
    assert decode_status(problem(), out=None) == -8
    assert decode_status(problem(heads=2, q_token_stride=256), ohs=4, ors=4) == -8


def test_nvfp4_requires_scales():
    p = problem()
    assert mm.lib.mm3idx_decode_nvfp4(ctypes.byref(p), 4, 1, 1, FAKE, 1024, 4, FAKE, 1 << 20,
                                      None) == -3


def test_empty_batch_is_ok_without_device():
    assert decode_status(problem(num_reqs=0)) == 0
    p = problem(num_reqs=0)
    assert mm.lib.mm3idx_score(ctypes.byref(p), FAKE, 1000, 8, None) == 0
    assert mm.lib.mm3idx_prefill(ctypes.byref(p), 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 20, None) == 0


def test_topk_validation():
    f = mm.lib.mm3idx_topk
    assert f(FAKE, 1000, 8, 1, FAKE, 2, 1, 0, 4, 1, 1, FAKE, 100, 4, None) == -6
    assert f(FAKE, 1000, 8, 1, FAKE, 2, 1, 1000, 4, 3, 2, FAKE, 100, 4, None) == -7
    assert f(FAKE, 1000, 7, 1, FAKE, 2, 1, 1000, 4, 1, 1, FAKE, 100, 4, None) == -8
    assert f(FAKE, 1000, 8, 1, FAKE, 0, 1, 1000, 4, 1, 1, FAKE, 100, 4, None) == 0


def sparse_status(p=None, topk=4, **kw):
    t = mm.SparseTable()
    vals = dict(attention_block_table=FAKE, attention_table_stride=8, attention_table_width=8,
                pages_per_block=2, block_page_stride=4, sparse_block_table_out=FAKE,
                sparse_table_stride=topk * 2, sparse_context_lens_out=FAKE)
    vals.update(kw)
    for k, v in vals.items():
        setattr(t, k, v)
    p = p or problem()
    return mm.lib.mm3idx_decode_sparse_table(ctypes.byref(p), topk, 1, 1, FAKE, 1024, 4,
                                             ctypes.byref(t), FAKE, 1 << 20, None)


@pytest.mark.parametrize("kw,code", [
    (dict(attention_block_table=None), -1),
    (dict(sparse_block_table_out=None), -1),
    (dict(sparse_context_lens_out=None), -1),
    (dict(pages_per_block=0), -1),
    (dict(pages_per_block=3, block_page_stride=3), -1),        # does not divide 128
    (dict(pages_per_block=2, block_page_stride=6), -1),        # neither P nor 2P
    (dict(pages_per_block=256, block_page_stride=256), -1),
    (dict(attention_table_width=7), -4),                       # < cdiv(1000, 128)
    (dict(attention_table_stride=4), -4),
    (dict(sparse_table_stride=7), -8),                         # < topk * P
])
def test_sparse_table_validation(kw, code):
    assert sparse_status(**kw) == code


def test_sparse_table_needs_one_head_and_a_table():
    assert sparse_status(problem(heads=2, q_token_stride=256)) == -10
    p = problem()
    assert mm.lib.mm3idx_decode_sparse_table(ctypes.byref(p), 4, 1, 1, FAKE, 1024, 4, None, FAKE,
                                             1 << 20, None) == -1


def test_nvfp4_prefill_validation_and_workspace():
    p = problem()                                   # no scales: not an NVFP4 problem
    f = mm.lib.mm3idx_prefill_nvfp4
    assert f(ctypes.byref(p), 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == -3
    p = problem(index_scales=FAKE, num_reqs=0)
    assert f(ctypes.byref(p), 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == 0
    p = problem(index_scales=FAKE)
    assert f(ctypes.byref(p), 32, 1, 1, FAKE, 1000, 32, FAKE, 1000, None) == -9


@pytest.mark.gpu
def test_prefill_workspace_sizes(cuda_device):
    """Tile records and two candidate lists (16 or 32 keys) per row of each
    tile a CTA touches; NVFP4 adds the bf16 copy of the pages and its table."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = ctypes.c_size_t(0)
    up = lambda x: -(-x // 256) * 256                # noqa: E731
    tiles = 2 * (-(-3 * 300 // 128) + 3)             # heads x (cdiv(rows, 128) + requests)
    for topk, tk in ((16, 16), (17, 32), (32, 32)):
        part_a = up((tiles + 1) * 64) + 2 * (sms + tiles) * 128 * tk * 8
        assert mm.lib.mm3idx_workspace_bytes(mm.OP_PREFILL, 2, 3, 300, 1000, topk,
                                             ctypes.byref(n)) == 0
        assert n.value == part_a
        assert mm.lib.mm3idx_workspace_bytes(mm.OP_PREFILL_NVFP4, 2, 3, 300, 1000, topk,
                                             ctypes.byref(n)) == 0
        slots = 3 * 8                                # requests x cdiv(1000, 128)
        assert n.value == up(part_a) + slots * 128 * 128 * 2 + up(slots * 4)


def test_ragged_validation():
    f = mm.lib.mm3idx_prefill_ragged
    p = problem(query_len=4)                        # 2 requests of at most 4 rows
    assert f(ctypes.byref(p), FAKE, 9, 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), None, 8, 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), FAKE + 2, 8, 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), FAKE, -1, 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), FAKE, 0, 4, 1, 1, FAKE, 1000, 4, FAKE, 1 << 30, None) == 0
    assert f(ctypes.byref(p), FAKE, 8, 32, 1, 1, FAKE, 1000, 32, FAKE, 100, None) == -9
    g = mm.lib.mm3idx_score_ragged
    assert g(ctypes.byref(p), FAKE, 9, FAKE, 1000, 8, None) == -1
    assert g(ctypes.byref(p), FAKE, 0, FAKE, 1000, 8, None) == 0
    assert g(ctypes.byref(p), FAKE, 8, FAKE, 1000, 7, None) == -8
    t = mm.lib.mm3idx_topk_ragged
    assert t(FAKE, 1000, 8, 1, FAKE, FAKE, 2, 9, 4, 1000, 4, 1, 1, FAKE, 100, 4, None) == -1
    assert t(FAKE, 1000, 8, 1, FAKE, FAKE, 2, 0, 4, 1000, 4, 1, 1, FAKE, 100, 4, None) == 0
    assert t(FAKE, 1000, 8, 1, FAKE, FAKE, 2, 8, 4, 1000, 40, 1, 1, FAKE, 100, 4, None) == -7


def test_wait_timeout_check_validates_warps_before_any_launch():
    assert mm.lib.mm3idx_check_wait_timeout(0, None) == -1
    assert mm.lib.mm3idx_check_wait_timeout(33, None) == -1


def test_workspace_query_validation():
    n = ctypes.c_size_t(0)
    assert mm.lib.mm3idx_workspace_bytes(9, 1, 1, 1, 128, 4, ctypes.byref(n)) == -1
    assert mm.lib.mm3idx_workspace_bytes(mm.OP_DECODE, 1, 1, 1, 128, 40, ctypes.byref(n)) == -7
    # topk is checked before the device is queried
    assert mm.lib.mm3idx_workspace_bytes(mm.OP_PREFILL, 2, 3, 300, 1000, 33, ctypes.byref(n)) == -7


def test_binding_layout_errors():
    import torch
    q = torch.zeros((2, 1, 64), dtype=torch.bfloat16)
    cache = torch.zeros((4, 128, 128), dtype=torch.bfloat16)
    t = torch.zeros((2, 8), dtype=torch.int32)
    lens = torch.zeros((2,), dtype=torch.int32)
    with pytest.raises(ValueError, match="BF16"):
        mm.decode(q, cache, t, lens, query_len=1, max_seq_len=512, topk=4, init_blocks=1,
                  local_blocks=1, sm_scale=0.1)
    q = torch.zeros((2, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="same GPU"):
        mm.decode(q, cache, t, lens, query_len=1, max_seq_len=512, topk=4, init_blocks=1,
                  local_blocks=1, sm_scale=0.1)
    with pytest.raises(ValueError, match="int32"):
        mm.decode(q, cache, t.long(), lens, query_len=1, max_seq_len=512, topk=4, init_blocks=1,
                  local_blocks=1, sm_scale=0.1)


def test_binding_rejects_host_tensors_and_bad_shapes():
    """Argument checks that run before any CUDA call: host tensors never reach
    the library, whose pointers are device pointers."""
    import torch
    score = torch.zeros((1, 8, 8), dtype=torch.float32)
    lens = torch.full((2,), 500, dtype=torch.int32)
    cu = torch.tensor([0, 4, 8], dtype=torch.int32)
    with pytest.raises(ValueError, match="same GPU"):
        mm.topk(score, lens, query_len=4, max_seq_len=1000, topk=4, init_blocks=1,
                local_blocks=1)
    with pytest.raises(ValueError, match="same GPU"):
        mm.topk_ragged(score, lens, cu, max_query_len=4, max_seq_len=1000, topk=4,
                       init_blocks=1, local_blocks=1)
    with pytest.raises(ValueError, match="cu_seqlens_q"):
        mm.topk_ragged(score, lens, cu.long(), max_query_len=4, max_seq_len=1000, topk=4,
                       init_blocks=1, local_blocks=1)
    q = torch.zeros((8, 1, 128), dtype=torch.bfloat16)
    cache = torch.zeros((4, 128, 128), dtype=torch.bfloat16)
    table = torch.zeros((2, 8), dtype=torch.int32)
    with pytest.raises(ValueError, match="more query rows"):
        mm.prefill_ragged(q, cache, table, lens, cu, max_query_len=3, max_seq_len=1000, topk=4,
                          init_blocks=1, local_blocks=1, sm_scale=0.1)
    with pytest.raises(ValueError, match="same GPU"):
        mm.prefill_ragged(q, cache, table, lens, cu, max_query_len=4, max_seq_len=1000, topk=4,
                          init_blocks=1, local_blocks=1, sm_scale=0.1)
    with pytest.raises(ValueError, match="same GPU"):
        mm.decode_sparse_table(q[:2], cache, table, lens, query_len=1, max_seq_len=1000, topk=4,
                               init_blocks=1, local_blocks=1, sm_scale=0.1,
                               attention_block_table=table,
                               sparse_block_table_out=torch.zeros((2, 8), dtype=torch.int32),
                               sparse_context_lens_out=torch.zeros((2,), dtype=torch.int32),
                               block_page_stride=2, pages_per_block=2)


def test_workload_generator_layout():
    import workloads as W
    wl = W.make("tiny")
    assert wl.num_pages == 16 and wl.width == 6
    used = {int(p) for i, s in enumerate(wl.seq_lens) for p in wl.block_table[i, :-(-int(s) // 128)]}
    assert len(used) == 3 + 6 and max(used) < 16
    assert wl.block_table[0, 3] == wl.num_pages + 7
    # tail slots of request 0's last page are poisoned
    last = wl.block_table[0, 2]
    assert np.all(wl.cache[last, 300 % 128:] == W.POISON_BF16)
    again = W.make("tiny")
    assert np.array_equal(again.cache, wl.cache) and np.array_equal(again.q, wl.q)


def test_score_nvfp4_validation_and_workspace():
    f = mm.lib.mm3idx_score_nvfp4
    p = problem()                                   # no scales: not an NVFP4 problem
    assert f(ctypes.byref(p), FAKE, 1000, 8, None, 0, None) == -3
    p = problem(index_scales=FAKE, num_reqs=0)
    assert f(ctypes.byref(p), FAKE, 1000, 8, None, 0, None) == 0
    # 300 rows per request: the bf16 copy needs a workspace, checked before any launch
    p = problem(index_scales=FAKE, query_len=300)
    assert f(ctypes.byref(p), FAKE, 1 << 20, 8, None, 0, None) == -9
    assert f(ctypes.byref(p), FAKE, 1 << 20, 8, FAKE, 1000, None) == -9
    assert f(ctypes.byref(p), FAKE, 1 << 20, 8, FAKE + 16, 1 << 30, None) == -9
    assert f(ctypes.byref(p), FAKE, 1 << 20, 7, FAKE, 1 << 30, None) == -8
    n = ctypes.c_size_t(7)
    assert mm.lib.mm3idx_workspace_bytes(mm.OP_SCORE_NVFP4, 4, 3, 8, 1000, 1,
                                         ctypes.byref(n)) == 0
    assert n.value == 0                              # 4 heads x 8 rows: on chip
    assert mm.lib.mm3idx_workspace_bytes(mm.OP_SCORE_NVFP4, 1, 3, 300, 1000, 1,
                                         ctypes.byref(n)) == 0
    slots = 3 * 8                                    # requests x cdiv(1000, 128)
    assert n.value == slots * 128 * 128 * 2 + 256
    c = header_constants()
    assert c["MM3IDX_OP_SCORE_NVFP4"] == mm.OP_SCORE_NVFP4


def test_binding_stream_workspace_and_out_must_be_on_the_inputs_gpu():
    """Checks the binding makes before a library call: an explicit stream,
    a caller's workspace and a caller's score output must all belong to the
    inputs' GPU (the library takes their addresses as that GPU's)."""
    import torch

    class FakeStream:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    dev0 = torch.device("cuda", 0)
    with pytest.raises(ValueError, match="stream"):
        mm._stream(dev0, FakeStream())
    with pytest.raises(ValueError, match="workspace"):
        mm._ws(torch.zeros(256, dtype=torch.uint8), dev0)
    with pytest.raises(ValueError, match="workspace"):
        mm._ws(None, dev0)
    with pytest.raises(ValueError, match="out must be on"):
        mm._score_out_ok(torch.zeros((1, 4, 8)), 1, 4, 8, dev0)


def test_every_library_call_runs_with_the_inputs_gpu_current():
    """The library reads the current device (SM count, status word, static
    scratch): every call that launches work or reads the status word sits
    inside a `with _on(device)` block, and gets its stream from _stream."""
    import ast
    src = open(os.path.join(ROOT, "sparse_attention_block_paged_gb300", "__init__.py")).read()
    tree = ast.parse(src)
    exempt = {"mm3idx_version", "mm3idx_status_string", "mm3idx_workspace_bytes",
              "mm3idx_forward_workspace_bytes"}
    found = 0

    def visit(node, guarded):
        nonlocal found
        if isinstance(node, ast.With):
            guarded = guarded or any(
                isinstance(i.context_expr, ast.Call) and getattr(i.context_expr.func, "id", "") == "_on"
                for i in node.items)
        lib_call = (isinstance(node, ast.Call) and isinstance(node.func, ast.Attribute)
                    and node.func.attr.startswith("mm3idx_") and node.func.attr not in exempt
                    and getattr(node.func.value, "id", "") == "lib")
        # _fused calls the entry point it is given as `fn`
        fused_call = isinstance(node, ast.Call) and getattr(node.func, "id", "") == "fn"
        if lib_call or fused_call:
            found += 1
            assert guarded, f"line {node.lineno}: library call outside `with _on(...)`"
            assert any(isinstance(a, ast.Call) and getattr(a.func, "id", "") == "_stream"
                       for a in node.args), f"line {node.lineno}: stream not from _stream"
        for child in ast.iter_child_nodes(node):
            visit(child, guarded)

    visit(tree, False)
    assert found >= 11


def test_forward_validation():
    """mm3idx_forward rejects bad splits and layouts before any device work."""
    f = mm.lib.mm3idx_forward
    p = problem(query_len=4, num_reqs=3)             # 3 requests of at most 4 decode rows
    # num_decodes outside 0..num_reqs
    assert f(ctypes.byref(p), 4, FAKE, 8, 300, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), -1, FAKE, 8, 300, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -1
    # prefill rows beyond num_prefills * max_query_len, missing or misaligned offsets
    assert f(ctypes.byref(p), 1, FAKE, 601, 300, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), 1, None, 8, 300, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -1
    assert f(ctypes.byref(p), 1, FAKE + 2, 8, 300, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30,
             None) == -1
    # prefill query rows longer than max_seq_len
    assert f(ctypes.byref(p), 1, FAKE, 8, 2000, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -6
    # decode rows per request over 32
    q = problem(query_len=16, heads=4, num_reqs=3)
    assert f(ctypes.byref(q), 1, FAKE, 8, 300, 16, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -10
    # topk and output layout
    assert f(ctypes.byref(p), 1, FAKE, 8, 300, 40, 1, 2, FAKE, 1 << 20, 16, FAKE, 1 << 30, None) == -7
    assert f(ctypes.byref(p), 1, FAKE, 8, 300, 16, 1, 2, FAKE, 1 << 20, 8, FAKE, 1 << 30, None) == -8
    # an empty batch is a no-op
    e = problem(num_reqs=0)
    assert f(ctypes.byref(e), 0, None, 0, 1, 16, 1, 2, None, 0, 16, None, 0, None) == 0
    n = ctypes.c_size_t(0)
    assert mm.lib.mm3idx_forward_workspace_bytes(1, 2, 4, 1, 300, 1000, 40, 0, ctypes.byref(n)) == -7
    assert mm.lib.mm3idx_forward_workspace_bytes(0, 2, 4, 1, 300, 1000, 16, 0, ctypes.byref(n)) == -1

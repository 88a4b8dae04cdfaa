"""GB300 (sm_103a) MiniMax-M3 lightning-indexer: causal block scoring of bf16
index queries against a paged index-K cache, and top-k block selection with
forced init/local blocks.

This module is the thin Python binding of ``libmm3idx.so`` (C ABI in
``include/mm3idx.h``).  It only marshals torch tensors into pointers, strides
and the current CUDA stream; every step of the computation runs in the
library's CUDA kernels.  Importing it fails loudly when the library has not
been built: there is no CPU or PyTorch fallback.

Entry points (names after the vLLM MiniMax-M3 ``index_topk`` page):

* :func:`score`        -- fp32 block scores [heads, rows, cdiv(max_seq_len,128)]
* :func:`score_nvfp4`  -- the same over NVFP4 index-K pages
* :func:`topk`         -- ids from a score tensor
* :func:`decode`       -- fused score + top-k for short query runs
* :func:`decode_nvfp4` -- the same over NVFP4 index-K pages
* :func:`prefill`      -- tensor-core scores + selector for long query runs
* :func:`forward`      -- a batch of decode requests followed by prefill requests
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libmm3idx.so")

OK = 0
OP_DECODE = 1
OP_PREFILL = 2
OP_PREFILL_NVFP4 = 3
OP_SCORE_NVFP4 = 4
MAX_TOPK = 32
MAX_DECODE_ROWS = 32
STATIC_SCRATCH_BYTES = 8 << 20
DEV_BAD_PAGE, DEV_SEQ_TOO_LONG, DEV_SEQ_TOO_SHORT, DEV_TIMEOUT, DEV_BAD_ROWS = 1, 2, 4, 8, 16


class Mm3idxError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class Problem(ctypes.Structure):
    """Mirror of ``mm3idx_problem_t``."""
    _fields_ = [
        ("idx_q", ctypes.c_void_p),
        ("q_token_stride", ctypes.c_int64),
        ("q_head_stride", ctypes.c_int64),
        ("heads", ctypes.c_int32),
        ("index_cache", ctypes.c_void_p),
        ("index_scales", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32),
        ("block_table", ctypes.c_void_p),
        ("table_stride", ctypes.c_int64),
        ("table_width", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p),
        ("num_reqs", ctypes.c_int32),
        ("query_len", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
    ]


class SparseTable(ctypes.Structure):
    """mm3idx_sparse_table_t."""
    _fields_ = [
        ("attention_block_table", ctypes.c_void_p),
        ("attention_table_stride", ctypes.c_int64),
        ("attention_table_width", ctypes.c_int32),
        ("pages_per_block", ctypes.c_int32),
        ("block_page_stride", ctypes.c_int32),
        ("sparse_block_table_out", ctypes.c_void_p),
        ("sparse_table_stride", ctypes.c_int64),
        ("sparse_context_lens_out", ctypes.c_void_p),
    ]


SYMBOLS = {
    "mm3idx_version": (ctypes.c_int32, []),
    "mm3idx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mm3idx_workspace_bytes": (ctypes.c_int, [ctypes.c_int32] * 6 + [ctypes.POINTER(ctypes.c_size_t)]),
    "mm3idx_score": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_int64, ctypes.c_void_p]),
    "mm3idx_score_nvfp4": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                          ctypes.c_void_p]),
    "mm3idx_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "mm3idx_decode": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "mm3idx_decode_nvfp4": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p]),
    "mm3idx_prefill": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "mm3idx_prefill_nvfp4": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                            ctypes.c_void_p]),
    "mm3idx_score_ragged": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p]),
    "mm3idx_topk_ragged": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_void_p]),
    "mm3idx_prefill_ragged": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_void_p,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p]),
    "mm3idx_get_device_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "mm3idx_decode_sparse_table": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32,
                                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                                  ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.POINTER(SparseTable), ctypes.c_void_p,
                                                  ctypes.c_size_t, ctypes.c_void_p]),
    "mm3idx_check_wait_timeout": (ctypes.c_int, [ctypes.c_int32, ctypes.c_void_p]),
    "mm3idx_forward": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_size_t, ctypes.c_void_p]),
    "mm3idx_forward_workspace_bytes": (ctypes.c_int, [ctypes.c_int32] * 8 +
                                       [ctypes.POINTER(ctypes.c_size_t)]),
    "mm3idx_decode_static": (ctypes.c_int, [ctypes.POINTER(Problem), ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
}


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it first "
            "(python sparse_attention_block_paged_gb300/build.py); there is no fallback")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in SYMBOLS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
LIB_PATH = _LIB_PATH


def status_string(status: int) -> str:
    return lib.mm3idx_status_string(status).decode()


def _check(status: int, what: str):
    if status != OK:
        raise Mm3idxError(status, what)


def _stream(device, stream=None):
    """The stream a call launches on: `stream`, which must belong to the
    inputs' GPU, else that GPU's current stream."""
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    _need(torch.device(stream.device) == torch.device(device),
          "stream must belong to the inputs' GPU")
    return ctypes.c_void_p(stream.cuda_stream)


def _on(device):
    """Make the inputs' GPU current for a library call: the library takes the
    SM count, its status word and its static scratch from the current device."""
    return torch.cuda.device(device)


def _ws(workspace, device):
    """(pointer, bytes) of a caller-provided workspace on the inputs' GPU."""
    _need(isinstance(workspace, torch.Tensor) and workspace.device == torch.device(device)
          and workspace.is_contiguous(),
          "workspace must be a contiguous tensor on the inputs' GPU")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def _cdiv(a, b):
    return (a + b - 1) // b


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _problem(idx_q, index_cache, block_table, seq_lens, query_len, max_seq_len, sm_scale,
             index_scales=None, nvfp4=False, rows=None):
    """Layout checks of check_context_score_inputs, then the C struct."""
    _need(idx_q.ndim == 3 and idx_q.shape[2] == 128 and idx_q.dtype == torch.bfloat16
          and idx_q.stride(2) == 1, "index queries must be BF16 [tokens,heads,128] with contiguous D")
    if nvfp4:
        _need(index_cache.dtype == torch.uint8 and index_cache.ndim == 3
              and tuple(index_cache.shape[1:]) == (128, 64) and index_cache.is_contiguous(),
              "NVFP4 codes must be contiguous uint8 [pages,128,64]")
        _need(index_scales is not None and index_scales.dtype == torch.uint8
              and tuple(index_scales.shape) == (index_cache.shape[0], 128, 8)
              and index_scales.is_contiguous(), "NVFP4 scales must be contiguous uint8 [pages,128,8]")
    else:
        _need(index_cache.ndim == 3 and tuple(index_cache.shape[1:]) == (128, 128)
              and index_cache.is_contiguous() and index_cache.shape[0] >= 1,
              "index cache must be contiguous non-empty [pages,128,128]")
        _need(index_cache.dtype == torch.bfloat16, "index cache must be bf16")
    _need(block_table.ndim == 2 and block_table.stride(1) == 1 and block_table.dtype == torch.int32
          and seq_lens.ndim == 1 and seq_lens.dtype == torch.int32 and seq_lens.is_contiguous(),
          "block table and lengths must be int32 with unit stride")
    dev = idx_q.device
    _need(dev.type == "cuda" and all(t.device == dev for t in (index_cache, block_table, seq_lens))
          and (index_scales is None or index_scales.device == dev),
          "all score inputs must be on the same GPU")
    num_reqs = seq_lens.shape[0]
    _need(idx_q.shape[0] == (num_reqs * query_len if rows is None else rows),
          "rows != batch * query_len")
    _need(block_table.shape[0] == num_reqs, "block table must have one row per request")
    p = Problem()
    p.idx_q = idx_q.data_ptr()
    p.q_token_stride = idx_q.stride(0)
    p.q_head_stride = idx_q.stride(1)
    p.heads = idx_q.shape[1]
    p.index_cache = index_cache.data_ptr()
    p.index_scales = index_scales.data_ptr() if index_scales is not None else None
    p.num_pages = index_cache.shape[0]
    p.block_table = block_table.data_ptr()
    p.table_stride = block_table.stride(0) if num_reqs > 1 else max(block_table.shape[1], 1)
    p.table_width = block_table.shape[1]
    p.seq_lens = seq_lens.data_ptr()
    p.num_reqs = num_reqs
    p.query_len = query_len
    p.max_seq_len = max_seq_len
    p.sm_scale = sm_scale
    return p


def workspace_bytes(op: int, heads: int, num_reqs: int, query_len: int, max_seq_len: int,
                    topk: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.mm3idx_workspace_bytes(op, heads, num_reqs, query_len, max_seq_len, topk,
                                      ctypes.byref(n)), "mm3idx_workspace_bytes")
    return n.value


def new_workspace(op, heads, num_reqs, query_len, max_seq_len, topk, device=None):
    """A workspace for :func:`decode` / :func:`prefill` (uint8, 256-byte
    aligned by the caching allocator, zero-filled as the decode requires;
    reusable across calls)."""
    n = workspace_bytes(op, heads, num_reqs, query_len, max_seq_len, topk)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def score(idx_q, index_cache, block_table, seq_lens, *, query_len, max_seq_len, sm_scale,
          out=None, stream=None):
    """fp32 [heads, rows, cdiv(max_seq_len,128)] block scores (-inf past each
    row's own block); written into ``out[:, :rows, :width]`` when given."""
    p = _problem(idx_q, index_cache, block_table, seq_lens, query_len, max_seq_len, sm_scale)
    rows, heads = idx_q.shape[0], idx_q.shape[1]
    width = _cdiv(max_seq_len, 128)
    if out is None:
        out = torch.empty((heads, rows, width), dtype=torch.float32, device=idx_q.device)
    _score_out_ok(out, heads, rows, width, idx_q.device)
    with _on(idx_q.device):
        _check(lib.mm3idx_score(ctypes.byref(p), out.data_ptr(), out.stride(0), out.stride(1),
                                _stream(idx_q.device, stream)), "mm3idx_score")
    return out[:, :rows, :width]


def _score_out_ok(out, heads, rows, width, device):
    _need(out.dtype == torch.float32 and out.ndim == 3 and out.shape[0] == heads
          and out.shape[1] >= rows and out.shape[2] >= width and out.stride(2) == 1,
          "out must be fp32 [heads, >=rows, >=cdiv(max_seq_len,128)] with unit inner stride")
    _need(out.device == torch.device(device), "out must be on the inputs' GPU")


def score_nvfp4(idx_q, codes, scales, block_table, seq_lens, *, query_len, max_seq_len,
                sm_scale, out=None, workspace=None, stream=None):
    """:func:`score` over NVFP4 pages (codes uint8 [pages,128,64], scales
    uint8 e4m3 [pages,128,8]).  Short query runs (heads * query_len <= 32)
    dequantise on chip in the streaming kernel; longer ones first make a
    bf16 copy of the visible pages in ``workspace`` (from
    ``new_workspace(OP_SCORE_NVFP4, ...)``; allocated when not given)."""
    p = _problem(idx_q, codes, block_table, seq_lens, query_len, max_seq_len, sm_scale,
                 index_scales=scales, nvfp4=True)
    rows, heads = idx_q.shape[0], idx_q.shape[1]
    width = _cdiv(max_seq_len, 128)
    if out is None:
        out = torch.empty((heads, rows, width), dtype=torch.float32, device=idx_q.device)
    _score_out_ok(out, heads, rows, width, idx_q.device)
    with _on(idx_q.device):
        if workspace is None:
            workspace = new_workspace(OP_SCORE_NVFP4, heads, seq_lens.shape[0], query_len,
                                      max_seq_len, 1, idx_q.device)
        wp, wn = _ws(workspace, idx_q.device)
        _check(lib.mm3idx_score_nvfp4(ctypes.byref(p), out.data_ptr(), out.stride(0),
                                      out.stride(1), wp, wn, _stream(idx_q.device, stream)),
               "mm3idx_score_nvfp4")
    return out[:, :rows, :width]


def _ids_out(out, heads, rows, topk, device):
    if out is None:
        out = torch.empty((heads, rows, topk), dtype=torch.int32, device=device)
    _need(out.dtype == torch.int32 and out.ndim == 3 and out.shape[0] == heads
          and out.shape[1] >= rows and out.shape[2] == topk and out.stride(2) == 1,
          "out must be int32 [heads, >=rows, topk] with unit inner stride")
    _need(out.device == torch.device(device), "out must be on the inputs' GPU")
    return out


def _on_gpu(ref, *tensors):
    """Every tensor on ref's device, and that device a GPU (the library takes
    the addresses as device addresses)."""
    _need(ref.device.type == "cuda" and all(t.device == ref.device for t in tensors),
          "all inputs must be on the same GPU")


def topk(score_t, seq_lens, *, query_len, max_seq_len, topk, init_blocks, local_blocks,
         out=None, stream=None):
    """int32 [heads, rows, topk] ids (ascending, -1 pad) from a score tensor."""
    _need(score_t.dtype == torch.float32 and score_t.ndim == 3 and score_t.stride(2) == 1,
          "score must be fp32 [heads, rows, blocks] with unit inner stride")
    _on_gpu(score_t, seq_lens)
    heads, rows = score_t.shape[0], seq_lens.shape[0] * query_len
    _need(score_t.shape[1] >= rows and score_t.shape[2] >= _cdiv(max_seq_len, 128),
          "score narrower than the rows or cdiv(max_seq_len,128)")
    out = _ids_out(out, heads, rows, topk, score_t.device)
    with _on(score_t.device):
        _check(lib.mm3idx_topk(score_t.data_ptr(), score_t.stride(0), score_t.stride(1), heads,
                               seq_lens.data_ptr(), seq_lens.shape[0], query_len, max_seq_len,
                               topk, init_blocks, local_blocks, out.data_ptr(), out.stride(0),
                               out.stride(1), _stream(score_t.device, stream)), "mm3idx_topk")
    return out[:, :rows, :]


def _fused(fn, name, op, idx_q, cache, block_table, seq_lens, scales, nvfp4, query_len,
           max_seq_len, topk, init_blocks, local_blocks, sm_scale, out, workspace, stream):
    p = _problem(idx_q, cache, block_table, seq_lens, query_len, max_seq_len, sm_scale,
                 index_scales=scales, nvfp4=nvfp4)
    rows, heads = idx_q.shape[0], idx_q.shape[1]
    out = _ids_out(out, heads, rows, topk, idx_q.device)
    with _on(idx_q.device):
        if workspace is None:
            workspace = new_workspace(op, heads, seq_lens.shape[0], query_len, max_seq_len, topk,
                                      idx_q.device)
        wp, wn = _ws(workspace, idx_q.device)
        _check(fn(ctypes.byref(p), topk, init_blocks, local_blocks, out.data_ptr(), out.stride(0),
                  out.stride(1), wp, wn, _stream(idx_q.device, stream)), name)
    return out[:, :rows, :]


def decode(idx_q, index_cache, block_table, seq_lens, *, query_len, max_seq_len, topk,
           init_blocks, local_blocks, sm_scale, out=None, workspace=None, stream=None):
    """Fused decode score + top-k (heads * query_len <= 32).  ``workspace``
    (from :func:`new_workspace`) may be reused across calls."""
    return _fused(lib.mm3idx_decode, "mm3idx_decode", OP_DECODE, idx_q, index_cache, block_table,
                  seq_lens, None, False, query_len, max_seq_len, topk, init_blocks, local_blocks,
                  sm_scale, out, workspace, stream)


def decode_nvfp4(idx_q, codes, scales, block_table, seq_lens, *, query_len, max_seq_len, topk,
                 init_blocks, local_blocks, sm_scale, out=None, workspace=None, stream=None):
    """:func:`decode` over NVFP4 pages (codes uint8 [pages,128,64], scales
    uint8 e4m3 [pages,128,8])."""
    return _fused(lib.mm3idx_decode_nvfp4, "mm3idx_decode_nvfp4", OP_DECODE, idx_q, codes,
                  block_table, seq_lens, scales, True, query_len, max_seq_len, topk, init_blocks,
                  local_blocks, sm_scale, out, workspace, stream)


def decode_sparse_table(idx_q, index_cache, block_table, seq_lens, *, query_len, max_seq_len,
                        topk, init_blocks, local_blocks, sm_scale, attention_block_table,
                        sparse_block_table_out, sparse_context_lens_out, block_page_stride,
                        pages_per_block, index_scales=None, out=None, workspace=None,
                        stream=None):
    """:func:`decode` (or :func:`decode_nvfp4` when ``index_scales`` is given)
    for one index head that also writes the sparse page table of its ids:
    ``sparse_block_table_out`` int32 [rows, topk * pages_per_block] (pages of
    block b: attention_block_table[i, b] * block_page_stride + 0.., -1 in
    unused slots) and ``sparse_context_lens_out`` int32 [rows] (visible
    tokens in the selected blocks).  Returns the ids."""
    nvfp4 = index_scales is not None
    p = _problem(idx_q, index_cache, block_table, seq_lens, query_len, max_seq_len, sm_scale,
                 index_scales=index_scales, nvfp4=nvfp4)
    rows, heads = idx_q.shape[0], idx_q.shape[1]
    at, st, ctx = attention_block_table, sparse_block_table_out, sparse_context_lens_out
    _need(all(t.dtype == torch.int32 and t.device == idx_q.device for t in (at, st, ctx)),
          "sparse tables must be int32 on the query device")
    _need(at.ndim == 2 and at.shape[0] == seq_lens.shape[0] and at.stride(1) == 1,
          "attention block table must be [num_reqs, blocks] with contiguous rows")
    _need(st.ndim == 2 and st.shape[0] >= rows and st.shape[1] == topk * pages_per_block
          and st.stride(1) == 1, "sparse block table must be [rows, topk * pages_per_block]")
    _need(ctx.ndim == 1 and ctx.shape[0] >= rows and ctx.stride(0) == 1,
          "sparse context lengths must be [rows]")
    t = SparseTable()
    t.attention_block_table = at.data_ptr()
    t.attention_table_stride = at.stride(0) if at.shape[0] > 1 else max(at.shape[1], 1)
    t.attention_table_width = at.shape[1]
    t.pages_per_block = pages_per_block
    t.block_page_stride = block_page_stride
    t.sparse_block_table_out = st.data_ptr()
    t.sparse_table_stride = st.stride(0) if st.shape[0] > 1 else max(st.shape[1], 1)
    t.sparse_context_lens_out = ctx.data_ptr()
    out = _ids_out(out, heads, rows, topk, idx_q.device)
    with _on(idx_q.device):
        if workspace is None:
            workspace = new_workspace(OP_DECODE, heads, seq_lens.shape[0], query_len,
                                      max_seq_len, topk, idx_q.device)
        wp, wn = _ws(workspace, idx_q.device)
        _check(lib.mm3idx_decode_sparse_table(ctypes.byref(p), topk, init_blocks, local_blocks,
                                              out.data_ptr(), out.stride(0), out.stride(1),
                                              ctypes.byref(t), wp, wn,
                                              _stream(idx_q.device, stream)),
               "mm3idx_decode_sparse_table")
    return out[:, :rows, :]


def prefill(idx_q, index_cache, block_table, seq_lens, *, query_len, max_seq_len, topk,
            init_blocks, local_blocks, sm_scale, out=None, workspace=None, stream=None):
    """Tensor-core prefill scores (to the workspace) followed by the selector."""
    return _fused(lib.mm3idx_prefill, "mm3idx_prefill", OP_PREFILL, idx_q, index_cache,
                  block_table, seq_lens, None, False, query_len, max_seq_len, topk, init_blocks,
                  local_blocks, sm_scale, out, workspace, stream)


def prefill_nvfp4(idx_q, codes, scales, block_table, seq_lens, *, query_len, max_seq_len, topk,
                  init_blocks, local_blocks, sm_scale, out=None, workspace=None, stream=None):
    """:func:`prefill` over NVFP4 pages (codes uint8 [pages,128,64], scales
    uint8 e4m3 [pages,128,8]): the visible pages are dequantised once into
    the workspace, then scored on the tensor cores and selected."""
    return _fused(lib.mm3idx_prefill_nvfp4, "mm3idx_prefill_nvfp4", OP_PREFILL_NVFP4, idx_q, codes,
                  block_table, seq_lens, scales, True, query_len, max_seq_len, topk, init_blocks,
                  local_blocks, sm_scale, out, workspace, stream)


def _ragged_problem(idx_q, cache, block_table, seq_lens, cu_seqlens_q, max_query_len,
                    max_seq_len, sm_scale, scales=None):
    _need(cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.ndim == 1
          and cu_seqlens_q.shape[0] == seq_lens.shape[0] + 1 and cu_seqlens_q.is_contiguous()
          and cu_seqlens_q.device == idx_q.device,
          "cu_seqlens_q must be contiguous int32 [num_reqs + 1] on the query device")
    num_reqs = seq_lens.shape[0]
    total_q = idx_q.shape[0]
    _need(total_q <= num_reqs * max_query_len, "more query rows than num_reqs * max_query_len")
    p = _problem(idx_q, cache, block_table, seq_lens, max_query_len, max_seq_len, sm_scale,
                 index_scales=scales, nvfp4=scales is not None, rows=total_q)
    return p, total_q


def score_ragged(idx_q, index_cache, block_table, seq_lens, cu_seqlens_q, *, max_query_len,
                 max_seq_len, sm_scale, out=None, stream=None):
    """:func:`score` of a ragged batch: request i owns query rows
    cu_seqlens_q[i]..cu_seqlens_q[i+1]-1 (at positions seq_len - rows_i + j)."""
    p, total_q = _ragged_problem(idx_q, index_cache, block_table, seq_lens, cu_seqlens_q,
                                 max_query_len, max_seq_len, sm_scale)
    heads = idx_q.shape[1]
    width = _cdiv(max_seq_len, 128)
    if out is None:
        out = torch.empty((heads, total_q, width), dtype=torch.float32, device=idx_q.device)
    _score_out_ok(out, heads, total_q, width, idx_q.device)
    with _on(idx_q.device):
        _check(lib.mm3idx_score_ragged(ctypes.byref(p), cu_seqlens_q.data_ptr(), total_q,
                                       out.data_ptr(), out.stride(0), out.stride(1),
                                       _stream(idx_q.device, stream)), "mm3idx_score_ragged")
    return out[:, :total_q, :width]


def topk_ragged(score_t, seq_lens, cu_seqlens_q, *, max_query_len, max_seq_len, topk,
                init_blocks, local_blocks, out=None, stream=None):
    """:func:`topk` of a ragged batch's score tensor [heads, total_q, blocks]."""
    _need(score_t.dtype == torch.float32 and score_t.ndim == 3 and score_t.stride(2) == 1,
          "score must be fp32 [heads, rows, blocks] with unit inner stride")
    _need(cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.ndim == 1
          and cu_seqlens_q.shape[0] == seq_lens.shape[0] + 1 and cu_seqlens_q.is_contiguous(),
          "cu_seqlens_q must be contiguous int32 [num_reqs + 1]")
    _on_gpu(score_t, seq_lens, cu_seqlens_q)
    heads, total_q = score_t.shape[0], score_t.shape[1]
    out = _ids_out(out, heads, total_q, topk, score_t.device)
    with _on(score_t.device):
        _check(lib.mm3idx_topk_ragged(score_t.data_ptr(), score_t.stride(0), score_t.stride(1),
                                      heads, cu_seqlens_q.data_ptr(), seq_lens.data_ptr(),
                                      seq_lens.shape[0], total_q, max_query_len, max_seq_len,
                                      topk, init_blocks, local_blocks, out.data_ptr(),
                                      out.stride(0), out.stride(1),
                                      _stream(score_t.device, stream)), "mm3idx_topk_ragged")
    return out[:, :total_q, :]


def prefill_ragged(idx_q, index_cache, block_table, seq_lens, cu_seqlens_q, *, max_query_len,
                   max_seq_len, topk, init_blocks, local_blocks, sm_scale, index_scales=None,
                   out=None, workspace=None, stream=None):
    """:func:`prefill` (or :func:`prefill_nvfp4` with ``index_scales``) of a
    ragged batch.  A workspace from ``new_workspace(OP_PREFILL[_NVFP4], heads,
    num_reqs, max_query_len, max_seq_len, topk)`` serves any batch under
    those bounds."""
    p, total_q = _ragged_problem(idx_q, index_cache, block_table, seq_lens, cu_seqlens_q,
                                 max_query_len, max_seq_len, sm_scale, scales=index_scales)
    heads = idx_q.shape[1]
    op = OP_PREFILL_NVFP4 if index_scales is not None else OP_PREFILL
    out = _ids_out(out, heads, total_q, topk, idx_q.device)
    with _on(idx_q.device):
        if workspace is None:
            workspace = new_workspace(op, heads, seq_lens.shape[0], max_query_len, max_seq_len,
                                      topk, idx_q.device)
        wp, wn = _ws(workspace, idx_q.device)
        _check(lib.mm3idx_prefill_ragged(ctypes.byref(p), cu_seqlens_q.data_ptr(), total_q, topk,
                                         init_blocks, local_blocks, out.data_ptr(), out.stride(0),
                                         out.stride(1), wp, wn, _stream(idx_q.device, stream)),
               "mm3idx_prefill_ragged")
    return out[:, :total_q, :]


def forward_workspace_bytes(heads: int, num_decodes: int, decode_query_len: int,
                            num_prefills: int, prefill_max_query_len: int, max_seq_len: int,
                            topk: int, nvfp4: bool = False) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.mm3idx_forward_workspace_bytes(heads, num_decodes, decode_query_len, num_prefills,
                                              prefill_max_query_len, max_seq_len, topk,
                                              1 if nvfp4 else 0, ctypes.byref(n)),
           "mm3idx_forward_workspace_bytes")
    return n.value


def forward(idx_q, index_cache, block_table, seq_lens, prefill_cu_seqlens_q, *, num_decodes,
            decode_query_len, prefill_max_query_len, max_seq_len, topk, init_blocks, local_blocks,
            sm_scale, index_scales=None, out=None, workspace=None, stream=None):
    """A batch of ``num_decodes`` decode requests (``decode_query_len`` rows
    each) followed by prefill requests whose rows are given by
    ``prefill_cu_seqlens_q`` (int32 [num_prefills + 1], from 0, counted from
    the first prefill row), scored and selected in one call: int32
    [heads, rows, topk] ids for every row of the batch.  NVFP4 pages when
    ``index_scales`` is given.  ``workspace`` (zero-filled, reusable) from
    :func:`forward_workspace_bytes`; allocated when not given."""
    num_reqs = seq_lens.shape[0]
    num_prefills = num_reqs - num_decodes
    _need(0 <= num_decodes <= num_reqs, "num_decodes must be within the batch")
    _need(prefill_cu_seqlens_q.dtype == torch.int32 and prefill_cu_seqlens_q.ndim == 1
          and prefill_cu_seqlens_q.shape[0] == num_prefills + 1
          and prefill_cu_seqlens_q.is_contiguous() and prefill_cu_seqlens_q.device == idx_q.device,
          "prefill_cu_seqlens_q must be contiguous int32 [num_prefills + 1] on the query device")
    dec_rows = num_decodes * decode_query_len
    total_q = idx_q.shape[0] - dec_rows
    _need(total_q >= 0 and total_q <= num_prefills * prefill_max_query_len,
          "rows after the decode rows exceed num_prefills * prefill_max_query_len")
    nvfp4 = index_scales is not None
    p = _problem(idx_q, index_cache, block_table, seq_lens, decode_query_len, max_seq_len, sm_scale,
                 index_scales=index_scales, nvfp4=nvfp4, rows=idx_q.shape[0])
    rows, heads = idx_q.shape[0], idx_q.shape[1]
    out = _ids_out(out, heads, rows, topk, idx_q.device)
    with _on(idx_q.device):
        if workspace is None:
            n = forward_workspace_bytes(heads, num_decodes, decode_query_len, num_prefills,
                                        prefill_max_query_len, max_seq_len, topk, nvfp4)
            workspace = torch.zeros(max(n, 256), dtype=torch.uint8, device=idx_q.device)
        wp, wn = _ws(workspace, idx_q.device)
        _check(lib.mm3idx_forward(ctypes.byref(p), num_decodes, prefill_cu_seqlens_q.data_ptr(),
                                  total_q, prefill_max_query_len, topk, init_blocks, local_blocks,
                                  out.data_ptr(), out.stride(0), out.stride(1), wp, wn,
                                  _stream(idx_q.device, stream)), "mm3idx_forward")
    return out[:, :rows, :]


def decode_static(idx_q, index_cache, block_table, seq_lens, *, query_len, max_seq_len, topk,
                  init_blocks, local_blocks, sm_scale, out=None, stream=None):
    """:func:`decode` for callers that cannot provide a workspace: the library
    uses its own fixed device array (STATIC_SCRATCH_BYTES), shared by every
    call, so calls that overlap on the GPU must not be issued."""
    p = _problem(idx_q, index_cache, block_table, seq_lens, query_len, max_seq_len, sm_scale)
    rows, heads = idx_q.shape[0], idx_q.shape[1]
    out = _ids_out(out, heads, rows, topk, idx_q.device)
    with _on(idx_q.device):
        _check(lib.mm3idx_decode_static(ctypes.byref(p), topk, init_blocks, local_blocks,
                                        out.data_ptr(), out.stride(0), out.stride(1),
                                        _stream(idx_q.device, stream)), "mm3idx_decode_static")
    return out[:, :rows, :]


def _stream_device(stream):
    return (torch.device(stream.device) if stream is not None
            else torch.device("cuda", torch.cuda.current_device()))


def check_wait_timeout(warps: int = 4, stream=None):
    """Make the bounded on-chip wait run out on purpose (about 2 s); the
    device status word of the stream's GPU then holds DEV_TIMEOUT (read it
    with get_device_error)."""
    dev = _stream_device(stream)
    with _on(dev):
        _check(lib.mm3idx_check_wait_timeout(warps, _stream(dev, stream)),
               "mm3idx_check_wait_timeout")


def get_device_error(stream=None) -> int:
    """Synchronise the stream (default: the current GPU's current stream),
    then read and clear the device status word of the stream's GPU."""
    dev = _stream_device(stream)
    v = ctypes.c_int32(0)
    with _on(dev):
        _check(lib.mm3idx_get_device_error(_stream(dev, stream), ctypes.byref(v)),
               "mm3idx_get_device_error")
    return v.value

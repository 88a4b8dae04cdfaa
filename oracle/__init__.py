"""CPU oracle for MiniMax-M3 lightning-indexer block scoring + top-k.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library does not
import, link or call anything here, and nothing here calls the CUDA library.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp64); this
module compiles it with gcc on first use and marshals numpy arrays to it.
Each C function cites the page passage it follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_F64 = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, no fast-math, no FMA
    contraction so results do not depend on the host architecture)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                    "-shared", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.mm3o_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.mm3o_e4m3_value.restype = _F64
        lib.mm3o_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.mm3o_e2m1_value.restype = _F64
        lib.mm3o_e4m3_rn_satfinite.argtypes = [_F64]
        lib.mm3o_e4m3_rn_satfinite.restype = ctypes.c_uint8
        lib.mm3o_nvfp4_value.argtypes = [ctypes.c_uint8, ctypes.c_uint8]
        lib.mm3o_nvfp4_value.restype = _F64
        lib.mm3o_block_scores_bf16.argtypes = [_P, _P, _I64, _P, _I64, _I64, _F64, _P]
        lib.mm3o_block_scores_bf16.restype = _I64
        lib.mm3o_block_scores_nvfp4.argtypes = [_P, _P, _P, _I64, _P, _I64, _I64, _F64, _P]
        lib.mm3o_block_scores_nvfp4.restype = _I64
        lib.mm3o_select.argtypes = [_P, _I64, _I32, _I32, _I32, _P]
        lib.mm3o_select.restype = _I32
        lib.mm3o_problem_bf16.argtypes = [_P, _I64, _I64, _I32, _P, _I64, _P, _I64,
                                          _I64, _P, _I32, _I32, _F64, _I32, _I32,
                                          _I32, _P, _I64, _P]
        lib.mm3o_problem_bf16.restype = _I32
        lib.mm3o_problem_nvfp4.argtypes = [_P, _I64, _I64, _I32, _P, _P, _I64, _P,
                                           _I64, _I64, _P, _I32, _I32, _F64, _I32,
                                           _I32, _I32, _P, _I64, _P]
        lib.mm3o_problem_nvfp4.restype = _I32
        lib.mm3o_select_problem.argtypes = [_P, _I64, _I64, _I32, _P, _I32, _I32,
                                            _I32, _I32, _I32, _P]
        lib.mm3o_select_problem.restype = _I32
        lib.mm3o_sparse_table.argtypes = [_P, _I32, _P, _I32, _I32, _P, _I64, _I32, _I32, _P,
                                          _I64, _P]
        lib.mm3o_sparse_table.restype = _I32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ numbers

def e4m3_value(b: int) -> float:
    return _load().mm3o_e4m3_value(b)


def e2m1_value(c: int) -> float:
    return _load().mm3o_e2m1_value(c)


def e4m3_rn_satfinite(x: float) -> int:
    return _load().mm3o_e4m3_rn_satfinite(x)


def nvfp4_value(code: int, scale: int) -> float:
    """e4m3_rn_satfinite(e2m1(code) * e4m3(scale)) as a float."""
    return _load().mm3o_nvfp4_value(code, scale)


def nvfp4_dequant_bf16(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise NVFP4 pages to bf16 bits (exact: every e4m3 value is a bf16
    value).  codes [..., 64], scales [..., 8] -> uint16 [..., 128]."""
    table = np.empty((256, 16), dtype=np.float32)
    for s in range(256):
        for c in range(16):
            table[s, c] = nvfp4_value(c, s)
    lo = codes & 15
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], 128)
    sc = np.repeat(scales, 16, axis=-1)
    vals = table[sc, nib]
    return (vals.view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------- per-row calls

def block_scores(wl, row: int, head: int) -> np.ndarray:
    """Scores (float64) of the visible blocks of one (row, head) of a workload."""
    lib = _load()
    i, j = divmod(row, wl.query_len)
    pos = int(wl.seq_lens[i]) - wl.query_len + j
    out = np.empty(max(1, wl.width), dtype=np.float64)
    q = np.ascontiguousarray(wl.q[row, head])
    trow = np.ascontiguousarray(wl.block_table[i])
    if wl.kv_format == "bf16":
        nb = lib.mm3o_block_scores_bf16(_ptr(q), _ptr(wl.cache), wl.num_pages,
                                        _ptr(trow), wl.width, pos, wl.sm_scale,
                                        _ptr(out))
    else:
        nb = lib.mm3o_block_scores_nvfp4(_ptr(q), _ptr(wl.codes), _ptr(wl.scales),
                                         wl.num_pages, _ptr(trow), wl.width, pos,
                                         wl.sm_scale, _ptr(out))
    if nb < 0:
        raise ValueError("oracle: table column or page out of range")
    return out[:nb].copy()


def select(scores: np.ndarray, topk: int, init_blocks: int, local_blocks: int) -> np.ndarray:
    """Top-k ids (ascending, -1 padded) of one row with len(scores) visible blocks."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    out = np.empty(topk, dtype=np.int32)
    if _load().mm3o_select(_ptr(s), s.shape[0], topk, init_blocks, local_blocks, _ptr(out)):
        raise ValueError("oracle: forced blocks exceed topk")
    return out


def row(wl, row_idx: int, head: int):
    s = block_scores(wl, row_idx, head)
    return s, select(s, wl.topk, wl.init_blocks, wl.local_blocks)


# --------------------------------------------------------- whole problems

def problem(wl, *, want_scores: bool = True, out_width: int | None = None):
    """Scores [heads, rows, out_width] (float64, -inf past each row's own block)
    and ids [heads, rows, topk] (int32) of a whole workload."""
    lib = _load()
    H, R = wl.heads, wl.rows
    W = out_width if out_width is not None else wl.width
    scores = np.empty((H, R, W), dtype=np.float64) if want_scores else None
    ids = np.empty((H, R, wl.topk), dtype=np.int32)
    q = np.ascontiguousarray(wl.q)
    tbl = np.ascontiguousarray(wl.block_table)
    sl = np.ascontiguousarray(wl.seq_lens, dtype=np.int32)
    sp = _ptr(scores) if want_scores else None
    if wl.kv_format == "bf16":
        rc = lib.mm3o_problem_bf16(_ptr(q), H * 128, 128, H, _ptr(wl.cache),
                                   wl.num_pages, _ptr(tbl), wl.width, wl.width,
                                   _ptr(sl), wl.num_reqs, wl.query_len, wl.sm_scale,
                                   wl.topk, wl.init_blocks, wl.local_blocks, sp, W,
                                   _ptr(ids))
    else:
        rc = lib.mm3o_problem_nvfp4(_ptr(q), H * 128, 128, H, _ptr(wl.codes),
                                    _ptr(wl.scales), wl.num_pages, _ptr(tbl),
                                    wl.width, wl.width, _ptr(sl), wl.num_reqs,
                                    wl.query_len, wl.sm_scale, wl.topk,
                                    wl.init_blocks, wl.local_blocks, sp, W, _ptr(ids))
    if rc:
        raise ValueError("oracle: table column, page or selection arguments out of range")
    return scores, ids


def problem_ragged(wl, *, want_scores: bool = True, out_width: int | None = None):
    """problem() of a ragged batch (wl.cu_seqlens set): every request is its
    own uniform problem of cu[i+1] - cu[i] query rows (index_topk,
    minimax_m3_index_score: cu_seqlens_q and prefix_lens give each request's
    query rows and their positions), and the rows are laid out in cu order."""
    import copy
    cu = wl.cu_seqlens
    H, R = wl.heads, wl.rows
    W = out_width if out_width is not None else wl.width
    scores = np.full((H, R, W), -np.inf) if want_scores else None
    ids = np.empty((H, R, wl.topk), dtype=np.int32)
    for i in range(wl.num_reqs):
        lo, hi = int(cu[i]), int(cu[i + 1])
        if hi == lo:
            continue
        sub = copy.copy(wl)
        sub.cu_seqlens = None
        sub.query_len = hi - lo
        sub.seq_lens = wl.seq_lens[i:i + 1].copy()
        sub.block_table = wl.block_table[i:i + 1].copy()
        sub.q = wl.q[lo:hi].copy()
        s, k = problem(sub, want_scores=want_scores, out_width=W)
        if want_scores:
            scores[:, lo:hi] = s
        ids[:, lo:hi] = k
    return scores, ids


def select_problem(scores: np.ndarray, seq_lens: np.ndarray, query_len: int,
                   topk: int, init_blocks: int, local_blocks: int) -> np.ndarray:
    """Ids [heads, rows, topk] selected from a given score tensor [heads, rows, W]."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    H, R, W = s.shape
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ids = np.empty((H, R, topk), dtype=np.int32)
    if _load().mm3o_select_problem(_ptr(s), R * W, W, H, _ptr(sl), sl.shape[0],
                                   query_len, topk, init_blocks, local_blocks, _ptr(ids)):
        raise ValueError("oracle: forced blocks exceed topk")
    return ids


def sparse_table(ids: np.ndarray, seq_lens: np.ndarray, query_len: int,
                 attention_block_table: np.ndarray, pages_per_block: int,
                 block_page_stride: int):
    """Sparse page table [rows, topk * pages_per_block] (int32, -1 in unused
    slots) and sparse context lengths [rows] (int32) of one head's ids
    [rows, topk], through the attention block table [num_reqs, >= blocks]."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rows, topk = ids.shape
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    at = np.ascontiguousarray(attention_block_table, dtype=np.int32)
    table = np.empty((rows, topk * pages_per_block), dtype=np.int32)
    ctx = np.empty((rows,), dtype=np.int32)
    if _load().mm3o_sparse_table(_ptr(ids), topk, _ptr(sl), sl.shape[0], query_len, _ptr(at),
                                 at.shape[1], pages_per_block, block_page_stride, _ptr(table),
                                 table.shape[1], _ptr(ctx)):
        raise ValueError("oracle: an id past the row's visible blocks")
    return table, ctx


def subset(wl, reqs):
    """The same workload restricted to the given requests (same pages)."""
    import copy
    reqs = np.asarray(reqs)
    sub = copy.copy(wl)
    sub.seq_lens = wl.seq_lens[reqs].copy()
    sub.block_table = wl.block_table[reqs].copy()
    rows = (reqs[:, None] * wl.query_len + np.arange(wl.query_len)[None, :]).reshape(-1)
    sub.q = wl.q[rows].copy()
    return sub

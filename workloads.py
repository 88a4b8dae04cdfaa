"""Seeded synthetic inputs for the lightning-indexer block scorer.

This module is shared by the CPU oracle's tests, the CUDA parity tests, the
smoke check and the benchmark.  It holds none of the method's arithmetic: no
dot products, masks, block maxima or selection.  It only draws random numbers,
rounds them to bf16, deals pages from a shuffled pool into block tables, and
encodes random keys as NVFP4 (e2m1 codes with one e4m3 scale per 16 elements).

Layouts produced (they follow the vLLM MiniMax-M3 "index_topk" page, module
docstring and `minimax_m3_index_decode` argument comments):

* ``q``      uint16 bf16 bits ``[tokens, heads, 128]``, tokens request-major,
  ``tokens = num_reqs * query_len``; query ``j`` of request ``i`` sits at
  position ``seq_len[i] - query_len + j``.
* ``cache``  uint16 bf16 bits ``[pages, 128, 128]``: one page is one 128-token
  sparse block; every index head reads the same key for a token.
* ``codes``/``scales`` (NVFP4 variant) uint8 ``[pages, 128, 64]`` with element
  ``2e`` in the low nibble and ``2e+1`` in the high nibble, and uint8
  ``[pages, 128, 8]`` e4m3 scale bytes, scale ``g`` covering ``d`` in
  ``[16g, 16g+16)``.
* ``block_table`` int32 ``[num_reqs, width]``, ``width = cdiv(max_seq_len,128)``;
  entries a request does not use hold ``num_pages + 7`` (never to be read).
* token slots of a request's last page past ``seq_len`` hold +100 (bf16) or
  the largest NVFP4 value, so that a kernel which fails to mask them is caught.

Recipes for the five named workloads are in ``WORKLOADS``; every draw comes from
``numpy.random.default_rng(seed)``.
"""

from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os

import numpy as np

D = 128
BLOCK = 128
POISON_BF16 = 0x42C8          # bf16 bit pattern of +100.0
POISON_CODE = 0x77            # two e2m1 codes of +6.0
POISON_SCALE = 0x7E           # e4m3 448.0


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); return
    uint16 bits.  (No finite float32 overflows the 32-bit sum below.)"""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    u += np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))
    return (u >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    heads: int
    query_len: int
    max_seq_len: int
    topk: int
    init_blocks: int
    local_blocks: int
    sm_scale: float
    seq_lens: np.ndarray          # int32 [num_reqs]
    block_table: np.ndarray       # int32 [num_reqs, width]
    q: np.ndarray                 # uint16 bf16 bits [tokens, heads, 128]
    num_pages: int
    kv_format: str = "bf16"       # "bf16" or "nvfp4"
    cache: np.ndarray | None = None    # uint16 [pages, 128, 128]
    codes: np.ndarray | None = None    # uint8  [pages, 128, 64]
    scales: np.ndarray | None = None   # uint8  [pages, 128, 8]
    # ragged batches: int32 [num_reqs + 1] query-row offsets (query_len then
    # holds the largest per-request count); None: query_len rows per request
    cu_seqlens: np.ndarray | None = None

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def rows(self) -> int:
        if self.cu_seqlens is not None:
            return int(self.cu_seqlens[-1])
        return self.num_reqs * self.query_len

    @property
    def width(self) -> int:
        return int(self.block_table.shape[1])

    def key_bytes(self) -> int:
        """Bytes of index-K a full pass must read: every block up to each
        request's last visible block (the visible pages, counted whole)."""
        per_tok = D * 2 if self.kv_format == "bf16" else D // 2 + D // 16
        nb = (self.seq_lens.astype(np.int64) + BLOCK - 1) // BLOCK
        return int(nb.sum()) * BLOCK * per_tok


def _deal_pages(rng, seq_lens, max_seq_len, pool_pages=None):
    need = (seq_lens.astype(np.int64) + BLOCK - 1) // BLOCK
    total = int(need.sum())
    pages = pool_pages if pool_pages is not None else int(math.ceil(1.25 * total))
    assert pages >= total
    perm = rng.permutation(pages).astype(np.int32)
    width = (max_seq_len + BLOCK - 1) // BLOCK
    table = np.full((len(seq_lens), width), pages + 7, dtype=np.int32)
    off = 0
    for i, n in enumerate(need):
        table[i, :n] = perm[off:off + n]
        off += n
    return table, pages


def _poison_tails_bf16(cache, table, seq_lens):
    for i, s in enumerate(seq_lens):
        s = int(s)
        if s % BLOCK:
            cache[table[i, s // BLOCK], s % BLOCK:, :] = POISON_BF16


def _poison_tails_nvfp4(codes, scales, table, seq_lens):
    for i, s in enumerate(seq_lens):
        s = int(s)
        if s % BLOCK:
            p = table[i, s // BLOCK]
            codes[p, s % BLOCK:, :] = POISON_CODE
            scales[p, s % BLOCK:, :] = POISON_SCALE


def _parallel_fill(seed_key, n_items, chunk, fn):
    """Run fn(rng, lo, hi) over [0, n_items) in chunks on a thread pool.  Chunk
    k always draws from child k of SeedSequence(seed_key), so the result does
    not depend on thread scheduling."""
    nchunks = max(1, (n_items + chunk - 1) // chunk)
    kids = np.random.SeedSequence(seed_key).spawn(nchunks)

    def work(k):
        fn(np.random.default_rng(kids[k]), k * chunk, min(n_items, (k + 1) * chunk))

    with cf.ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 4)) as ex:
        list(ex.map(work, range(nchunks)))


def _normal_bf16(seed_key, shape, chunk=1 << 22):
    """Standard normals rounded to bf16."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(rng, lo, hi):
        out[lo:hi] = bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))

    _parallel_fill(seed_key, n, chunk, fill)
    return out.reshape(shape)


# e2m1 magnitudes (OCP MX v1.0, FP4 E2M1): codes 0..7 -> these values.
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def _e4m3_scale_bytes(amax_over_6: np.ndarray) -> np.ndarray:
    """Scale bytes for the quantiser: torch's float8_e4m3fn rounding of amax/6
    (a data-generation choice; the method only ever decodes these bytes)."""
    import torch
    t = torch.from_numpy(np.minimum(amax_over_6, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_decode_table() -> np.ndarray:
    import torch
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float32).numpy()


_E4M3_TABLE = _e4m3_decode_table()
_E2M1_MID = (_E2M1[1:] + _E2M1[:-1]) / 2


def nvfp4_encode(x: np.ndarray):
    """Encode float32 keys ``[..., 128]`` as (codes ``[..., 64]``, scales ``[..., 8]``).

    Per 16-element group: scale byte = e4m3(amax/6); code = the e2m1
    magnitude nearest to ``|x|/scale`` (clamped to 6; a value exactly half
    way goes to the larger magnitude) with the sign in bit 3.
    """
    shape = x.shape
    g = x.reshape(-1, 16)
    ag = np.abs(g)
    amax = ag.max(axis=1)
    sb = _e4m3_scale_bytes(amax / 6.0)
    sv = _E4M3_TABLE[sb]
    inv = np.where(sv > 0, 1.0 / np.where(sv > 0, sv, 1.0), 0.0).astype(np.float32)
    mag = np.searchsorted(_E2M1_MID, ag * inv[:, None], side="right").astype(np.uint8)
    code = mag | ((g < 0).astype(np.uint8) << 3)
    code = code.reshape(-1, 8, 2)
    packed = (code[..., 0] | (code[..., 1] << 4)).astype(np.uint8)
    codes = packed.reshape(*shape[:-1], 64)
    scales = sb.reshape(*shape[:-1], 8)
    return codes, scales


def build(name, *, seed, seq_lens, query_len, heads, topk, init_blocks,
          local_blocks, max_seq_len, sm_scale=1.0 / math.sqrt(128.0),
          kv_format="bf16", block_offset_std=0.0, pool_pages=None,
          poison=True, query_lens=None):
    """Draw a workload with the given shape.  default_rng(seed) draws the
    block-table permutation and the block offsets; keys and queries come from
    the child streams of SeedSequence([seed, 1]) and ([seed, 2]).  With
    ``query_lens`` (one count per request) the batch is ragged: request i
    owns query rows cu[i]..cu[i+1]-1 at positions seq_len - count + j."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    table, pages = _deal_pages(rng, seq_lens, max_seq_len, pool_pages)
    wl = Workload(name=name, heads=heads, query_len=query_len,
                  max_seq_len=max_seq_len, topk=topk, init_blocks=init_blocks,
                  local_blocks=local_blocks, sm_scale=float(sm_scale),
                  seq_lens=seq_lens, block_table=table, q=None, num_pages=pages,
                  kv_format=kv_format)
    if kv_format == "bf16":
        if block_offset_std:
            # One scalar offset per page; a page is one (request, logical
            # block), so this is the per-block offset of the recipe.
            offs = rng.normal(0.0, block_offset_std, size=pages).astype(np.float32)
            cache = np.empty((pages, BLOCK, D), dtype=np.uint16)

            def fill(r, lo, hi):
                k = r.standard_normal((hi - lo, BLOCK, D), dtype=np.float32)
                k += offs[lo:hi, None, None]
                cache[lo:hi] = bf16_bits(k)

            _parallel_fill([seed, 1], pages, 256, fill)
        else:
            cache = _normal_bf16([seed, 1], (pages, BLOCK, D))
        if poison:
            _poison_tails_bf16(cache, table, seq_lens)
        wl.cache = cache
    elif kv_format == "nvfp4":
        codes = np.empty((pages, BLOCK, D // 2), dtype=np.uint8)
        scales = np.empty((pages, BLOCK, D // 16), dtype=np.uint8)

        def fill(r, lo, hi):
            k = r.standard_normal((hi - lo, BLOCK, D), dtype=np.float32)
            codes[lo:hi], scales[lo:hi] = nvfp4_encode(k)

        _parallel_fill([seed, 1], pages, 256, fill)
        if poison:
            _poison_tails_nvfp4(codes, scales, table, seq_lens)
        wl.codes, wl.scales = codes, scales
    else:
        raise ValueError(kv_format)
    if query_lens is not None:
        ql = np.asarray(query_lens, dtype=np.int64)
        wl.cu_seqlens = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        wl.query_len = int(ql.max()) if len(ql) else 1
        tokens = int(wl.cu_seqlens[-1])
    else:
        tokens = len(seq_lens) * query_len
    wl.q = _normal_bf16([seed, 2], (tokens, heads, D))
    return wl


def _tiny_decode(seed=0):
    return build("tiny decode", seed=seed, seq_lens=[300, 700], query_len=1,
                 heads=1, topk=4, init_blocks=1, local_blocks=1,
                 max_seq_len=700, pool_pages=16)


def _spec_decode(seed=1, num_reqs=64):
    rng = np.random.default_rng(1000 + seed)
    seq = rng.integers(4096, 32768, size=num_reqs, endpoint=True)
    return build("spec-decode batch", seed=seed, seq_lens=seq, query_len=4,
                 heads=1, topk=16, init_blocks=1, local_blocks=2,
                 max_seq_len=32768)


def _high_batch(seed=2, num_reqs=256):
    rng = np.random.default_rng(1000 + seed)
    seq = np.exp(rng.uniform(math.log(1024), math.log(65536), size=num_reqs))
    seq = np.clip(np.round(seq), 1024, 65536).astype(np.int32)
    return build("high-batch decode", seed=seed, seq_lens=seq, query_len=4,
                 heads=4, topk=16, init_blocks=1, local_blocks=2,
                 max_seq_len=65536, block_offset_std=0.5)


def _causal_prefill(seed=3, seq=32768):
    return build("causal prefill", seed=seed, seq_lens=[seq], query_len=seq,
                 heads=1, topk=16, init_blocks=1, local_blocks=2,
                 max_seq_len=seq)


def _causal_prefill_topk32(seed=3, seq=32768):
    """The causal prefill's inputs with 32 selected blocks a row; not one of
    the five named configurations."""
    return build("causal prefill, topk 32", seed=seed, seq_lens=[seq], query_len=seq,
                 heads=1, topk=32, init_blocks=1, local_blocks=2,
                 max_seq_len=seq)


def _nvfp4_decode(seed=4, num_reqs=128):
    rng = np.random.default_rng(1000 + seed)
    seq = rng.integers(32768, 131072, size=num_reqs, endpoint=True)
    return build("NVFP4 decode", seed=seed, seq_lens=seq, query_len=4,
                 heads=1, topk=16, init_blocks=1, local_blocks=2,
                 max_seq_len=131072, kv_format="nvfp4")


def _nvfp4_prefill(seed=5, seq=32768):
    """The causal prefill over NVFP4 keys (indexer_nvfp4 prefill branch);
    not one of the five named configurations."""
    return build("NVFP4 causal prefill", seed=seed, seq_lens=[seq], query_len=seq,
                 heads=1, topk=16, init_blocks=1, local_blocks=2,
                 max_seq_len=seq, kv_format="nvfp4")


def _chunked_prefill(seed=6, num_reqs=8):
    """A ragged prefill batch: request i brings U[1000, 8000] new tokens after
    U[0, 24000] earlier ones (chunked prefill); not one of the five named
    configurations."""
    rng = np.random.default_rng(1000 + seed)
    ql = rng.integers(1000, 8000, size=num_reqs, endpoint=True)
    pre = rng.integers(0, 24000, size=num_reqs, endpoint=True)
    return ragged_case(seed, query_lens=ql, prefix_lens=pre, heads=1, topk=16, init_blocks=1,
                       local_blocks=2, max_seq_len=32768, name="chunked prefill batch")


def _mixed_batch(seed=8):
    """The spec-decode batch's 64 decode requests (4 rows each, 4K-32K tokens)
    followed by two chunked prefills of 4096 new tokens after 8192 and 16384
    earlier ones, as one ragged batch (decode rows first); not one of the
    five named configurations."""
    rng = np.random.default_rng(1000 + 1)
    seq = rng.integers(4096, 32768, size=64, endpoint=True)
    ql = [4] * 64 + [4096, 4096]
    pre = [int(x) - 4 for x in seq] + [8192, 16384]
    return ragged_case(seed, query_lens=ql, prefix_lens=pre, heads=1, topk=16, init_blocks=1,
                       local_blocks=2, max_seq_len=32768, name="mixed decode + prefill batch")


# The five named workloads, by short key, the NVFP4 prefill, the causal
# prefill at topk 32, a chunked (ragged) prefill batch and a mixed batch.  The second argument of each maker
# (request count / sequence length) lets tests draw a smaller case with the
# same recipe.
WORKLOADS = {
    "tiny": _tiny_decode,
    "spec_decode": _spec_decode,
    "high_batch": _high_batch,
    "prefill": _causal_prefill,
    "prefill_topk32": _causal_prefill_topk32,
    "nvfp4_decode": _nvfp4_decode,
    "nvfp4_prefill": _nvfp4_prefill,
    "chunked_prefill": _chunked_prefill,
    "mixed_batch": _mixed_batch,
}


def make(key: str, **kw) -> Workload:
    return WORKLOADS[key](**kw)


def random_case(seed, *, num_reqs, query_len, heads, topk, init_blocks,
                local_blocks, min_len, max_len, max_seq_len=None,
                kv_format="bf16", sm_scale=None, block_offset_std=0.0):
    """A small random case for parity sweeps (lengths uniform in
    [min_len, max_len], at least ``query_len``)."""
    rng = np.random.default_rng(50_000 + seed)
    lo = max(min_len, query_len)
    seq = rng.integers(lo, max(lo, max_len), size=num_reqs, endpoint=True)
    msl = max_seq_len or int(seq.max())
    return build(f"random-{seed}", seed=seed, seq_lens=seq, query_len=query_len,
                 heads=heads, topk=topk, init_blocks=init_blocks,
                 local_blocks=local_blocks, max_seq_len=msl,
                 sm_scale=sm_scale if sm_scale is not None else 1.0 / math.sqrt(128.0),
                 kv_format=kv_format, block_offset_std=block_offset_std)


def ragged_case(seed, *, query_lens, prefix_lens, heads, topk, init_blocks, local_blocks,
                max_seq_len=None, kv_format="bf16", sm_scale=None, name=None):
    """A ragged batch: request i has query_lens[i] new tokens after
    prefix_lens[i] earlier ones (seq_len = prefix + count)."""
    ql = np.asarray(query_lens, dtype=np.int64)
    seq = (np.asarray(prefix_lens, dtype=np.int64) + ql).astype(np.int32)
    msl = max_seq_len or int(max(1, seq.max()))
    return build(name or f"ragged-{seed}", seed=seed, seq_lens=seq, query_len=1, heads=heads,
                 topk=topk, init_blocks=init_blocks, local_blocks=local_blocks,
                 max_seq_len=msl,
                 sm_scale=sm_scale if sm_scale is not None else 1.0 / math.sqrt(128.0),
                 kv_format=kv_format, query_lens=ql)


def attention_block_table(wl: Workload, seed: int, spare: int = 3) -> np.ndarray:
    """A seeded attention block table for the sparse page table: int32
    ``[num_reqs, width]``, the blocks a request uses drawn without
    repetition from a pool ``spare`` times the need; entries a request does
    not use hold -7777 (never to be read)."""
    rng = np.random.default_rng(90_000 + seed)
    width = wl.block_table.shape[1]
    used = [min(width, -(-int(max(s, 0)) // 128)) for s in wl.seq_lens]
    pool = rng.permutation(max(1, spare * sum(used))).astype(np.int32)
    out = np.full((wl.num_reqs, width), -7777, dtype=np.int32)
    k = 0
    for i, n in enumerate(used):
        out[i, :n] = pool[k:k + n]
        k += n
    return out

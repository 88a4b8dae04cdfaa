"""The benchmark's own arithmetic, on CPU: the algorithmic bytes and flops
the roofline divides by, the lookup of ncu traffic in the committed
summaries (only when they were taken on the current kernel sources), and
the JSON line's required keys in the reference arm."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_prefill_flops_closed_form():
    # one request of S tokens, all rows new: sum over rows of 2*128*(pos+1)
    wl = W.build("f", seed=1, seq_lens=[300], query_len=300, heads=1, topk=4, init_blocks=1,
                 local_blocks=1, max_seq_len=300)
    assert bench.prefill_flops(wl) == 2 * 128 * (300 * 301 // 2)
    # 128 new rows after a 1000-token prefix, 2 heads
    wl = W.build("f", seed=1, seq_lens=[1128], query_len=128, heads=2, topk=4, init_blocks=1,
                 local_blocks=1, max_seq_len=1128)
    assert bench.prefill_flops(wl) == 2 * 2 * 128 * sum(p + 1 for p in range(1000, 1128))
    # ragged: the sum of its requests'
    wl = W.ragged_case(3, query_lens=[5, 0, 130], prefix_lens=[10, 7, 300], heads=1, topk=4,
                       init_blocks=1, local_blocks=1)
    want = sum(2 * 128 * sum(p + 1 for p in range(pre, pre + q))
               for q, pre in [(5, 10), (0, 7), (130, 300)])
    assert bench.prefill_flops(wl) == want


def test_decode_bytes_closed_form():
    wl = W.make("tiny")   # seq 300 and 700, one head, query_len 1, topk 4
    keys = (300 + 700) * 256
    queries = 2 * 1 * 128 * 2
    table = (3 + 6) * 4
    lengths = 2 * 4
    ids = 1 * 2 * 4 * 4
    assert bench.decode_bytes(wl) == keys + queries + table + lengths + ids
    wl4 = W.random_case(2, num_reqs=3, query_len=2, heads=1, topk=4, init_blocks=1,
                        local_blocks=1, min_len=100, max_len=900, kv_format="nvfp4")
    assert bench.decode_bytes(wl4) == (int(wl4.seq_lens.sum()) * 72 + wl4.q.nbytes
                                       + int(((wl4.seq_lens + 127) // 128).sum()) * 4
                                       + wl4.seq_lens.nbytes + wl4.rows * 4 * 4)


def test_profiled_traffic_requires_matching_sources(tmp_path, monkeypatch):
    sha = bench.kernel_sources_sha(bench.DECODE_SOURCES)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "match.md").write_text(f"source_sha256: {sha}\ntraffic_bytes_per_launch: 1234\n")
    (prof / "stale.md").write_text("source_sha256: 0123456789abcdef\n"
                                   "traffic_bytes_per_launch: 99\n")
    csrc = tmp_path / "sparse_attention_block_paged_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for n in bench.DECODE_SOURCES:
        src = os.path.join(ROOT, "sparse_attention_block_paged_gb300", "csrc", n)
        (csrc / n).write_bytes(open(src, "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("match.md", bench.DECODE_SOURCES) == 1234
    assert bench.profiled_traffic("stale.md", bench.DECODE_SOURCES) is None
    assert bench.profiled_traffic("missing.md", bench.DECODE_SOURCES) is None
    (csrc / bench.DECODE_SOURCES[0]).write_bytes(b"// changed\n")
    assert bench.profiled_traffic("match.md", bench.DECODE_SOURCES) is None


def test_committed_summaries_carry_sha_and_traffic():
    for name in ("decode_spec_decode.md", "decode_high_batch.md", "decode_nvfp4_decode.md",
                 "prefill_scorer_causal_prefill.md"):
        txt = open(os.path.join(ROOT, "profiles", name)).read()
        assert "source_sha256:" in txt and "traffic_bytes_per_launch:" in txt, name
        assert "--clock-control none" in txt, name


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["value"] > 0
    assert d["warmup"] >= 3          # at least three warm-up steps, whatever is asked

"""The benchmark's host-side parts: the oracle sample behind `cpu_baseline` and the
`--impl reference` arm (one JSON line, rank 0) on the tiny workload, and the page
accounting of the all-BF16 comparison at a fixed HBM budget."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import oscar_synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_sample_all_cores_and_one_core():
    r = bench.oracle_sample(syn.WORKLOADS["tiny_gqa4_1k"], 0.4)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s"
    assert r["cores"] >= 1
    assert r["value"] > 0 and r["single_core_value"] > 0
    assert f"on {r['cores']} host cores" in r["sample"]


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_gqa4_1k", "--steps", "2", "--warmup", "3", "--cpu-seconds", "0.6"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] == d["cpu_baseline"]["value"] == d["e2e"]["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s"


def test_bf16_budget_batch_ragged_shared_prefix():
    # the ragged batch of 32 with a 16,384-token shared prefix: an all-BF16 cache of the same HBM
    # footprint holds the first 4 requests (prefix pages once)
    w = syn.WORKLOADS["qwen3_8b_b32_ragged"]
    seq = syn.context_lengths(w)
    pl = syn.page_layout(w, seq)
    r = bench.bf16_budget_batch(w, seq, pl.n_int2_pages, pl.n_bf16_pages)
    int2_page, bf16_page = bench.cache_page_bytes(w)
    assert r["budget_bytes"] == (pl.n_int2_pages * int2_page + pl.n_bf16_pages * bf16_page) * w.layers
    assert r["batch"] == 4
    assert r["bf16_cache_bytes"] <= r["budget_bytes"]
    table, n = bench.bf16_cache_table(w, seq[:r["batch"] + 1], max((t + 63) // 64 for t in seq))
    assert n * bf16_page * w.layers > r["budget_bytes"]                # one more request does not fit
    table, n = bench.bf16_cache_table(w, seq[:r["batch"]], pl.int2_table.shape[1])
    assert n * bf16_page * w.layers == r["bf16_cache_bytes"]


def test_bf16_cache_table_shares_prefix_pages():
    w = syn.WORKLOADS["qwen3_8b_b32_ragged"]
    seq = [20000, 17000, 16384 + 64 * 3 + 1]
    table, n = bench.bf16_cache_table(w, seq, 400)
    shared = w.shared_prefix // w.page_size
    assert (table[1, :shared] == table[0, :shared]).all() and (table[2, :shared] == table[0, :shared]).all()
    own = [(t + 63) // 64 for t in seq]
    assert n == own[0] + (own[1] - shared) + (own[2] - shared)
    used = np.concatenate([table[0, :own[0]], table[1, shared:own[1]], table[2, shared:own[2]]])
    assert sorted(used.tolist()) == list(range(n))                 # every physical page once
    assert (table[0, own[0]:] == -1).all() and (table[2, own[2]:] == -1).all()


def test_bf16_budget_single_request_always_runs():
    # at batch 1 the BF16 cache never fits the INT2 footprint; the comparison still runs one request
    w = syn.WORKLOADS["qwen3_8b_100k"]
    seq = syn.context_lengths(w)
    pl = syn.page_layout(w, seq)
    r = bench.bf16_budget_batch(w, seq, pl.n_int2_pages, pl.n_bf16_pages)
    assert r["batch"] == 1 and r["bf16_cache_bytes"] > r["budget_bytes"]

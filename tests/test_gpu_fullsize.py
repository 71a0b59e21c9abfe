"""Parity at the workloads' full sizes, on sampled (request, query head) outputs.

Each case runs the decode step exactly as bench.py does (oscar_decode_attention_fused
with the history taken in dynamic 64-token units, then oscar_merge, launch overlap on,
the library's split suggestion for the batch), then compares sampled heads with the
oracle's fp64 attention over its own demotion of those heads' history.  Samples
always include the shortest and the longest request.  K/V are drawn on the GPU
(the oracle reads back the sampled heads), so the same tensors feed both sides.
"""
import numpy as np
import pytest
import torch

import oracle
import oscar_synthetic as syn
from bit_kv_cache_oscar_gb300 import binding as ob
from tests import scenario as sc
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu

D = 128


def _run_like_bench(case, dynamic=True, demote=False):
    L, dev = case.layout, case.dev
    B = len(case.seq)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S = ob.oscar_suggest_splits(L, B, int(max(case.hist_end)) - L.sink, sms)
    part = ob.Partials.empty(L, B, S)
    out32 = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    out = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    # with demote: the token at hist_end leaves the recent window and is demoted in the same launch
    dem = dict(demote_pos=dev["hist_end"].clone(), R_V=dev["RV"], c_K=oracle.C_K, c_V=oracle.C_V) if demote else {}
    try:
        ob.oscar_set_launch_overlap(True)
        tiles = torch.zeros(2 * B, dtype=torch.int32, device="cuda") if dynamic else None
        ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                        dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part,
                                        tile_counters=tiles, **dem)
        ob.oscar_merge(L, part, dev["RV"], out, out32, None)
        torch.cuda.synchronize()
        assert tiles is None or not tiles.any()
    finally:
        ob.oscar_set_launch_overlap(False)
    assert ob.oscar_get_device_status() == 0
    return out, out32


def _check(case, out, out32, pairs, ref=None):
    ref = ref or sc.oracle_outputs(case, pairs)
    o32 = out32.cpu().numpy()
    ob16 = out.float().cpu().numpy()
    for (b, hq), (o_ref, _) in ref.items():
        ok, r, m = sc.tolerance_ok(o32[b, hq][None], o_ref[None])
        assert ok, (b, hq, r, m)
        # the bf16 output is the fp32 one rounded to nearest even
        assert np.array_equal(ob16[b, hq], torch.from_numpy(o32[b, hq]).bfloat16().float().numpy())


def _pairs(seq, gqa, kv_heads, per_head=2):
    """Shortest and longest request x the given kv heads x per_head of their query heads."""
    reqs = sorted({int(np.argmin(seq)), int(np.argmax(seq))})
    pairs = []
    for b in reqs:
        for h in kv_heads:
            for j in range(per_head):
                pairs.append((b, h * gqa + (j * (gqa - 1)) // max(per_head - 1, 1)))
    return pairs


@pytest.mark.parametrize("dynamic", [False, True])
def test_fullsize_qwen3_8b_100k(dynamic):
    """The benchmark's workload: 32 q / 8 kv heads, one request of 100,000 tokens, page 64; fixed
    history splits and dynamic 64-token units."""
    w = syn.WORKLOADS["qwen3_8b_100k"]
    case = sc.make_case(n_kv=w.n_kv_heads, gqa=w.n_q_heads // w.n_kv_heads, page_size=w.page_size,
                        group=w.group, seq=(w.context,), gen_device="cuda")
    sc.upload(case, keep_rotated=False)
    out, out32 = _run_like_bench(case, dynamic)
    pairs = [(0, hq) for hq in (0, 3, 9, 14, 17, 22, 28, 31)]     # kv heads 0, 2, 4, 7
    _check(case, out, out32, pairs)


@pytest.mark.parametrize("dynamic", [False, True])
def test_fullsize_qwen3_8b_32k_step_with_demotion(dynamic):
    """The 32K workload's decode step: 32 q / 8 kv heads, one request of 32,768 tokens, page 64,
    the token at hist_end = T - 257 leaving the recent window and demoted by the same launch (in
    the window CTAs with fixed splits, in the first history CTAs with dynamic units).  Sampled
    heads' outputs against the oracle's attention (that token still read from BF16 this step),
    and the demoted row's codes, scale and zero of every kv head against the oracle's demotion."""
    w = syn.WORKLOADS["qwen3_8b_32k"]
    T = w.context
    he = T - w.recent - 1
    case = sc.make_case(n_kv=w.n_kv_heads, gqa=w.n_q_heads // w.n_kv_heads, page_size=w.page_size,
                        group=w.group, seq=(T,), gen_device="cuda", hist_end=[he])
    sc.upload(case, keep_rotated=False)
    out, out32 = _run_like_bench(case, dynamic, demote=True)
    pairs = [(0, hq) for hq in (1, 6, 8, 15, 19, 20, 26, 29)]      # kv heads 0, 1, 2, 3, 4, 5, 6, 7
    _check(case, out, out32, pairs)
    L, i2 = case.layout, case.dev["int2"]
    pg, sl = int(case.pages.int2_table[0, he // L.page_size]), he % L.page_size
    for h in range(L.n_kv_heads):
        kb = bf16_bits(case.K[0][he:he + 1, h])
        vb = bf16_bits(case.V[0][he:he + 1, h])
        _, pk, zk, sk = oracle.demote_rows(kb, case.RK[h], L.group, oracle.C_K)
        _, pv, zv, sv = oracle.demote_rows(vb, case.RV[h], L.group, oracle.C_V)
        assert np.array_equal(i2.codes_k[pg, sl, h].cpu().numpy(), pk[0]), h
        assert np.array_equal(i2.codes_v[pg, sl, h].cpu().numpy(), pv[0]), h
        assert np.array_equal(bf16_bits(i2.zero_k[pg, sl, h]), zk[0]), h
        assert np.array_equal(bf16_bits(i2.scale_k[pg, sl, h]), sk[0]), h
        assert np.array_equal(bf16_bits(i2.zero_v[pg, sl, h]), zv[0]), h
        assert np.array_equal(bf16_bits(i2.scale_v[pg, sl, h]), sv[0]), h


@pytest.mark.parametrize("name", ["qwen3_32b_131k_g128", "qwen3_32b_131k_g32"])
def test_fullsize_qwen3_32b_131k(name):
    """64 q / 8 kv heads (GQA 8), 4 requests of 131,072 tokens, groups of 128 and of 32."""
    w = syn.WORKLOADS[name]
    seq = tuple([w.context] * w.batch)
    case = sc.make_case(n_kv=w.n_kv_heads, gqa=w.n_q_heads // w.n_kv_heads, page_size=w.page_size,
                        group=w.group, seq=seq, gen_device="cuda")
    sc.upload(case, keep_rotated=False)
    out, out32 = _run_like_bench(case)
    pairs = [(0, 8), (0, 15), (0, 48), (0, 55), (3, 8), (3, 15), (3, 48), (3, 55)]
    _check(case, out, out32, pairs)


def test_fullsize_ragged_shared_prefix():
    """The ragged-batch shape (contexts drawn from 65,536..100,000, a 16,384-token prefix shared
    through the page tables) at 4 requests instead of 32."""
    w = syn.WORKLOADS["qwen3_8b_b32_ragged"]
    seq = tuple(int(t) for t in syn.context_lengths(w)[:4])
    case = sc.make_case(n_kv=w.n_kv_heads, gqa=w.n_q_heads // w.n_kv_heads, page_size=w.page_size,
                        group=w.group, seq=seq, gen_device="cuda", shared_prefix=w.shared_prefix)
    sc.upload(case, keep_rotated=False)
    out, out32 = _run_like_bench(case)
    _check(case, out, out32, _pairs(seq, case.layout.gqa, (1, 6)))


def test_fullsize_ragged_batch32():
    """The batch-32 target shape at its full size: 32 requests with contexts drawn from
    65,536..100,000, a 16,384-token prefix shared through the page tables, run as the benchmark
    runs it (one window cluster per request, the library's split suggestion for 32 requests),
    with fixed history splits and then with dynamic 64-token units; sampled heads of the shortest
    and the longest request and of two more requests against the oracle."""
    w = syn.WORKLOADS["qwen3_8b_b32_ragged"]
    seq = tuple(int(t) for t in syn.context_lengths(w))
    assert len(seq) == 32
    case = sc.make_case(n_kv=w.n_kv_heads, gqa=w.n_q_heads // w.n_kv_heads, page_size=w.page_size,
                        group=w.group, seq=seq, gen_device="cuda", shared_prefix=w.shared_prefix)
    sc.upload(case, keep_rotated=False)
    reqs = sorted({int(np.argmin(seq)), int(np.argmax(seq)), 5, 21})
    pairs = [(b, hq) for b in reqs for hq in (4, 7, 25, 26)]          # kv heads 1 and 6
    ref = sc.oracle_outputs(case, pairs)
    for dynamic in (False, True):
        out, out32 = _run_like_bench(case, dynamic)
        _check(case, out, out32, pairs, ref)

"""CUDA path vs the oracle, through the C ABI (liboscar.so).

Bars: codes / scale / zero / rotated rows / q_rot / merge bit-exact; attention
outputs (fp32, before the bf16 rounding) within relative L2 1e-3 and
max |err| <= 2e-3 * max |o_ref|; the bf16 output equal to the round-to-nearest-
even of the fp32 one.
"""
import math

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


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("clip", [1.0, 0.96, 0.92])
def test_quantize_rotated_bit_exact(group, clip):
    x = syn.rotated_rows(7, 300)
    x[3, :] = 0.0
    x[4, ::3] = -0.0
    x[5] = np.float32(np.round(x[5] * 4) / 4)             # many values on a coarse grid: exact ties
    L = ob.Layout(1, 1, 16, group)
    xd = torch.from_numpy(x).cuda()
    codes = torch.empty((300, D // 4), dtype=torch.uint8, device="cuda")
    scale = torch.empty((300, D // group), dtype=torch.bfloat16, device="cuda")
    zero = torch.empty_like(scale)
    ob.oscar_quantize_rotated(L, xd, clip, codes, scale, zero)
    torch.cuda.synchronize()
    p, z, s = oracle.quantize_rows(x, group, clip)
    assert np.array_equal(codes.cpu().numpy(), p)
    assert np.array_equal(bf16_bits(scale), s)
    assert np.array_equal(bf16_bits(zero), z)


def test_rotate_q_bit_exact():
    case = sc.make_case(n_kv=2, gqa=4, seq=(500, 300))
    sc.upload(case, demote_history=False)
    L = case.layout
    q_rot = torch.empty((2, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    ob.oscar_rotate_q(L, case.dev["q"], case.dev["RK"], q_rot)
    torch.cuda.synchronize()
    qb = bf16_bits(case.q)
    got = q_rot.cpu().numpy()
    for b in range(2):
        for hq in range(L.n_q_heads):
            ref = oracle.rotate_f32(qb[b, hq][None], case.RK[hq // L.gqa])[0]
            assert np.array_equal(got[b, hq], ref)


@pytest.mark.parametrize("group,page_size", [(128, 16), (32, 64)])
def test_demote_bit_exact(group, page_size):
    case = sc.make_case(n_kv=2, gqa=4, page_size=page_size, group=group, seq=(1024, 777))
    dev = sc.upload(case)
    torch.cuda.synchronize()
    rot = dev["rotated"].cpu().numpy()
    req = dev["demote_req"].cpu().numpy()
    pos = dev["demote_pos"].cpu().numpy()
    L = case.layout
    for b in range(2):
        he = int(case.hist_end[b])
        sel = np.flatnonzero(req == b)
        assert list(pos[sel]) == list(range(L.sink, he))
        for h in range(L.n_kv_heads):
            kb = bf16_bits(case.K[b][L.sink:he, h])
            vb = bf16_bits(case.V[b][L.sink:he, h])
            rk, pk, zk, sk = oracle.demote_rows(kb, case.RK[h], group, oracle.C_K)
            rv, pv, zv, sv = oracle.demote_rows(vb, case.RV[h], group, oracle.C_V)
            assert np.array_equal(rot[sel, 0, h], rk)
            assert np.array_equal(rot[sel, 1, h], rv)
            ck, cv, gzk, gsk, gzv, gsv = sc.gather_int2(case, b, h)
            assert np.array_equal(ck[L.sink:he], pk)
            assert np.array_equal(cv[L.sink:he], pv)
            assert np.array_equal(gzk[L.sink:he], zk) and np.array_equal(gsk[L.sink:he], sk)
            assert np.array_equal(gzv[L.sink:he], zv) and np.array_equal(gsv[L.sink:he], sv)


def _check_outputs(case, out, out32, lse, pairs=None):
    ref = sc.oracle_outputs(case, pairs)
    o32 = out32.cpu().numpy()
    ob16 = bf16_bits(out)
    lse_g = lse.cpu().numpy()
    got = np.stack([o32[b, hq] for (b, hq) in ref])
    exp = np.stack([ref[k][0] for k in ref])
    ok, r, m = sc.tolerance_ok(got, exp)
    assert ok, f"rel-L2 {r:.3e}, max-abs frac {m:.3e}"
    for (b, hq), (o, l) in ref.items():
        one_ok, r1, m1 = sc.tolerance_ok(o32[b, hq], o)
        assert one_ok, f"head {(b, hq)}: rel-L2 {r1:.3e}, max-abs {m1:.3e}"
        assert abs(lse_g[b, hq] - l) <= 1e-4 * max(1.0, abs(l))
        assert np.array_equal(ob16[b, hq], oracle.f32_to_bf16(o32[b, hq]))


@pytest.mark.parametrize("n_splits", [1, 3, 16])
def test_decode_tiny_parity(n_splits):
    """1 layer, 8 q / 2 kv heads, 1,024 tokens = 64 sink + 704 history + 256 recent, 16-token pages."""
    case = sc.make_case(n_kv=2, gqa=4, page_size=16, seq=(1024,))
    sc.upload(case)
    out, out32, lse, _ = sc.run_decode(case, n_splits)
    _check_outputs(case, out, out32, lse)
    assert ob.oscar_get_device_status() == 0


def test_partials_per_split_match_oracle():
    """Each split's (m, l, acc) against the oracle's fp64 partial over the documented tile-balanced range."""
    S = 5
    case = sc.make_case(n_kv=2, gqa=4, page_size=16, seq=(1024, 613))
    sc.upload(case)
    _, _, _, part = sc.run_decode(case, S)
    L = case.layout
    m, l, acc = part.m.cpu().numpy(), part.l.cpu().numpy(), part.acc.cpu().numpy()
    qb = bf16_bits(case.q)
    for b, T in enumerate(case.seq):
        he = int(case.hist_end[b])
        first = L.sink // 16
        n = -(-he // 16) - first
        for h in range(L.n_kv_heads):
            cache = sc.oracle_head_cache(case, b, h)
            for g in range(L.gqa):
                hq = h * L.gqa + g
                for s in range(S + 1):
                    if s < S:
                        lo = max(L.sink, (first + s * n // S) * 16)
                        hi = min(he, (first + (s + 1) * n // S) * 16)
                        ranges = [(lo, hi)] if lo < hi else []
                    else:
                        ranges = [(0, L.sink), (he, T)]
                    rm, rl, racc = oracle.partial(qb[b, hq], case.RK[h], cache, case.sm_scale, ranges)
                    if rl == 0.0:
                        assert m[b, hq, s] == -np.inf and l[b, hq, s] == 0.0 and not acc[b, hq, s].any()
                        continue
                    assert abs(m[b, hq, s] - rm) <= 1e-4 * max(1.0, abs(rm))
                    assert abs(l[b, hq, s] - rl) <= 1e-4 * rl
                    err = np.linalg.norm(acc[b, hq, s] - racc) / np.linalg.norm(racc)
                    assert err <= 1e-4, (b, hq, s, err)


@pytest.mark.parametrize("S,empty", [(1, ()), (7, (2, 3)), (64, (0, 63)), (5, (5,))])
def test_merge_bit_exact(S, empty):
    """Equal partials -> equal bits: the merge against the oracle's ordered fp32 fold."""
    L = ob.Layout(2, 4, 16)
    B = 2
    part = ob.Partials.empty(L, B, S)
    m = np.empty((B, L.n_q_heads, S + 1), np.float32)
    l = np.empty_like(m)
    acc = np.empty((B, L.n_q_heads, S + 1, D), np.float32)
    for b in range(B):
        for hq in range(L.n_q_heads):
            m[b, hq], l[b, hq], acc[b, hq] = syn.split_partials(1000 * b + hq + 17 * S, S, D, empty)
    part.m.copy_(torch.from_numpy(m))
    part.l.copy_(torch.from_numpy(l))
    part.acc.copy_(torch.from_numpy(acc))
    rng = np.random.default_rng(S)
    RV = np.stack([np.linalg.qr(rng.normal(size=(D, D)))[0] for _ in range(2)]).astype(np.float32)
    out = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    ob.oscar_merge(L, part, torch.from_numpy(RV).cuda(), out, out32)
    torch.cuda.synchronize()
    o32, ob16 = out32.cpu().numpy(), bf16_bits(out)
    for b in range(B):
        for hq in range(L.n_q_heads):
            r32, rb = oracle.merge_f32(m[b, hq], l[b, hq], acc[b, hq], RV[hq // L.gqa])
            assert np.array_equal(o32[b, hq].view(np.uint32), r32.view(np.uint32)), (b, hq)
            assert np.array_equal(ob16[b, hq], rb)


@pytest.mark.parametrize("n_kv", [2, 8])          # 8 kv heads: the tensor-map copy path
@pytest.mark.parametrize("seq,hist,gqa,ps,group,S", [
    ((1024, 700, 333), None, 4, 16, 128, 4),          # ragged batch, short request with little history
    ((40,), None, 4, 16, 128, 2),                      # shorter than the sink: no history at all
    ((500,), (64,), 4, 16, 128, 3),                    # history end at the sink: all BF16
    ((2000,), None, 8, 64, 32, 40),                    # more splits than history pages, group 32, G=8
    ((1500,), None, 1, 32, 64, 6),                     # G=1, group 64
    ((1100,), (843,), 2, 16, 128, 5),                  # history end mid-page, one demoted row still BF16
])
def test_decode_edge_cases(seq, hist, gqa, ps, group, S, n_kv):
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq, hist_end=hist)
    sc.upload(case)
    out, out32, lse, _ = sc.run_decode(case, S)
    _check_outputs(case, out, out32, lse)
    assert ob.oscar_get_device_status() == 0


def test_decode_cuda_core_kernel_three_kv_heads():
    """3 kv heads (not a divisor of 8): the CUDA-core split kernel serves this shape."""
    case = sc.make_case(n_kv=3, gqa=2, page_size=16, seq=(900, 500))
    sc.upload(case)
    out, out32, lse, _ = sc.run_decode(case, 4)
    _check_outputs(case, out, out32, lse)
    assert ob.oscar_get_device_status() == 0


def test_decode_qwen3_8b_layer_shape():
    """One layer of the Qwen3-8B shape (32 q / 8 kv heads, 64-token pages) over a ragged batch
    spanning many splits and a ragged last page."""
    case = sc.make_case(n_kv=8, gqa=4, page_size=64, seq=(6000, 3333, 1234))
    sc.upload(case)
    out, out32, lse, _ = sc.run_decode(case, 24)
    _check_outputs(case, out, out32, lse)


def test_halves_on_two_streams_equal_the_combined_call():
    """History and window halves launched on two streams write exactly what the combined call writes."""
    case = sc.make_case(n_kv=8, gqa=4, page_size=64, seq=(3000, 1800))
    sc.upload(case)
    L, dev = case.layout, case.dev
    _, _, _, ref = sc.run_decode(case, 6)
    part = ob.Partials.empty(L, 2, 6)
    part.m.fill_(float("nan"))
    part.acc.fill_(float("nan"))
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    with torch.cuda.stream(side):
        ob.oscar_decode_attention_window(L, dev["q"], dev["bf16"], dev["bf16_table"], dev["seq_len"],
                                         dev["hist_end"], case.sm_scale, part, stream=side)
    ob.oscar_decode_attention_history(L, dev["q_rot"], dev["int2"], dev["int2_table"], dev["seq_len"],
                                      dev["hist_end"], case.sm_scale, part)
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert torch.equal(part.m, ref.m) and torch.equal(part.l, ref.l) and torch.equal(part.acc, ref.acc)


def _layers_back_to_back(case, qs, n_splits, sync=True):
    """rotate_q -> decode_attention -> merge for several queries in one stream, sharing q_rot and
    the partials buffer between them (so a launch that overlapped too far would change bits)."""
    L, dev = case.layout, case.dev
    B = len(case.seq)
    q_rot = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    part = ob.Partials.empty(L, B, n_splits)
    outs = []
    for q in qs:
        o32 = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
        ob.oscar_rotate_q(L, q, dev["RK"], q_rot)
        ob.oscar_decode_attention(L, q, q_rot, dev["bf16"], dev["bf16_table"], dev["int2"], dev["int2_table"],
                                  dev["seq_len"], dev["hist_end"], case.sm_scale, part)
        ob.oscar_merge(L, part, dev["RV"], None, o32, None)
        outs.append(o32)
    if sync:
        torch.cuda.synchronize()
    return outs


def test_launch_overlap_gives_identical_bits():
    """Programmatic dependent launch between the decode kernels changes no output bit, eagerly
    and inside a CUDA graph."""
    case = sc.make_case(n_kv=8, gqa=4, page_size=64, seq=(5000, 2100))
    sc.upload(case)
    gen = torch.Generator(device="cpu").manual_seed(7)
    qs = [torch.randn(case.dev["q"].shape, generator=gen).to(torch.bfloat16).cuda() for _ in range(5)]
    assert not ob.oscar_get_launch_overlap()
    ref = _layers_back_to_back(case, qs, 20)
    try:
        ob.oscar_set_launch_overlap(True)
        assert ob.oscar_get_launch_overlap()
        got = _layers_back_to_back(case, qs, 20)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            holder = [None]
            holder[0] = _layers_back_to_back(case, qs, 20, sync=False)
        g.replay()
        torch.cuda.synchronize()
        got_graph = holder[0]
    finally:
        ob.oscar_set_launch_overlap(False)
    for r, a, b in zip(ref, got, got_graph):
        assert torch.equal(r, a) and torch.equal(r, b)
    assert ob.oscar_get_device_status() == 0


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq,S", [
    (8, 4, 64, 128, (3000, 1700), 6),     # the benchmark's shape, clusters of 8: one kv head per CTA
    (8, 8, 64, 32, (2500,), 5),            # GQA 8, group 32
    (4, 2, 32, 64, (1800, 900), 4),
    (2, 4, 16, 128, (1200,), 3),            # more CTAs per cluster than kv heads
    (1, 8, 16, 128, (900,), 2),             # R_K staged in 16 KB chunks
    (1, 1, 16, 32, (700,), 2),
])
def test_fused_rotation_matches_rotate_then_decode(n_kv, gqa, ps, group, seq, S):
    """oscar_decode_attention_fused writes the partials of oscar_rotate_q + oscar_decode_attention
    up to the fp32 rounding of q . R_K: the fused rotation sums the same products in another order
    (eight row blocks, then their sum), so the partials agree to a few fp32 ulps of the logits."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq)
    sc.upload(case)
    L, dev = case.layout, case.dev
    _, _, _, ref = sc.run_decode(case, S)
    part = ob.Partials.empty(L, len(seq), S)
    part.m.fill_(float("nan"))
    part.l.fill_(float("nan"))
    part.acc.fill_(float("nan"))
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part)
    torch.cuda.synchronize()
    _assert_partials_close(part, ref)
    assert ob.oscar_get_device_status() == 0


def _assert_partials_close(part, ref, rtol=2e-5):
    """Equal empty slots, and (m, l, acc) within rtol of the reference in each query head's own
    scale: the partials of one slot share the weights 2^(logit - m), so a logit that moves by a
    few fp32 ulps moves l and acc by about that much times |logit|."""
    empty = ~torch.isfinite(ref.m)
    assert torch.equal(empty, ~torch.isfinite(part.m))
    mr, mp = ref.m[~empty], part.m[~empty]
    assert torch.allclose(mp, mr, rtol=0, atol=rtol * max(1.0, float(mr.abs().max())))
    lr, lp = ref.l[~empty], part.l[~empty]
    assert torch.allclose(lp, lr, rtol=rtol * max(1.0, float(mr.abs().max())), atol=0)
    ar, ap = ref.acc[~empty], part.acc[~empty]
    assert torch.allclose(ap, ar, rtol=0, atol=rtol * max(1.0, float(mr.abs().max())) * float(ar.abs().max()))


def _pool_bytes(i2):
    return [t.clone() for t in (i2.codes_k, i2.codes_v, i2.scale_k, i2.zero_k, i2.scale_v, i2.zero_v)]


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq,S", [
    (8, 4, 64, 128, (3000, 1700), 6),
    (8, 8, 16, 32, (1400,), 3),
    (4, 2, 32, 64, (1800, 900), 4),
    (1, 4, 16, 128, (900,), 2),
])
def test_fused_demotion_matches_oscar_demote(n_kv, gqa, ps, group, seq, S):
    """The per-step demotion done by the decode launch writes the bytes oscar_demote writes, and
    leaves that step's partials unchanged; with dynamic history units (the demotion then runs in
    the first history CTAs) it writes the same bytes."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq)
    sc.upload(case)
    L, dev = case.layout, case.dev
    B = len(seq)
    pos = dev["hist_end"].clone()                      # the token that left the recent window
    before = _pool_bytes(dev["int2"])
    # reference: oscar_demote of the same positions
    ob.oscar_demote(L, dev["bf16"], dev["bf16_table"], dev["int2"], dev["int2_table"],
                    torch.arange(B, dtype=torch.int32, device="cuda"), pos, dev["RK"], dev["RV"],
                    oracle.C_K, oracle.C_V)
    torch.cuda.synchronize()
    want = _pool_bytes(dev["int2"])
    for t, b0 in zip((dev["int2"].codes_k, dev["int2"].codes_v, dev["int2"].scale_k, dev["int2"].zero_k,
                      dev["int2"].scale_v, dev["int2"].zero_v), before):
        t.copy_(b0)
    ref = ob.Partials.empty(L, B, S)
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, ref)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(_pool_bytes(dev["int2"]), before))
    part = ob.Partials.empty(L, B, S)
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part,
                                    demote_pos=pos, R_V=dev["RV"], c_K=oracle.C_K, c_V=oracle.C_V)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(_pool_bytes(dev["int2"]), want))
    assert torch.equal(part.m, ref.m) and torch.equal(part.l, ref.l) and torch.equal(part.acc, ref.acc)
    # dynamic history units: the same bytes
    for t, b0 in zip((dev["int2"].codes_k, dev["int2"].codes_v, dev["int2"].scale_k, dev["int2"].zero_k,
                      dev["int2"].scale_v, dev["int2"].zero_v), before):
        t.copy_(b0)
    tiles = torch.zeros(2 * B, dtype=torch.int32, device="cuda")
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale,
                                    ob.Partials.empty(L, B, S), demote_pos=pos, R_V=dev["RV"], c_K=oracle.C_K,
                                    c_V=oracle.C_V, tile_counters=tiles)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(_pool_bytes(dev["int2"]), want))
    assert not tiles.any()
    assert ob.oscar_get_device_status() == 0


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq,S", [
    (8, 4, 64, 128, (3000, 1700), 6),     # the benchmark's shape
    (8, 8, 16, 32, (1400,), 3),            # GQA 8, group 32
    (4, 2, 32, 64, (1800, 900), 4),
    (2, 4, 16, 128, (1200, 300), 3),        # a request with no history
    (1, 1, 16, 128, (700,), 2),             # one kv head
])
def test_fused_merge_matches_oscar_merge(n_kv, gqa, ps, group, seq, S):
    """The merge launched by the fused call, started per request on the decode clusters' arrival
    counts, gives oscar_merge's bits (out, out_f32, lse), leaves the counters at zero, and repeated
    or graph-captured calls (back to back on the same partials) with launch overlap agree."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq)
    sc.upload(case)
    L, dev = case.layout, case.dev
    B, Hq = len(seq), L.n_q_heads
    part = ob.Partials.empty(L, B, S)
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part)
    ref = [torch.empty((B, Hq, D), dtype=t, device="cuda") for t in (torch.bfloat16, torch.float32)]
    ref_lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ob.oscar_merge(L, part, dev["RV"], ref[0], ref[1], ref_lse)
    counters = torch.zeros(2 * B, dtype=torch.int32, device="cuda")

    def fused(p2, outs):
        ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                        dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, p2,
                                        R_V=dev["RV"], out=outs[0], out_f32=outs[1], lse=outs[2],
                                        merge_counters=counters)

    runs = []
    for _ in range(3):
        outs = (torch.full_like(ref[0], float("nan")), torch.full_like(ref[1], float("nan")),
                torch.full_like(ref_lse, float("nan")))
        fused(ob.Partials.empty(L, B, S), outs)
        runs.append(outs)
    try:
        ob.oscar_set_launch_overlap(True)
        outs_g = (torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref_lse))
        p_g = ob.Partials.empty(L, B, S)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fused(p_g, outs_g)
            fused(p_g, outs_g)
        g.replay()
        g.replay()
    finally:
        ob.oscar_set_launch_overlap(False)
    torch.cuda.synchronize()
    runs.append(outs_g)
    for o in runs:
        assert torch.equal(o[0], ref[0]) and torch.equal(o[1], ref[1]) and torch.equal(o[2], ref_lse)
    assert not counters.any()
    assert ob.oscar_get_device_status() == 0


def test_fused_demotion_refuses_a_position_inside_the_history():
    case = sc.make_case(n_kv=8, gqa=4, page_size=64, seq=(1500,))
    sc.upload(case)
    L, dev = case.layout, case.dev
    before = _pool_bytes(dev["int2"])
    pos = dev["hist_end"] - 10                          # still read from INT2 by this launch
    part = ob.Partials.empty(L, 1, 2)
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part,
                                    demote_pos=pos, R_V=dev["RV"], c_K=oracle.C_K, c_V=oracle.C_V)
    torch.cuda.synchronize()
    assert ob.oscar_get_device_status() & 0x4
    assert all(torch.equal(a, b) for a, b in zip(_pool_bytes(dev["int2"]), before))


def test_fused_rotation_rejects_other_head_counts():
    case = sc.make_case(n_kv=3, gqa=2, page_size=16, seq=(400,))
    sc.upload(case)
    L, dev = case.layout, case.dev
    part = ob.Partials.empty(L, 1, 2)
    with pytest.raises(ob.OscarError, match="kv heads"):
        ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                        dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part)


@pytest.mark.parametrize("n_kv,gqa,ps,seq,S", [
    (2, 4, 16, (1024, 555), 9),         # cp.async path
    (8, 4, 64, (3000, 1700), 12),       # 8 kv heads: tensor-map boxes, one tile of every head per stage
    (8, 8, 16, (1500,), 5),
])
def test_bf16_full_cache_parity(n_kv, gqa, ps, seq, S):
    """The all-BF16 comparison kernel: oracle with no history region (sink = h_end = 0)."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, seq=seq)
    L = case.layout
    dev = sc.upload(case, demote_history=False)
    part = ob.Partials.empty(L, len(seq), S)
    ob.oscar_bf16_decode_attention(L, dev["q"], dev["stage"], dev["stage_table"], dev["seq_len"], case.sm_scale, part)
    out32 = torch.empty((len(seq), L.n_q_heads, D), dtype=torch.float32, device="cuda")
    ob.oscar_merge(L, part, None, None, out32)
    torch.cuda.synchronize()
    assert ob.oscar_get_device_status() == 0
    qb = bf16_bits(case.q)
    got, exp = [], []
    for b, T in enumerate(case.seq):
        for h in range(L.n_kv_heads):
            kb, vb = bf16_bits(case.K[b][:, h]), bf16_bits(case.V[b][:, h])
            z8 = np.zeros((T, D // 4), np.uint8)
            z16 = np.zeros((T, 1), np.uint16)
            cache = oracle.HeadCache(kb, vb, z8, z8, z16, z16, z16, z16, 0, 0, 128)
            I = np.eye(D, dtype=np.float32)
            for g in range(L.gqa):
                o, _ = oracle.attend_head(qb[b, h * L.gqa + g], I, I, cache, case.sm_scale)
                got.append(out32.cpu().numpy()[b, h * L.gqa + g])
                exp.append(o)
    ok, r, m = sc.tolerance_ok(np.stack(got), np.stack(exp))
    assert ok, (r, m)


def test_layouts_sharing_a_kernel_run_in_any_order():
    """Layouts served by one kernel instance with different shared-memory sizes (4, 1 and 2 kv
    heads at GQA 4): running a smaller one must not break a larger one run before it."""
    cases = [sc.make_case(n_kv=h, gqa=4, page_size=16, seq=(700,)) for h in (4, 1, 2)]
    for c in cases:
        sc.upload(c)
    for c in cases + cases[:1]:
        out, out32, lse, _ = sc.run_decode(c, 3)
        _check_outputs(c, out, out32, lse)
    assert ob.oscar_get_device_status() == 0


def test_bad_page_id_is_flagged_not_faulted():
    case = sc.make_case(n_kv=2, gqa=4, page_size=16, seq=(1024,))
    dev = sc.upload(case)
    assert ob.oscar_get_device_status() == 0
    bad = dev["int2_table"].clone()
    bad[0, 10] = case.dev["int2"].n_pages + 5
    dev["int2_table"] = bad
    sc.run_decode(case, 4)
    assert ob.oscar_get_device_status() & 0x1
    assert ob.oscar_get_device_status() == 0                     # read clears it


def test_host_validation_errors():
    L = ob.Layout(2, 3, 16)                                       # gqa 3 unsupported
    x = torch.zeros((4, D), dtype=torch.float32, device="cuda")
    c = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros((4, 1), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ob.OscarError, match="gqa"):
        ob.oscar_quantize_rotated(L, x, 0.96, c, s, s)
    with pytest.raises(ob.OscarError, match="clip"):
        ob.oscar_quantize_rotated(ob.Layout(2, 4, 16), x, 0.0, c, s, s)


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq,S", [
    (8, 4, 64, 128, (3000, 1700), 6),     # the benchmark's layout
    (2, 4, 16, 32, (1200, 300), 3),        # group 32, a request with no history
    (8, 8, 16, 64, (1400,), 4),            # GQA 8, group 64
    (1, 1, 32, 128, (900, 2100), 2),       # one kv head (no tensor maps)
])
def test_dynamic_tile_scheduling(n_kv, gqa, ps, group, seq, S):
    """History CTAs taking 64-token units from a shared per-request counter: the merged output
    meets the bar against the oracle and agrees with the fixed splits' up to fp32 rounding order;
    eager, repeated and graph-captured (launch overlap) calls leave the counters at zero."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq)
    sc.upload(case)
    L, dev = case.layout, case.dev
    B, Hq = len(seq), L.n_q_heads
    tiles = torch.zeros(2 * B, dtype=torch.int32, device="cuda")

    def run(p2, outs, dyn):
        ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                        dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, p2,
                                        R_V=dev["RV"], out=outs[0], out_f32=outs[1], lse=outs[2],
                                        tile_counters=tiles if dyn else None)

    def fresh():
        return (torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda"),
                torch.empty((B, Hq, D), dtype=torch.float32, device="cuda"),
                torch.empty((B, Hq), dtype=torch.float32, device="cuda"))
    fixed = fresh()
    run(ob.Partials.empty(L, B, S), fixed, False)
    runs = []
    for _ in range(3):
        o = fresh()
        run(ob.Partials.empty(L, B, S), o, True)
        runs.append(o)
    try:
        ob.oscar_set_launch_overlap(True)
        og = fresh()
        pg = ob.Partials.empty(L, B, S)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(pg, og, True)
            run(pg, og, True)
        g.replay()
        g.replay()
    finally:
        ob.oscar_set_launch_overlap(False)
    torch.cuda.synchronize()
    runs.append(og)
    assert not tiles.any()
    assert ob.oscar_get_device_status() == 0
    ref = sc.oracle_outputs(case)
    f32 = fixed[1].cpu().numpy()
    for o in runs:
        o32 = o[1].cpu().numpy()
        assert np.array_equal(bf16_bits(o[0]), oracle.f32_to_bf16(o32))
        assert np.allclose(o32, f32, rtol=1e-5, atol=1e-5 * np.abs(f32).max())
        for (b, hq), (oref, lref) in ref.items():
            ok, r, m = sc.tolerance_ok(o32[b, hq], oref)
            assert ok, ((b, hq), r, m)


@pytest.mark.parametrize("n_kv,gqa,ps,group,vf,qf", [
    (8, 4, 64, 128, 50.0, 1.0),       # value scales ~1e3 (P * scale_v would leave the f16 range unscaled)
    (8, 4, 64, 128, 1e-6, 1.0),       # value scales ~1e-5 (f16 subnormals unscaled)
    (8, 4, 64, 128, 1.0, 300.0),      # queries ~1e3: q_rot / code factor beyond the f16 range unscaled
    (8, 8, 16, 32, 50.0, 1.0),        # groups of 32 (group-pure loop, tensor-map copies)
    (2, 4, 16, 128, 1e-6, 300.0),     # 2 kv heads (cp.async copies)
    (4, 2, 32, 64, 50.0, 1.0),
])
def test_value_and_query_scale_range(n_kv, gqa, ps, group, vf, qf):
    """Values and queries far from the synthetic data's magnitudes: the decode kernel normalises
    the value scales by a running power-of-two bound and the rotated queries by a power of two
    per kv head, so its f16 split operands stay in range; outputs against the oracle (both the
    rotate + decode + merge calls and the fused launch)."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=(2000, 900))
    case.V = [(v.float() * vf).to(torch.bfloat16) for v in case.V]
    case.q = (case.q.float() * qf).to(torch.bfloat16)
    sc.upload(case)
    out, out32, lse, _ = sc.run_decode(case, 5)
    assert ob.oscar_get_device_status() == 0
    _check_outputs(case, out, out32, lse)
    L, dev = case.layout, case.dev
    part = ob.Partials.empty(L, 2, 5)
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part)
    ob.oscar_merge(L, part, dev["RV"], out, out32, lse)
    torch.cuda.synchronize()
    assert ob.oscar_get_device_status() == 0
    _check_outputs(case, out, out32, lse)

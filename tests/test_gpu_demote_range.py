"""Bulk demotion on the tensor cores (oscar_demote_range) vs the oracle, through the C ABI.

Bars: each rotated row within 2^-14 * ||x||_2 of the oracle's fp64 product x . R (the
tensor-core product x . R_hi + x . R_lo carries R to about 16 bits); codes, scale and zero
bit-exact against the oracle's quantizer applied to the kernel's own rotated rows; every INT2
slot and rotated-row slot outside the ranges left as it was.
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
SENTINEL_CODE = 0xA5
SENTINEL_BF16 = 0x7FC1


def _setup(L, seqs, K, V, seed):
    """Pools with shuffled physical pages (plus spare ones), BF16 rows placed by the page table,
    the INT2 pool and the rotated-row buffer filled with sentinels."""
    rng = np.random.default_rng(seed)
    ps, B = L.page_size, len(seqs)
    max_pages = max((T + ps - 1) // ps for T in seqs)
    n_pages = B * max_pages + 3
    bt = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    it = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    bf = ob.Bf16Pool.empty(L, n_pages)
    bf.k.normal_()
    bf.v.normal_()
    for b, T in enumerate(seqs):
        pos = np.arange(T)
        pg = torch.from_numpy(bt[b, pos // ps].astype(np.int64)).cuda()
        sl = torch.from_numpy((pos % ps).astype(np.int64)).cuda()
        bf.k[pg, sl] = K[b].cuda()
        bf.v[pg, sl] = V[b].cuda()
    i2 = ob.Int2Pool.empty(L, n_pages)
    for t in (i2.codes_k, i2.codes_v):
        t.fill_(SENTINEL_CODE)
    for t in (i2.scale_k, i2.zero_k, i2.scale_v, i2.zero_v):
        t.view(torch.int16).fill_(SENTINEL_BF16)
    rot = torch.full((n_pages, ps, 2, L.n_kv_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    return bf, i2, rot, torch.from_numpy(bt).cuda(), torch.from_numpy(it).cuda(), it


def _run(L, bf, i2, rot, btab, itab, ranges, RK, RV, cK, cV):
    pb = torch.tensor([r[0] for r in ranges], dtype=torch.int32, device="cuda")
    pe = torch.tensor([r[1] for r in ranges], dtype=torch.int32, device="cuda")
    ob.oscar_demote_range(L, bf, btab, i2, itab, pb, pe, torch.from_numpy(RK).cuda(), torch.from_numpy(RV).cuda(),
                          cK, cV, rotated_out=rot)
    torch.cuda.synchronize()


def _check(L, K, V, ranges, it, i2, rot, RK, RV, cK, cV):
    ps, H = L.page_size, L.n_kv_heads
    g = L.group
    codes = (i2.codes_k.cpu().numpy(), i2.codes_v.cpu().numpy())
    scale = (bf16_bits(i2.scale_k), bf16_bits(i2.scale_v))
    zero = (bf16_bits(i2.zero_k), bf16_bits(i2.zero_v))
    rr = rot.cpu().numpy()
    written = np.zeros(rr.shape[:2], dtype=bool)
    for b, (lo, hi) in enumerate(ranges):
        if hi <= lo:
            continue
        pos = np.arange(lo, hi)
        pg, sl = it[b, pos // ps], pos % ps
        written[pg, sl] = True
        for kind, (X, R, c) in enumerate(((K[b], RK, cK), (V[b], RV, cV))):
            for h in range(H):
                xb = bf16_bits(X[lo:hi, h])
                got = rr[pg, sl, kind, h]
                ref = oracle.rotate_f64(xb, R[h])
                norm = np.linalg.norm(oracle.bf16_to_f64(xb), axis=1)
                err = np.abs(got.astype(np.float64) - ref).max(axis=1)
                assert np.all(err <= 2.0 ** -14 * norm + 1e-30), (b, kind, h, float((err / norm).max()))
                p, z, s = oracle.quantize_rows(got, g, c)
                assert np.array_equal(codes[kind][pg, sl, h], p), (b, kind, h)
                assert np.array_equal(zero[kind][pg, sl, h], z), (b, kind, h)
                assert np.array_equal(scale[kind][pg, sl, h], s), (b, kind, h)
    # nothing outside the ranges was written
    for kind in (0, 1):
        assert np.all(codes[kind][~written] == SENTINEL_CODE)
        assert np.all(scale[kind][~written] == SENTINEL_BF16)
        assert np.all(zero[kind][~written] == SENTINEL_BF16)
    assert np.all(np.isnan(rr[~written]))
    assert ob.oscar_get_device_status() == 0


@pytest.mark.parametrize("n_kv,ps,group,seqs,ranges", [
    (8, 64, 128, (3000, 1800), [(64, 2744), (64, 1544)]),            # the benchmark's layout, ragged ends
    (2, 16, 32, (1400, 300, 500), [(100, 1333), (0, 0), (64, 200)]),  # 8 pages per tile, empty range
    (4, 32, 64, (1000,), [(64, 1000)]),
    (1, 32, 128, (700, 10), [(64, 700), (5, 6)]),                      # one kv head, a one-position range
    (2, 16, 64, (900,), [(200, 900)]),
])
def test_demote_range_matches_oracle(n_kv, ps, group, seqs, ranges):
    L = ob.Layout(n_kv, 2, ps, group)
    prof, RK, RV = sc.oracle_rotations(0, 0, n_kv, 2)
    K, V = [], []
    for b, T in enumerate(seqs):
        k, v = syn.kv_rows(0, 0, b, 0, T, prof)
        K.append(k)
        V.append(v)
    bf, i2, rot, btab, itab, it = _setup(L, seqs, K, V, seed=len(seqs) + ps)
    _run(L, bf, i2, rot, btab, itab, ranges, RK, RV, oracle.C_K, oracle.C_V)
    _check(L, K, V, ranges, it, i2, rot, RK, RV, oracle.C_K, oracle.C_V)


@pytest.mark.parametrize("group", [32, 128])
def test_demote_range_half_step_ties(group):
    """Identity rotations and clip 1 make the rotated rows the inputs themselves: every group holds
    0 and 4.5 (scale 1.5, zero 0) and the values 0.75, 2.25, 3.75 whose quotients are exactly
    0.5, 1.5, 2.5, where the product by the rounded reciprocal 1/1.5 is not exact; ties round to
    even (codes 0, 2, 2)."""
    n_kv, ps, T = 2, 64, 640
    L = ob.Layout(n_kv, 1, ps, group)
    rng = np.random.default_rng(5)
    grid = np.arange(0, 4.5 + 1e-9, 2.0 ** -5, dtype=np.float32)          # bf16-exact values in [0, 4.5]
    X = []
    for _ in range(2):
        x = rng.choice(grid, size=(T, n_kv, D)).astype(np.float32)
        for g0 in range(0, D, group):
            x[..., g0:g0 + 8] = np.array([0.0, 4.5, 0.75, 2.25, 3.75, -0.0, 1.5, 3.0], np.float32)
        X.append(torch.from_numpy(x).bfloat16())
    eye = np.stack([np.eye(D, dtype=np.float32)] * n_kv)
    bf, i2, rot, btab, itab, it = _setup(L, (T,), [X[0]], [X[1]], seed=11)
    _run(L, bf, i2, rot, btab, itab, [(64, T)], eye, eye, 1.0, 1.0)
    _check(L, [X[0]], [X[1]], [(64, T)], it, i2, rot, eye, eye, 1.0, 1.0)
    pos = np.arange(64, T)
    codes = i2.codes_k.cpu().numpy()[it[0, pos // ps], pos % ps]           # [n, H, 32]
    for g0 in range(0, D, group):
        unpacked = np.stack([(codes[..., (g0 + i) // 4] >> (2 * ((g0 + i) % 4))) & 3 for i in range(8)], -1)
        assert np.all(unpacked == np.array([0, 3, 0, 2, 2, 0, 1, 2]))


def test_demote_range_fullsize_qwen3_8b_100k():
    """One layer of the benchmark's workload: the whole history [64, 99,744) of a 100,000-token
    request, 8 kv heads, K and V; 4,000 sampled (position, head, K/V) rows checked."""
    w = syn.WORKLOADS["qwen3_8b_100k"]
    L = ob.Layout(w.n_kv_heads, w.gqa, w.page_size, w.group)
    T, ps = w.context, w.page_size
    he = T - w.recent
    prof, RK, RV = sc.oracle_rotations(w.seed, 0, w.n_kv_heads, w.gqa)
    k, v = syn.kv_rows(w.seed, 0, 0, 0, T, prof, device="cuda")
    n_log = (T + ps - 1) // ps
    table = torch.arange(n_log, dtype=torch.int32, device="cuda").view(1, n_log)
    bf = ob.Bf16Pool.empty(L, n_log)
    bf.k.view(-1, w.n_kv_heads, D)[:T] = k
    bf.v.view(-1, w.n_kv_heads, D)[:T] = v
    i2 = ob.Int2Pool.empty(L, n_log)
    rot = torch.empty((n_log, ps, 2, w.n_kv_heads, D), dtype=torch.float32, device="cuda")
    _run(L, bf, i2, rot, table, table, [(w.sink, he)], RK, RV, oracle.C_K, oracle.C_V)
    assert ob.oscar_get_device_status() == 0
    rng = np.random.default_rng(3)
    pos = np.concatenate([[w.sink, he - 1], rng.integers(w.sink, he, 3998)])
    heads = rng.integers(0, w.n_kv_heads, pos.size)
    kinds = rng.integers(0, 2, pos.size)
    rr = rot.view(-1, 2, w.n_kv_heads, D)[torch.from_numpy(pos).cuda()].cpu().numpy()
    xs = (k[torch.from_numpy(pos).cuda()].cpu(), v[torch.from_numpy(pos).cuda()].cpu())
    codes = (i2.codes_k.view(-1, w.n_kv_heads, D // 4)[torch.from_numpy(pos).cuda()].cpu().numpy(),
             i2.codes_v.view(-1, w.n_kv_heads, D // 4)[torch.from_numpy(pos).cuda()].cpu().numpy())
    scales = (bf16_bits(i2.scale_k.view(-1, w.n_kv_heads, 1)[torch.from_numpy(pos).cuda()]),
              bf16_bits(i2.scale_v.view(-1, w.n_kv_heads, 1)[torch.from_numpy(pos).cuda()]))
    for kind, R, c in ((0, RK, oracle.C_K), (1, RV, oracle.C_V)):
        for h in range(w.n_kv_heads):
            sel = np.flatnonzero((kinds == kind) & (heads == h))
            if sel.size == 0:
                continue
            xb = bf16_bits(xs[kind][sel, h])
            got = rr[sel, kind, h]
            ref = oracle.rotate_f64(xb, R[h])
            norm = np.linalg.norm(oracle.bf16_to_f64(xb), axis=1)
            assert np.all(np.abs(got - ref).max(axis=1) <= 2.0 ** -14 * norm)
            p, z, s = oracle.quantize_rows(got, w.group, c)
            assert np.array_equal(codes[kind][sel, h], p)
            assert np.array_equal(scales[kind][sel, h], s)


def test_demote_range_rejects_and_flags():
    """An unsupported page size is refused on the host; a range past the page table is skipped and
    flagged on the device, nothing written."""
    L48 = ob.Layout(2, 1, 48, 128)
    bf = ob.Bf16Pool.empty(L48, 4)
    i2 = ob.Int2Pool.empty(L48, 4)
    tab = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    R = torch.zeros((2, D, D), dtype=torch.float32, device="cuda")
    rg = torch.tensor([64, 100], dtype=torch.int32, device="cuda")
    with pytest.raises(ob.OscarError):
        ob.oscar_demote_range(L48, bf, tab, i2, tab, rg[:1], rg[1:], R, R, 1.0, 1.0)
    L = ob.Layout(2, 1, 64, 128)
    bf = ob.Bf16Pool.empty(L, 2)
    i2 = ob.Int2Pool.empty(L, 2)
    i2.codes_k.fill_(SENTINEL_CODE)
    tab = torch.arange(2, dtype=torch.int32, device="cuda").view(1, 2)
    ob.oscar_get_device_status()              # clear
    bad = torch.tensor([64, 129], dtype=torch.int32, device="cuda")     # 129 > 2 pages x 64
    ob.oscar_demote_range(L, bf, tab, i2, tab, bad[:1], bad[1:], R, R, 1.0, 1.0)
    torch.cuda.synchronize()
    assert ob.oscar_get_device_status() & 0x4          # OSCAR_DEV_BAD_LENGTH
    assert torch.all(i2.codes_k == SENTINEL_CODE)

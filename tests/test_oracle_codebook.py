"""Pins of the oracle's non-uniform (Lloyd-Max) codebook: its design routine, its quantizer and
its dequantisation inside the attention.

The pages name the codebook (OSCAR news article, closing paragraph on the latest codebase) and
give no levels, so the design routine is pinned by the mathematics: on a unit Gaussian it must
reach the continuous Lloyd-Max fixed point (computed here independently from the normal
distribution's integrals) and Max's published 4-level quantizer, and on its own design sample
every level must be the centroid of its cell and every threshold the midpoint of its levels.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import norm

import oracle


def _continuous_gaussian_lloyd_max(n=4, iters=2000):
    """Lloyd's iteration on the unit normal density itself: the centroid of [a, b) is
    (phi(a) - phi(b)) / (Phi(b) - Phi(a))."""
    lv = norm.ppf((np.arange(n) + 0.5) / n)
    for _ in range(iters):
        t = np.concatenate([[-np.inf], 0.5 * (lv[:-1] + lv[1:]), [np.inf]])
        lv = (norm.pdf(t[:-1]) - norm.pdf(t[1:])) / (norm.cdf(t[1:]) - norm.cdf(t[:-1]))
    return lv, 0.5 * (lv[:-1] + lv[1:])


def test_lloyd_max_unit_gaussian():
    exact, exact_t = _continuous_gaussian_lloyd_max()
    # Max (1960), table for N = 4 levels: outputs +-0.4528, +-1.510; inputs 0, +-0.9816
    assert np.allclose(exact, [-1.5104, -0.4528, 0.4528, 1.5104], atol=2e-4)
    assert np.allclose(exact_t, [-0.9816, 0.0, 0.9816], atol=2e-4)
    rng = np.random.default_rng(11)
    lv, t = oracle.lloyd_max(rng.standard_normal(2_000_000))
    assert np.allclose(lv, exact, atol=6e-3), lv
    assert np.allclose(t, exact_t, atol=6e-3), t


@pytest.mark.parametrize("clip", [oracle.C_K, oracle.C_V])
def test_codebook_is_a_lloyd_fixed_point_of_its_design_sample(clip):
    u = np.sort(oracle.normalised_gaussian_groups(8192, 128, clip, 0))
    lv, t = oracle.lloyd_max(u)
    assert np.all(np.diff(lv) > 0)
    assert np.array_equal(t, 0.5 * (lv[:-1] + lv[1:]))
    cell = np.searchsorted(t, u, side="right")            # a value on a threshold: the upper cell
    for k in range(4):
        assert abs(u[cell == k].mean() - lv[k]) <= 1e-9 * max(1.0, abs(lv[k]))
    # the fp32 codebook the library receives is that design rounded once
    assert np.array_equal(oracle.lloyd_max_codebook(clip), lv.astype(np.float32))


def _rows(seed, n=64, D=128):
    """Rotated-like rows: Gaussian with a few large coordinates."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 2.0, size=(n, D)).astype(np.float32)
    x[:, rng.integers(0, D, size=4)] *= 6
    return x


@pytest.mark.parametrize("group", [128, 64, 32])
def test_codebook_quantizer_takes_the_nearest_level(group):
    lv = oracle.lloyd_max_codebook(oracle.C_K)
    x = _rows(1)
    packed, zero, scale = oracle.quantize_rows(x, group, oracle.C_K, levels=lv)
    # the zero and scale are the uniform quantizer's
    _, zu, su = oracle.quantize_rows(x, group, oracle.C_K)
    assert np.array_equal(zero, zu) and np.array_equal(scale, su)
    z = oracle.bf16_to_f64(zero).astype(np.float32)
    s = oracle.bf16_to_f64(scale).astype(np.float32)
    gi = np.arange(128) // group
    u = (x - z[:, gi]) / s[:, gi]                          # fp32, as the quantizer divides
    t = ((lv[:-1] + lv[1:]) * np.float32(0.5)).astype(np.float32)
    brute = (u[..., None] >= t).sum(-1)
    codes = np.stack([oracle.unpack_row(p, 128) for p in packed])
    assert np.array_equal(codes, brute)
    # nearest level (no value sits on a midpoint in this sample)
    assert np.array_equal(codes, np.argmin(np.abs(u[..., None].astype(np.float64) - lv), axis=-1))


def test_codebook_with_uniform_levels_is_the_uniform_quantizer():
    x = _rows(2)
    a = oracle.quantize_rows(x, 128, oracle.C_V, levels=np.array([0, 1, 2, 3], np.float32))
    b = oracle.quantize_rows(x, 128, oracle.C_V)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))


@pytest.mark.parametrize("clip", [oracle.C_K, oracle.C_V])
def test_codebook_lowers_the_error_on_gaussian_groups(clip):
    lv = oracle.lloyd_max_codebook(clip)
    x = np.random.default_rng(7).standard_normal((512, 128)).astype(np.float32)
    err = {}
    for name, levels in (("uniform", None), ("lloyd", lv)):
        packed, zero, scale = oracle.quantize_rows(x, 128, clip, levels=levels)
        xh = np.stack([oracle.dequant_row(packed[r], zero[r], scale[r], 128, 128, levels=levels)
                       for r in range(x.shape[0])])
        err[name] = np.mean((xh - x) ** 2)
    assert err["lloyd"] < 0.8 * err["uniform"], err


def test_attend_head_with_codebooks_is_textbook_attention():
    """R_K = R_V = I, history rows coded with a codebook: the oracle equals softmax attention over
    zero + level[code] * scale (history) and the BF16 rows."""
    rng = np.random.default_rng(3)
    T, sink, h_end, D, g = 90, 8, 60, 128, 64
    lk = oracle.lloyd_max_codebook(oracle.C_K)
    lvv = oracle.lloyd_max_codebook(oracle.C_V)
    kb = oracle.f32_to_bf16(rng.normal(0, 1.5, size=(T, D)).astype(np.float32))
    vb = oracle.f32_to_bf16(rng.normal(0, 1.5, size=(T, D)).astype(np.float32))
    zk = oracle.f32_to_bf16(rng.uniform(-3, -1, size=(T, D // g)).astype(np.float32))
    sk = oracle.f32_to_bf16(rng.uniform(0.5, 2, size=(T, D // g)).astype(np.float32))
    zv = oracle.f32_to_bf16(rng.uniform(-3, -1, size=(T, D // g)).astype(np.float32))
    sv = oracle.f32_to_bf16(rng.uniform(0.5, 2, size=(T, D // g)).astype(np.float32))
    codes_k = rng.integers(0, 4, size=(T, D))
    codes_v = rng.integers(0, 4, size=(T, D))
    ck = np.stack([oracle.pack_row(c.astype(np.uint8)) for c in codes_k])
    cv = np.stack([oracle.pack_row(c.astype(np.uint8)) for c in codes_v])
    gi = np.arange(D) // g
    yk = oracle.bf16_to_f64(zk)[:, gi] + lk.astype(np.float64)[codes_k] * oracle.bf16_to_f64(sk)[:, gi]
    yv = oracle.bf16_to_f64(zv)[:, gi] + lvv.astype(np.float64)[codes_v] * oracle.bf16_to_f64(sv)[:, gi]
    hist = (np.arange(T) >= sink) & (np.arange(T) < h_end)
    K = np.where(hist[:, None], yk, oracle.bf16_to_f64(kb))
    V = np.where(hist[:, None], yv, oracle.bf16_to_f64(vb))
    cache = oracle.HeadCache(kb, vb, ck, cv, zk, sk, zv, sv, sink, h_end, g, levels_k=lk, levels_v=lvv)
    qb = oracle.f32_to_bf16(rng.normal(0, 1, size=D).astype(np.float32))
    q = oracle.bf16_to_f64(qb)
    I = np.eye(D, dtype=np.float32)
    o, lse = oracle.attend_head(qb, I, I, cache, 1 / math.sqrt(D))
    logits = K @ q / math.sqrt(D)
    ref = softmax(logits) @ V
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
    assert abs(lse - (np.max(logits) + math.log(np.sum(np.exp(logits - np.max(logits)))))) <= 1e-12
    # and it differs from the same codes read with the uniform levels
    uni = oracle.HeadCache(kb, vb, ck, cv, zk, sk, zv, sv, sink, h_end, g)
    assert not np.allclose(oracle.attend_head(qb, I, I, uni, 1 / math.sqrt(D))[0], o)


def test_product_codebook_designer_matches_the_oracle_design():
    """The library's offline designer (calibrate.codebook, torch) on normalised Gaussian rows: its
    levels satisfy the centroid conditions on its own sample and agree with the oracle's design
    on an independent sample to within sampling error."""
    import torch
    from bit_kv_cache_oscar_gb300 import calibrate
    g = torch.Generator().manual_seed(21)
    x = torch.randn((8192, 128), generator=g, dtype=torch.float64)
    lv = np.array(calibrate.codebook(x, 128, oracle.C_K), dtype=np.float64)
    assert np.all(np.diff(lv) > 0)
    ref = oracle.lloyd_max_codebook(oracle.C_K).astype(np.float64)
    assert np.allclose(lv, ref, atol=2e-2), (lv, ref)
    xs = x.numpy()
    lo = oracle.C_K * xs.min(1, keepdims=True)
    hi = oracle.C_K * xs.max(1, keepdims=True)
    u = np.sort(((xs - lo) / ((hi - lo) / 3.0)).reshape(-1))
    t = 0.5 * (lv[:-1] + lv[1:])
    cell = np.searchsorted(t, u, side="right")
    for k in range(4):
        assert abs(u[cell == k].mean() - lv[k]) <= 1e-5 * max(1.0, abs(lv[k]))

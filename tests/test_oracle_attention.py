"""Pins of the oracle's decode attention, split partials, merges and exp2."""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _random_orthogonal(rng, D=128):
    return np.linalg.qr(rng.normal(size=(D, D)))[0]


def _exact_cache(rng, T, sink, h_end, D=128, g=128):
    """A head cache whose history rows are exactly representable: codes, bf16 zero/scale
    drawn at random; returns the cache and the fp64 history rows y = zero + code*scale
    (in the rotated basis) plus the BF16 rows as fp64."""
    kb = oracle.f32_to_bf16(rng.normal(0, 1.5, size=(T, D)).astype(np.float32))
    vb = oracle.f32_to_bf16(rng.normal(0, 1.5, size=(T, D)).astype(np.float32))
    ck = np.zeros((T, D // 4), np.uint8)
    cv = np.zeros((T, D // 4), np.uint8)
    zk = oracle.f32_to_bf16(rng.uniform(-3, -1, size=(T, D // g)).astype(np.float32))
    sk = oracle.f32_to_bf16(rng.uniform(0.5, 2, size=(T, D // g)).astype(np.float32))
    zv = oracle.f32_to_bf16(rng.uniform(-3, -1, size=(T, D // g)).astype(np.float32))
    sv = oracle.f32_to_bf16(rng.uniform(0.5, 2, size=(T, D // g)).astype(np.float32))
    yk = np.zeros((T, D))
    yv = np.zeros((T, D))
    for p in range(T):
        codes_k = rng.integers(0, 4, size=D).astype(np.uint8)
        codes_v = rng.integers(0, 4, size=D).astype(np.uint8)
        ck[p] = oracle.pack_row(codes_k)
        cv[p] = oracle.pack_row(codes_v)
        gi = np.arange(D) // g
        yk[p] = oracle.bf16_to_f64(zk[p])[gi] + codes_k * oracle.bf16_to_f64(sk[p])[gi]
        yv[p] = oracle.bf16_to_f64(zv[p])[gi] + codes_v * oracle.bf16_to_f64(sv[p])[gi]
    cache = oracle.HeadCache(kb, vb, ck, cv, zk, sk, zv, sv, sink, h_end, g)
    return cache, yk, yv, oracle.bf16_to_f64(kb), oracle.bf16_to_f64(vb)


def _textbook(q, K, V, scale):
    p = softmax(scale * (K @ q))
    return p @ V, math.log(np.sum(np.exp(scale * (K @ q) - np.max(scale * (K @ q))))) + np.max(scale * (K @ q))


@pytest.mark.parametrize("g", [128, 32])
def test_identity_rotation_equals_textbook_softmax(g):
    """R_K = R_V = I and exactly-representable history: the oracle equals plain softmax attention
    over the cache's true keys/values (BF16 rows where BF16, zero + code*scale in history)."""
    rng = np.random.default_rng(0)
    T, sink, h_end, D = 100, 8, 70, 128
    cache, yk, yv, kf, vf = _exact_cache(rng, T, sink, h_end, D, g)
    hist = (np.arange(T) >= sink) & (np.arange(T) < h_end)
    K = np.where(hist[:, None], yk, kf)
    V = np.where(hist[:, None], yv, vf)
    qb = oracle.f32_to_bf16(rng.normal(0, 1, size=D).astype(np.float32))
    q = oracle.bf16_to_f64(qb)
    I = np.eye(D, dtype=np.float32)
    o, lse = oracle.attend_head(qb, I, I, cache, 1 / math.sqrt(D))
    ref, ref_lse = _textbook(q, K, V, 1 / math.sqrt(D))
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
    assert abs(lse - ref_lse) < 1e-12


def test_rotated_history_is_invariant():
    """History stored in the rotated basis y = x·R: with q rotated by R_K and the history value
    sum rotated back by R_V^T, attention equals plain attention over x_k = y_k R_K^T,
    x_v = y_v R_V^T.  A transposed rotation anywhere breaks this."""
    rng = np.random.default_rng(1)
    T, sink, h_end, D = 90, 8, 60, 128
    cache, yk, yv, kf, vf = _exact_cache(rng, T, sink, h_end, D, 128)
    RK = _random_orthogonal(rng).astype(np.float32)
    RV = _random_orthogonal(rng).astype(np.float32)
    hist = (np.arange(T) >= sink) & (np.arange(T) < h_end)
    K = np.where(hist[:, None], yk @ RK.astype(np.float64).T, kf)
    V = np.where(hist[:, None], yv @ RV.astype(np.float64).T, vf)
    qb = oracle.f32_to_bf16(rng.normal(0, 1, size=D).astype(np.float32))
    o, lse = oracle.attend_head(qb, RK, RV, cache, 0.09)
    ref, ref_lse = _textbook(oracle.bf16_to_f64(qb), K, V, 0.09)
    assert np.allclose(o, ref, rtol=1e-10, atol=1e-10)
    assert abs(lse - ref_lse) < 1e-10


def _splits(sink, h_end, S, ps):
    """Page-aligned history splits used by the tests (any partition works for the merge)."""
    first, last = sink // ps, (h_end + ps - 1) // ps
    n = last - first
    per = -(-n // S)
    out = []
    for s in range(S):
        a = (first + s * per) * ps
        b = min((first + (s + 1) * per) * ps, h_end)
        out.append((max(a, sink), b) if a < b else (0, 0))
    return out


@pytest.mark.parametrize("S", [1, 3, 7])
def test_split_partials_merge_equals_direct(S):
    rng = np.random.default_rng(2)
    T, sink, h_end, D = 200, 16, 150, 128
    cache, *_ = _exact_cache(rng, T, sink, h_end, D, 128)
    RK = _random_orthogonal(rng).astype(np.float32)
    RV = _random_orthogonal(rng).astype(np.float32)
    qb = oracle.f32_to_bf16(rng.normal(0, 2, size=D).astype(np.float32))
    scale = 1 / math.sqrt(D)
    m2, l, acc = [], [], []
    for (a, b) in _splits(sink, h_end, S, 16):
        r = oracle.partial(qb, RK, cache, scale, [(a, b)] if b > a else [])
        m2.append(r[0]); l.append(r[1]); acc.append(r[2])
    r = oracle.partial(qb, RK, cache, scale, [(0, sink), (h_end, T)])
    m2.append(r[0]); l.append(r[1]); acc.append(r[2])
    o, lse = oracle.merge_f64(np.array(m2), np.array(l), np.array(acc), RV)
    ref, ref_lse = oracle.attend_head(qb, RK, RV, cache, scale)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
    assert abs(lse - ref_lse) < 1e-12


def test_single_partial_merge_is_normalisation():
    rng = np.random.default_rng(3)
    acc = rng.normal(size=(1, 128))
    o, lse = oracle.merge_f64(np.array([1.5]), np.array([4.0]), acc, None)
    assert np.allclose(o, acc[0] / 4.0, rtol=1e-15)
    assert abs(lse - (1.5 + math.log2(4.0)) * math.log(2)) < 1e-14


def test_exp2f_accuracy_and_exact_points():
    for n in range(-125, 10):
        assert oracle.exp2f(float(n)) == 2.0 ** n
    assert oracle.exp2f(-math.inf) == 0.0
    assert oracle.exp2f(-200.0) == 0.0
    xs = np.float32(np.linspace(-60, 0, 20001))
    for x in xs:
        got = np.float32(oracle.exp2f(float(x)))
        ref = 2.0 ** float(x)
        ulp = np.spacing(np.float32(ref))
        assert abs(float(got) - ref) <= 2 * float(ulp), x


@pytest.mark.parametrize("S,empty", [(1, ()), (5, (2,)), (16, (0, 15)), (4, (4,))])
def test_merge_f32_close_to_f64(S, empty):
    import oscar_synthetic as syn
    rng = np.random.default_rng(4)
    RV = _random_orthogonal(rng).astype(np.float32)
    m2, l, acc = syn.split_partials(S, S, 128, empty)
    o32, ob = oracle.merge_f32(m2, l, acc, RV)
    o64, _ = oracle.merge_f64(m2.astype(np.float64), l.astype(np.float64), acc.astype(np.float64), RV)
    err = np.linalg.norm(o32 - o64) / np.linalg.norm(o64)
    assert err < 1e-6
    assert np.array_equal(ob, oracle.f32_to_bf16(o32))


def test_merge_f32_single_partial_exact():
    """One non-empty partial, no rotation: o = acc / l with one IEEE division per element."""
    acc = np.array([[3.0, -7.5, 1e-3] + [0.0] * 125], np.float32)
    o, _ = oracle.merge_f32(np.array([2.0], np.float32), np.array([3.0], np.float32), acc, None)
    assert o[0] == np.float32(3.0) / np.float32(3.0)
    assert o[1] == np.float32(-7.5) / np.float32(3.0)
    assert o[2] == np.float32(1e-3) / np.float32(3.0)

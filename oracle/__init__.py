"""OSCAR oracle: the plain CPU reference that the CUDA path is checked against.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package; the product library never
does, and the two share no code.  The numeric core is ``oscar_oracle.c`` (plain
C, fp64 definitions, fp32 only where the method takes an integer decision or a
bit-exact fold is specified); the offline rotation builder below is numpy fp64.

Sources, cited by page title and section:
  * OSCAR news article (m.kljzs.com mirror), paragraphs on the offline
    calibration ("R = U·Hadamard·bit-reversal") and the online layout.
  * "Together AI 開源 OSCAR" (news.chathome.org), section "OSCAR 的不同之處":
    key error identity ||QK^T - QK_hat^T||_F^2 = tr((K-K_hat) Q^T Q (K-K_hat)^T),
    C_Q = (1/N) sum q_n^T q_n, C_S = (1/N) V^T S^T S V, R_K = U_Q·H·P_br,
    R_V = U_S·H·P_br; section "服務系統" (64 sink + 256 recent tokens in BF16).
  * "OSCAR — 离线转个方向，把 KV Cache 压到 2-bit" (estelledc study notes),
    "核心要点" items 2-3 and "案例 2" (c_K ~ 0.96, c_V ~ 0.92).

Parity status of each function is listed in ``PINS`` at the bottom; every one
is pinned by a ``-m "not gpu"`` test against closed forms, special cases,
printed page values or brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oscar_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboscar_oracle.so")
_lib = None

C_K = 0.96   # key clip ratio ("案例 2", estelledc notes)
C_V = 0.92   # value clip ratio
SINK = 64    # "服務系統" (chathome): first 64 tokens stay BF16
RECENT = 256  # last 256 tokens stay BF16


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fused multiply-add contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i, f, d = ctypes.c_int, ctypes.c_float, ctypes.c_double
        L.ora_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.ora_bf16_to_f64.restype = d
        L.ora_f32_to_bf16.argtypes = [f]
        L.ora_f32_to_bf16.restype = ctypes.c_uint16
        L.ora_rotate_f32.argtypes = [P, P, i, P]
        L.ora_rotate_f64.argtypes = [P, P, i, P]
        L.ora_quantize_row.argtypes = [P, i, i, f, P, P, P]
        L.ora_pack_row.argtypes = [P, i, P]
        L.ora_unpack_row.argtypes = [P, i, P]
        L.ora_dequant_row.argtypes = [P, P, P, i, i, P]
        L.ora_dequant_row_cb.argtypes = [P, P, P, i, i, P, P]
        L.ora_quantize_row_cb.argtypes = [P, i, i, f, P, P, P, P]
        L.ora_demote_rows.argtypes = [P, P, i, i, i, f, P, P, P, P]
        L.ora_demote_rows_cb.argtypes = [P, P, i, i, i, f, P, P, P, P, P]
        L.ora_quantize_rows.argtypes = [P, i, i, i, f, P, P, P, P]
        L.ora_attend_head_f64.argtypes = [i, i, i, i, i, d] + [P] * 13 + [P, P]
        L.ora_partial_f64.argtypes = [i, i, i, i, i, d] + [P] * 12 + [i, P, P, P, P, P]
        L.ora_merge_f64.argtypes = [i, i, P, P, P, P, P, P]
        L.ora_exp2f.argtypes = [f]
        L.ora_exp2f.restype = f
        L.ora_merge_f32.argtypes = [i, i, P, P, P, P, P, P]
        L.ora_bits_per_element.argtypes = [ctypes.c_longlong, i, i, i]
        L.ora_bits_per_element.restype = d
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bf16 ----

def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16(x) -> np.ndarray:
    """binary32 -> bf16 bit patterns, round to nearest even (element by element)."""
    x = np.asarray(x, dtype=np.float32)
    L = lib()
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for n in range(flat_in.size):
        flat_out[n] = L.ora_f32_to_bf16(float(flat_in[n]))
    return out


# -------------------------------------------------------------- rotation ----

def rotate_f32(x_bf16: np.ndarray, R: np.ndarray) -> np.ndarray:
    """x·R for rows of bf16 x, fp32 fused multiply-add chain in ascending index order."""
    x = _c(x_bf16, np.uint16)
    R = _c(R, np.float32)
    D = R.shape[0]
    rows = x.reshape(-1, D)
    out = np.empty(rows.shape, dtype=np.float32)
    L = lib()
    for r in range(rows.shape[0]):
        L.ora_rotate_f32(_p(rows[r]), _p(R), D, _p(out[r]))
    return out.reshape(x.shape)


def rotate_f64(x_bf16: np.ndarray, R: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    R = _c(R, np.float32)
    D = R.shape[0]
    rows = x.reshape(-1, D)
    out = np.empty(rows.shape, dtype=np.float64)
    L = lib()
    for r in range(rows.shape[0]):
        L.ora_rotate_f64(_p(rows[r]), _p(R), D, _p(out[r]))
    return out.reshape(x.shape)


# ------------------------------------------------------------- quantizer ----

def _levels(levels):
    """A codebook as fp32 [4] (None: the uniform levels 0, 1, 2, 3)."""
    if levels is None:
        return None
    lv = _c(levels, np.float32).reshape(-1)
    assert lv.shape == (4,) and np.all(np.isfinite(lv)) and np.all(np.diff(lv) > 0), lv
    return lv


def quantize_rows(x_rot: np.ndarray, group: int, clip: float, levels=None):
    """Codec on fp32 rotated rows [..., D] -> (packed uint8 [..., D/4], zero, scale bf16 [..., D/g]);
    levels: a 4-level codebook on the normalised axis (ora_quantize_row_cb), None = uniform."""
    x = _c(x_rot, np.float32)
    D = x.shape[-1]
    n = x.size // D
    packed = np.empty(x.shape[:-1] + (D // 4,), dtype=np.uint8)
    zero = np.empty(x.shape[:-1] + (D // group,), dtype=np.uint16)
    scale = np.empty_like(zero)
    lv = _levels(levels)
    lib().ora_quantize_rows(_p(x), n, D, group, float(np.float32(clip)), _p(lv), _p(packed), _p(zero), _p(scale))
    return packed, zero, scale


def quantize_row_codes(x_rot: np.ndarray, group: int, clip: float):
    """One row -> (codes 0..3 [D] uint8, zero, scale)."""
    x = _c(x_rot, np.float32)
    D = x.shape[0]
    codes = np.empty(D, dtype=np.uint8)
    zero = np.empty(D // group, dtype=np.uint16)
    scale = np.empty(D // group, dtype=np.uint16)
    lib().ora_quantize_row(_p(x), D, group, float(np.float32(clip)), _p(codes), _p(zero), _p(scale))
    return codes, zero, scale


def pack_row(codes: np.ndarray) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape[0] // 4, dtype=np.uint8)
    lib().ora_pack_row(_p(c), c.shape[0], _p(out))
    return out


def unpack_row(packed: np.ndarray, D: int) -> np.ndarray:
    p = _c(packed, np.uint8)
    out = np.empty(D, dtype=np.uint8)
    lib().ora_unpack_row(_p(p), D, _p(out))
    return out


def dequant_row(packed, zero, scale, D: int, group: int, levels=None) -> np.ndarray:
    out = np.empty(D, dtype=np.float64)
    lib().ora_dequant_row_cb(_p(_c(packed, np.uint8)), _p(_c(zero, np.uint16)),
                             _p(_c(scale, np.uint16)), D, group, _p(_levels(levels)), _p(out))
    return out


def demote_rows(x_bf16: np.ndarray, R: np.ndarray, group: int, clip: float, levels=None):
    """Rotate (fp32 chain) + quantize + pack rows [n, D] sharing one R (levels: a codebook, None = uniform).

    Returns (rotated fp32 [n, D], packed [n, D/4], zero [n, D/g], scale [n, D/g]).
    """
    x = _c(x_bf16, np.uint16)
    R = _c(R, np.float32)
    n, D = x.shape
    rot = np.empty((n, D), dtype=np.float32)
    packed = np.empty((n, D // 4), dtype=np.uint8)
    zero = np.empty((n, D // group), dtype=np.uint16)
    scale = np.empty_like(zero)
    lib().ora_demote_rows_cb(_p(x), _p(R), n, D, group, float(np.float32(clip)), _p(_levels(levels)),
                             _p(rot), _p(packed), _p(zero), _p(scale))
    return rot, packed, zero, scale


# ------------------------------------------------------------- attention ----

class HeadCache:
    """One kv head's logical (token-major, unpaged) cache of one request.

    k, v: bf16 bits [T, D] (meaningful at BF16 positions); ck, cv: packed
    codes [T, D/4]; zk, sk, zv, sv: bf16 bits [T, D/g] (meaningful at history
    positions [sink, h_end)); levels_k / levels_v: the codebooks the codes index (None = uniform).
    """

    def __init__(self, k, v, ck, cv, zk, sk, zv, sv, sink, h_end, group, levels_k=None, levels_v=None):
        self.k = _c(k, np.uint16)
        self.v = _c(v, np.uint16)
        self.ck = _c(ck, np.uint8)
        self.cv = _c(cv, np.uint8)
        self.zk = _c(zk, np.uint16)
        self.sk = _c(sk, np.uint16)
        self.zv = _c(zv, np.uint16)
        self.sv = _c(sv, np.uint16)
        self.T, self.D = self.k.shape
        self.sink, self.h_end, self.group = int(sink), int(h_end), int(group)
        self.lk, self.lv = _levels(levels_k), _levels(levels_v)

    def _args(self):
        return [_p(self.k), _p(self.v), _p(self.ck), _p(self.cv),
                _p(self.zk), _p(self.sk), _p(self.zv), _p(self.sv), _p(self.lk), _p(self.lv)]


def attend_head(q_bf16, RK, RV, cache: HeadCache, sm_scale: float):
    """Full fp64 decode attention of one query head -> (o [D] fp64, lse)."""
    q = _c(q_bf16, np.uint16)
    RK = _c(RK, np.float32)
    RV = _c(RV, np.float32)
    out = np.empty(cache.D, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib().ora_attend_head_f64(cache.D, cache.T, cache.sink, cache.h_end, cache.group, float(sm_scale),
                              _p(q), _p(RK), _p(RV), *cache._args(), _p(out), _p(lse))
    return out, float(lse[0])


def partial(q_bf16, RK, cache: HeadCache, sm_scale: float, ranges):
    """Base-2 split partial (m2, l, acc[D]) over token ranges [(lo, hi), ...], fp64."""
    q = _c(q_bf16, np.uint16)
    RK = _c(RK, np.float32)
    lo = np.array([r[0] for r in ranges] or [0], dtype=np.int32)
    hi = np.array([r[1] for r in ranges] or [0], dtype=np.int32)
    m2 = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    acc = np.zeros(cache.D, dtype=np.float64)
    lib().ora_partial_f64(cache.D, cache.T, cache.sink, cache.h_end, cache.group, float(sm_scale),
                          _p(q), _p(RK), *cache._args(), len(ranges), _p(lo), _p(hi),
                          _p(m2), _p(l), _p(acc))
    return float(m2[0]), float(l[0]), acc


def merge_f64(m2, l, acc, RV):
    """fp64 merge of S history partials + 1 BF16 partial -> (o [D], lse)."""
    m2 = _c(m2, np.float64)
    l = _c(l, np.float64)
    acc = _c(acc, np.float64)
    S = m2.shape[0] - 1
    D = acc.shape[-1]
    out = np.empty(D, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib().ora_merge_f64(D, S, _p(m2), _p(l), _p(acc), None if RV is None else _p(_c(RV, np.float32)),
                        _p(out), _p(lse))
    return out, float(lse[0])


def merge_f32(m2, l, acc, RV):
    """Ordered fp32 merge (bit-exact contract) -> (o fp32 [D], o bf16 bits [D])."""
    m2 = _c(m2, np.float32)
    l = _c(l, np.float32)
    acc = _c(acc, np.float32)
    S = m2.shape[0] - 1
    D = acc.shape[-1]
    out = np.empty(D, dtype=np.float32)
    ob = np.empty(D, dtype=np.uint16)
    lib().ora_merge_f32(D, S, _p(m2), _p(l), _p(acc), None if RV is None else _p(_c(RV, np.float32)),
                        _p(out), _p(ob))
    return out, ob


def exp2f(x: float) -> float:
    return float(lib().ora_exp2f(float(np.float32(x))))


def bits_per_element(T: int, group: int = 128, sink: int = SINK, recent: int = RECENT) -> float:
    return float(lib().ora_bits_per_element(int(T), int(group), int(sink), int(recent)))


# ------------------------------------------------- offline rotation (fp64) ----

def hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_n / sqrt(n) (orthogonal, entries +-1/sqrt(n))."""
    assert n >= 1 and (n & (n - 1)) == 0
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H / np.sqrt(n)


def bit_reverse(i: int, bits: int) -> int:
    r = 0
    for b in range(bits):
        r |= ((i >> b) & 1) << (bits - 1 - b)
    return r


def bit_reversal_permutation(n: int) -> np.ndarray:
    """P_br with P[i, br(i)] = 1 (an involution, so P = P^T)."""
    bits = n.bit_length() - 1
    P = np.zeros((n, n))
    for i in range(n):
        P[i, bit_reverse(i, bits)] = 1.0
    return P


def eig_basis(C: np.ndarray) -> np.ndarray:
    """Eigenvectors of symmetric C as columns, eigenvalues descending.

    Sign convention: the largest-magnitude component of each column is positive
    (first such index on ties).  Equal eigenvalues keep eigh's order.
    """
    w, U = np.linalg.eigh(np.asarray(C, dtype=np.float64))
    order = np.argsort(-w, kind="stable")
    U = U[:, order].copy()
    for j in range(U.shape[1]):
        i = int(np.argmax(np.abs(U[:, j])))
        if U[i, j] < 0:
            U[:, j] = -U[:, j]
    return U


def query_covariance(q: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n for query rows q [N, D] ("OSCAR 的不同之處")."""
    q = np.asarray(q, dtype=np.float64)
    return q.T @ q / q.shape[0]


def score_weighted_value_covariance(q, k, v, sm_scale: float) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V with S = softmax(sm_scale q K^T) row-wise ("OSCAR 的不同之處")."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    logits = sm_scale * (q @ k.T)
    logits -= logits.max(axis=1, keepdims=True)
    S = np.exp(logits)
    S /= S.sum(axis=1, keepdims=True)
    SV = S @ v
    return SV.T @ SV / q.shape[0]


def rotation_from_covariance(C: np.ndarray) -> np.ndarray:
    """R = U · H_Had · P_br (fp64), U the descending eigenbasis of C."""
    D = C.shape[0]
    return eig_basis(C) @ hadamard(D) @ bit_reversal_permutation(D)


def key_logit_error(Q, K, K_hat) -> float:
    """||Q K^T - Q K_hat^T||_F^2 (the quantity the key rotation targets)."""
    Q = np.asarray(Q, dtype=np.float64)
    return float(np.sum((Q @ np.asarray(K, np.float64).T - Q @ np.asarray(K_hat, np.float64).T) ** 2))


def key_logit_error_trace(Q, K, K_hat) -> float:
    """tr((K - K_hat) Q^T Q (K - K_hat)^T), the same quantity through the query covariance."""
    Q = np.asarray(Q, dtype=np.float64)
    dK = np.asarray(K, np.float64) - np.asarray(K_hat, np.float64)
    return float(np.trace(dK @ (Q.T @ Q) @ dK.T))


# ------------------------------------------------ Lloyd-Max codebook (fp64) ----

def lloyd_max(samples, n_levels: int = 4, iters: int = 1000, tol: float = 1e-13):
    """Lloyd's algorithm (Lloyd 1957; Max 1960) for the n-level scalar quantizer of least mean
    squared error on an empirical distribution: starting from the sample quantiles at
    (k + 1/2)/n, alternately put each threshold at the midpoint of its two levels and each level at
    the mean of the samples of its cell (a value on a threshold belongs to the upper cell, as in
    the quantizer; a cell that empties keeps its level), until no level moves by more than tol.
    Returns (levels [n], thresholds [n - 1]) in fp64.  The codebook's use: OSCAR news article,
    closing paragraph (the latest codebase's Lloyd-Max codebook); the pages give no levels."""
    x = np.sort(np.asarray(samples, dtype=np.float64).reshape(-1))
    assert x.size >= n_levels and np.all(np.isfinite(x))
    lv = np.quantile(x, (np.arange(n_levels) + 0.5) / n_levels)
    cs = np.concatenate([[0.0], np.cumsum(x)])
    for _ in range(iters):
        t = 0.5 * (lv[:-1] + lv[1:])
        cut = np.concatenate([[0], np.searchsorted(x, t, side="left"), [x.size]])
        new = lv.copy()
        for k in range(n_levels):
            a, b = cut[k], cut[k + 1]
            if b > a:
                new[k] = (cs[b] - cs[a]) / (b - a)
        moved = np.max(np.abs(new - lv))
        lv = new
        if moved <= tol:
            break
    return lv, 0.5 * (lv[:-1] + lv[1:])


def normalised_gaussian_groups(n_groups: int, group: int, clip: float, seed: int) -> np.ndarray:
    """Design sample of the codebook: u = (y - lo) / ((hi - lo) / 3) for groups of `group`
    standard normal values y with lo = clip * min, hi = clip * max, i.e. the uniform quantizer's
    per-group normalisation (in fp64, without its bf16 rounding).  The rotated coordinates are
    modelled as Gaussian within a group (the rotation mixes every channel into each)."""
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((n_groups, group))
    lo = clip * y.min(axis=1, keepdims=True)
    hi = clip * y.max(axis=1, keepdims=True)
    return ((y - lo) / ((hi - lo) / 3.0)).reshape(-1)


def lloyd_max_codebook(clip: float, group: int = 128, n_groups: int = 8192, seed: int = 0) -> np.ndarray:
    """The 4-level codebook (fp32, increasing) on the normalised axis for a clip ratio: Lloyd's
    algorithm on normalised_gaussian_groups.  Passed to the library as the layout's levels."""
    lv, _ = lloyd_max(normalised_gaussian_groups(n_groups, group, clip, seed))
    return lv.astype(np.float32)


PINS = {
    "rotate_f32": "fp64 bound + ascending-order rounding case (tests/test_oracle_codec.py)",
    "quantize_rows": "hand-derived worked rows (tests/test_oracle_codec.py::test_quantizer_worked_rows), "
                     "brute-force nearest level, error bound",
    "pack_row/unpack_row": "all 256 bytes round trip, worked byte",
    "attend_head": "textbook softmax attention on exactly quantizable caches, rotation invariance",
    "partial/merge_f64": "split + merge equals direct attention; one split is the identity",
    "merge_f32/exp2f": "against fp64 merge and exp2 within ulp bounds; exact at integers",
    "rotation_from_covariance": "Hadamard/permutation closed forms, orthogonality, diagonalisation, q=0 rank-one C_S",
    "bits_per_element": "page values 2.28 / 2.38 bits and 0.24% BF16 share (tests/golden/pages_numbers.json)",
    "score_weighted_value_covariance": "the value rotation built from it lowers the attention-weighted value "
                                       "error below H·P_br alone on synthetic data (tests/test_oracle_quality.py)",
    "lloyd_max": "unit Gaussian levels against the continuous Lloyd-Max fixed point (scipy normal "
                 "integrals) and Max's published 4-level table; centroid and midpoint conditions "
                 "(tests/test_oracle_codebook.py)",
    "quantize_rows/demote_rows/dequant_row with levels": "brute-force nearest level, uniform levels "
                 "reproduce the uniform quantizer off ties, lower error than uniform on fresh Gaussian groups",
    "attend_head with codebooks": "textbook softmax attention over the dequantised rows",
}

"""One decode-step scenario for the parity tests and the smoke check.

Builds seeded inputs (oscar_synthetic), the oracle's rotations, paged pools on
the device, runs the CUDA path through the C ABI, and gives the oracle the same
inputs in logical (unpaged) order.  Host plumbing only: placing rows in pages
and gathering them back is memory layout, not the method's arithmetic.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

import oracle
import oscar_synthetic as syn
from bit_kv_cache_oscar_gb300 import binding as ob
from tests.helpers import bf16_bits

D = 128


def oracle_rotations(seed: int, layer: int, n_kv: int, gqa: int):
    """fp32 R_K, R_V [Hkv, D, D] from the oracle's offline builder (fp64, rounded once)."""
    prof = syn.channel_profile(seed, layer, n_kv)
    q, k, v = syn.calibration_set(seed, layer, gqa, prof)
    RK = np.empty((n_kv, D, D), np.float32)
    RV = np.empty((n_kv, D, D), np.float32)
    for h in range(n_kv):
        qd = oracle.bf16_to_f64(bf16_bits(q[h]))
        kd = oracle.bf16_to_f64(bf16_bits(k[h]))
        vd = oracle.bf16_to_f64(bf16_bits(v[h]))
        RK[h] = oracle.rotation_from_covariance(oracle.query_covariance(qd)).astype(np.float32)
        RV[h] = oracle.rotation_from_covariance(
            oracle.score_weighted_value_covariance(qd, kd, vd, 1.0 / math.sqrt(D))).astype(np.float32)
    return prof, RK, RV


@dataclasses.dataclass
class Case:
    layout: ob.Layout
    seq: List[int]
    hist_end: np.ndarray
    K: List[torch.Tensor]          # per request bf16 [T, Hkv, D] (CPU)
    V: List[torch.Tensor]
    q: torch.Tensor                # bf16 [B, Hq, D] (CPU)
    RK: np.ndarray
    RV: np.ndarray
    pages: syn.PageLayout
    sm_scale: float
    # device side
    dev: dict = dataclasses.field(default_factory=dict)


def make_case(n_kv=2, gqa=4, page_size=16, group=128, seq=(1024,), seed=0, layer=0, hist_end=None,
              sink=64, recent=256, device="cuda", gen_device="cpu", shared_prefix=0, levels=None) -> Case:
    """gen_device="cuda" draws K/V on the GPU (long contexts); both sides still get the same
    tensors (the oracle reads the sampled heads back).  levels: (key, value) codebooks."""
    lk, lv = (None, None) if levels is None else (tuple(float(x) for x in levels[0]),
                                                   tuple(float(x) for x in levels[1]))
    layout = ob.Layout(n_kv, gqa, page_size, group, sink, recent, levels_k=lk, levels_v=lv)
    prof, RK, RV = oracle_rotations(seed, layer, n_kv, gqa)
    w = syn.Workload("case", 1, n_kv * gqa, n_kv, len(seq), max(seq), page_size, group=group,
                     sink=sink, recent=recent, seed=seed, shared_prefix=shared_prefix)
    pages = syn.page_layout(w, list(seq), hist_end=hist_end)
    K, V = [], []
    for b, T in enumerate(seq):
        k, v = syn.kv_rows(seed, layer, b, 0, T, prof, device=gen_device, shared_prefix=shared_prefix)
        K.append(k)
        V.append(v)
    q = syn.queries(seed, layer, len(seq), gqa, prof)
    return Case(layout, list(seq), pages.hist_end.copy(), K, V, q, RK, RV, pages, 1.0 / math.sqrt(D))


def upload(case: Case, device="cuda", demote_history=True, keep_rotated=True):
    """Allocate pools and fill them: BF16 rows where the page layout keeps BF16 pages, and the
    history demoted through oscar_demote from a staging pool holding every row."""
    L, P = case.layout, case.pages
    ps, B = L.page_size, len(case.seq)
    dev = case.dev
    bf = ob.Bf16Pool.empty(L, max(P.n_bf16_pages, 1), device)
    i2 = ob.Int2Pool.empty(L, max(P.n_int2_pages, 1), device)
    for b, T in enumerate(case.seq):
        for lp in range(P.bf16_table.shape[1]):
            pg = int(P.bf16_table[b, lp])
            if pg < 0:
                continue
            p0, p1 = lp * ps, min(T, (lp + 1) * ps)
            if p0 >= p1:
                continue
            bf.k[pg, :p1 - p0] = case.K[b][p0:p1].to(device)
            bf.v[pg, :p1 - p0] = case.V[b][p0:p1].to(device)
    # staging pool: every logical page of every request, in order
    n_log = [(T + ps - 1) // ps for T in case.seq]
    stage = ob.Bf16Pool.empty(L, sum(n_log), device)
    st_table = -np.ones((B, P.int2_table.shape[1]), np.int32)
    base = 0
    for b, T in enumerate(case.seq):
        n = n_log[b]                       # logical pages of request b sit at base .. base+n-1
        stage.k[base:base + n].reshape(n * ps, L.n_kv_heads, D)[:T] = case.K[b].to(device)
        stage.v[base:base + n].reshape(n * ps, L.n_kv_heads, D)[:T] = case.V[b].to(device)
        st_table[b, :n] = np.arange(base, base + n, dtype=np.int32)
        base += n
    dev.update(
        bf16=bf, int2=i2, stage=stage,
        bf16_table=torch.from_numpy(P.bf16_table).to(device),
        int2_table=torch.from_numpy(P.int2_table).to(device),
        stage_table=torch.from_numpy(st_table).to(device),
        seq_len=torch.tensor(case.seq, dtype=torch.int32, device=device),
        hist_end=torch.from_numpy(case.hist_end.astype(np.int32)).to(device),
        RK=torch.from_numpy(case.RK).to(device), RV=torch.from_numpy(case.RV).to(device),
        q=case.q.to(device))
    if demote_history:
        req, pos = [], []
        for b, T in enumerate(case.seq):
            for p in range(L.sink, int(case.hist_end[b])):
                req.append(b)
                pos.append(p)
        dev["demote_req"] = torch.tensor(req, dtype=torch.int32, device=device)
        dev["demote_pos"] = torch.tensor(pos, dtype=torch.int32, device=device)
        if req:
            if keep_rotated:
                dev["rotated"] = torch.empty((len(req), 2, L.n_kv_heads, D), dtype=torch.float32, device=device)
            ob.oscar_demote(L, stage, dev["stage_table"], i2, dev["int2_table"], dev["demote_req"],
                            dev["demote_pos"], dev["RK"], dev["RV"], oracle.C_K, oracle.C_V,
                            rotated_out=dev.get("rotated"))
    return dev


def run_decode(case: Case, n_splits: int, device="cuda"):
    """rotate_q -> decode_attention -> merge through the C ABI; returns (out bf16, out fp32, lse, partials)."""
    L, dev = case.layout, case.dev
    B = len(case.seq)
    q_rot = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device=device)
    ob.oscar_rotate_q(L, dev["q"], dev["RK"], q_rot)
    part = ob.Partials.empty(L, B, n_splits, device)
    ob.oscar_decode_attention(L, dev["q"], q_rot, dev["bf16"], dev["bf16_table"], dev["int2"], dev["int2_table"],
                              dev["seq_len"], dev["hist_end"], case.sm_scale, part)
    out = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device=device)
    out32 = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device=device)
    lse = torch.empty((B, L.n_q_heads), dtype=torch.float32, device=device)
    ob.oscar_merge(L, part, dev["RV"], out, out32, lse)
    torch.cuda.synchronize()
    dev["q_rot"] = q_rot
    return out, out32, lse, part


def gather_int2(case: Case, b: int, h: int):
    """The device INT2 pool of request b, kv head h, in logical order [T, ...] (zeros outside history)."""
    L, P, i2 = case.layout, case.pages, case.dev["int2"]
    T, ps, g = case.seq[b], L.page_size, L.group
    ck = np.zeros((T, D // 4), np.uint8)
    cv = np.zeros((T, D // 4), np.uint8)
    zk, sk, zv, sv = (np.zeros((T, D // g), np.uint16) for _ in range(4))
    codes_k = i2.codes_k[:, :, h].cpu().numpy()
    codes_v = i2.codes_v[:, :, h].cpu().numpy()
    zk_a, sk_a = bf16_bits(i2.zero_k[:, :, h]), bf16_bits(i2.scale_k[:, :, h])
    zv_a, sv_a = bf16_bits(i2.zero_v[:, :, h]), bf16_bits(i2.scale_v[:, :, h])
    for p in range(L.sink, int(case.hist_end[b])):
        pg, sl = int(P.int2_table[b, p // ps]), p % ps
        ck[p], cv[p] = codes_k[pg, sl], codes_v[pg, sl]
        zk[p], sk[p], zv[p], sv[p] = zk_a[pg, sl], sk_a[pg, sl], zv_a[pg, sl], sv_a[pg, sl]
    return ck, cv, zk, sk, zv, sv


def oracle_head_cache(case: Case, b: int, h: int) -> oracle.HeadCache:
    """The oracle's own cache of (request b, kv head h): its own demotion of the history rows."""
    L = case.layout
    T, he, g = case.seq[b], int(case.hist_end[b]), L.group
    kb = bf16_bits(case.K[b][:, h])
    vb = bf16_bits(case.V[b][:, h])
    ck = np.zeros((T, D // 4), np.uint8)
    cv = np.zeros((T, D // 4), np.uint8)
    zk, sk, zv, sv = (np.zeros((T, D // g), np.uint16) for _ in range(4))
    if he > L.sink:
        _, ck[L.sink:he], zk[L.sink:he], sk[L.sink:he] = oracle.demote_rows(kb[L.sink:he], case.RK[h], g, oracle.C_K,
                                                                            levels=L.levels_k)
        _, cv[L.sink:he], zv[L.sink:he], sv[L.sink:he] = oracle.demote_rows(vb[L.sink:he], case.RV[h], g, oracle.C_V,
                                                                            levels=L.levels_v)
    return oracle.HeadCache(kb, vb, ck, cv, zk, sk, zv, sv, L.sink, he, g, levels_k=L.levels_k, levels_v=L.levels_v)


def oracle_outputs(case: Case, heads: Optional[list] = None):
    """fp64 oracle output and lse for (b, q-head) pairs (all by default)."""
    L = case.layout
    qb = bf16_bits(case.q)
    B = len(case.seq)
    pairs = heads or [(b, hq) for b in range(B) for hq in range(L.n_q_heads)]
    caches = {}
    out = {}
    for b, hq in pairs:
        h = hq // L.gqa
        if (b, h) not in caches:
            caches[(b, h)] = oracle_head_cache(case, b, h)
        out[(b, hq)] = oracle.attend_head(qb[b, hq], case.RK[h], case.RV[h], caches[(b, h)], case.sm_scale)
    return out


def tolerance_ok(got: np.ndarray, ref: np.ndarray, rel_l2=1e-3, max_abs_frac=2e-3):
    """The attention-output bar: relative L2 <= 1e-3 and max |err| <= 2e-3 * max |ref|."""
    err = got.astype(np.float64) - ref
    r = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    m = np.abs(err).max() / max(np.abs(ref).max(), 1e-300)
    return r <= rel_l2 and m <= max_abs_frac, r, m

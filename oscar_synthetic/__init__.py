"""Seeded synthetic inputs for the OSCAR INT2 KV-cache decode path.

Shared by the tests, the benchmark and the oracle runs, and the only code the
two sides share.  It holds random draws and page-table layouts only, none of
the method's arithmetic (no rotation, no quantization, no attention).

Distributions (the workloads' recipe): every query/key/value channel c of
every (layer, kv head) draws sigma_c ~ U[0.5, 2]; values are N(0, sigma_c^2)
rounded to bf16.  Each kv head has 4 outlier channels (drawn without
replacement from 0..D-1) whose key and value sigma is multiplied by 20.  The
query heads of one GQA group share one query sigma profile and have no
outliers.  Calibration data for the offline rotation: 4096 queries per kv head
(pooled over its query heads) and a 1024-token calibration key/value set.

Large tensors are drawn with ``torch.randn`` from a ``torch.Generator`` on the
requested device, chunk by chunk with one seed per chunk, so that a slice can
be drawn again on its own.  CPU and CUDA generators give different streams:
a test that compares both sides hands the very same tensors to each.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional, Sequence

import numpy as np
import torch

OUTLIERS_PER_KV_HEAD = 4
OUTLIER_SCALE = 20.0
SIGMA_LO, SIGMA_HI = 0.5, 2.0
CAL_QUERIES_PER_KV_HEAD = 4096
CAL_TOKENS = 1024
ROW_CHUNK = 4096


@dataclasses.dataclass(frozen=True)
class Workload:
    """A decode-step workload: model shape, batch, context and cache layout."""
    name: str
    layers: int
    n_q_heads: int
    n_kv_heads: int
    batch: int
    context: int                     # tokens per request, current token included
    page_size: int
    group: int = 128
    head_dim: int = 128
    sink: int = 64
    recent: int = 256
    ragged: Optional[tuple] = None   # (lo, hi): per-request context ~ U{lo..hi}
    shared_prefix: int = 0           # tokens shared by all requests via page tables
    demote_per_step: bool = False    # one demotion per request/layer/kv head per step
    seed: int = 0

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    # 1 layer, 8 q / 2 kv heads, 1,024 tokens = 64 sink + 704 history + 256 recent, 16-token pages
    "tiny_gqa4_1k": Workload("tiny_gqa4_1k", 1, 8, 2, 1, 1024, 16),
    # Qwen3-8B shape, 36 layers, 32 q / 8 kv heads, batch 1, 32K context, one demotion per step
    "qwen3_8b_32k": Workload("qwen3_8b_32k", 36, 32, 8, 1, 32768, 64, demote_per_step=True),
    # Qwen3-8B shape at 100,000 tokens, whole history already INT2
    "qwen3_8b_100k": Workload("qwen3_8b_100k", 36, 32, 8, 1, 100000, 64),
    # Qwen3-8B shape, batch 32, contexts U{65536..100000}, 16K shared prefix, batched demotion
    "qwen3_8b_b32_ragged": Workload("qwen3_8b_b32_ragged", 36, 32, 8, 32, 100000, 64,
                                    ragged=(65536, 100000), shared_prefix=16384,
                                    demote_per_step=True),
    # Qwen3-32B shape, 64 layers, 64 q / 8 kv heads, batch 4, 131,072 tokens, groups of 128 / 32
    "qwen3_32b_131k_g128": Workload("qwen3_32b_131k_g128", 64, 64, 8, 4, 131072, 64, group=128),
    "qwen3_32b_131k_g32": Workload("qwen3_32b_131k_g32", 64, 64, 8, 4, 131072, 64, group=32),
}


def _seed(*parts) -> int:
    """Stable 63-bit seed from a tuple of ints/strings (blake2b of their text)."""
    h = hashlib.blake2b(repr(parts).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


@dataclasses.dataclass
class ChannelProfile:
    sigma_q: np.ndarray     # [Hkv, D] float32
    sigma_k: np.ndarray     # [Hkv, D]
    sigma_v: np.ndarray     # [Hkv, D]
    outliers: np.ndarray    # [Hkv, 4] int


def channel_profile(seed: int, layer: int, n_kv_heads: int, head_dim: int = 128) -> ChannelProfile:
    rng = np.random.default_rng(_seed("profile", seed, layer))
    sq = rng.uniform(SIGMA_LO, SIGMA_HI, size=(n_kv_heads, head_dim)).astype(np.float32)
    sk = rng.uniform(SIGMA_LO, SIGMA_HI, size=(n_kv_heads, head_dim)).astype(np.float32)
    sv = rng.uniform(SIGMA_LO, SIGMA_HI, size=(n_kv_heads, head_dim)).astype(np.float32)
    out = np.stack([rng.choice(head_dim, OUTLIERS_PER_KV_HEAD, replace=False) for _ in range(n_kv_heads)])
    for h in range(n_kv_heads):
        sk[h, out[h]] *= OUTLIER_SCALE
        sv[h, out[h]] *= OUTLIER_SCALE
    return ChannelProfile(sq, sk, sv, out)


def normal_rows(tag: str, seed: int, layer: int, start: int, stop: int, sigma: np.ndarray,
                device="cpu") -> torch.Tensor:
    """bf16 rows [stop-start, Hkv, D] ~ N(0, sigma^2), token index in [start, stop).

    Drawn in fixed chunks of ROW_CHUNK tokens with one seed per chunk, so any
    token range reproduces the same values.
    """
    Hkv, D = sigma.shape
    sig = torch.as_tensor(sigma, dtype=torch.float32, device=device)
    out = torch.empty((stop - start, Hkv, D), dtype=torch.bfloat16, device=device)
    c0 = start // ROW_CHUNK
    c1 = (stop + ROW_CHUNK - 1) // ROW_CHUNK
    for c in range(c0, c1):
        g = _gen(device, tag, seed, layer, c)
        blk = torch.randn((ROW_CHUNK, Hkv, D), generator=g, device=device, dtype=torch.float32)
        lo = max(start, c * ROW_CHUNK)
        hi = min(stop, (c + 1) * ROW_CHUNK)
        out[lo - start:hi - start] = (blk[lo - c * ROW_CHUNK:hi - c * ROW_CHUNK] * sig).to(torch.bfloat16)
    return out


def kv_rows(seed: int, layer: int, request: int, start: int, stop: int, prof: ChannelProfile,
            device="cpu", shared_prefix: int = 0):
    """(K, V) bf16 [stop-start, Hkv, D] of one request; positions below shared_prefix
    come from the stream of request 0 so that requests really share that prefix."""
    parts_k, parts_v = [], []
    if start < shared_prefix:
        e = min(stop, shared_prefix)
        parts_k.append(normal_rows("k", seed, layer * 1000003, start, e, prof.sigma_k, device))
        parts_v.append(normal_rows("v", seed, layer * 1000003, start, e, prof.sigma_v, device))
        start = e
    if start < stop:
        parts_k.append(normal_rows("k", seed, layer * 1000003 + request + 1, start, stop, prof.sigma_k, device))
        parts_v.append(normal_rows("v", seed, layer * 1000003 + request + 1, start, stop, prof.sigma_v, device))
    return torch.cat(parts_k), torch.cat(parts_v)


def queries(seed: int, layer: int, batch: int, gqa: int, prof: ChannelProfile, device="cpu",
            step: int = 0) -> torch.Tensor:
    """bf16 decode queries [B, Hq, D]; query head h belongs to kv head h // gqa."""
    Hkv, D = prof.sigma_q.shape
    g = _gen(device, "q", seed, layer, step)
    z = torch.randn((batch, Hkv, gqa, D), generator=g, device=device, dtype=torch.float32)
    sig = torch.as_tensor(prof.sigma_q, device=device)[None, :, None, :]
    return (z * sig).reshape(batch, Hkv * gqa, D).to(torch.bfloat16)


def calibration_set(seed: int, layer: int, gqa: int, prof: ChannelProfile, device="cpu"):
    """Calibration tensors of one layer: q [Hkv, 4096, D], k, v [Hkv, 1024, D] (bf16)."""
    Hkv, D = prof.sigma_q.shape
    g = _gen(device, "calq", seed, layer)
    zq = torch.randn((Hkv, CAL_QUERIES_PER_KV_HEAD, D), generator=g, device=device)
    q = (zq * torch.as_tensor(prof.sigma_q, device=device)[:, None, :]).to(torch.bfloat16)
    k = normal_rows("calk", seed, layer, 0, CAL_TOKENS, prof.sigma_k, device).transpose(0, 1).contiguous()
    v = normal_rows("calv", seed, layer, 0, CAL_TOKENS, prof.sigma_v, device).transpose(0, 1).contiguous()
    return q, k, v


def context_lengths(w: Workload) -> list:
    """Per-request context lengths (current token included)."""
    if w.ragged is None:
        return [w.context] * w.batch
    rng = np.random.default_rng(_seed("ctx", w.seed))
    lo, hi = w.ragged
    return [int(x) for x in rng.integers(lo, hi + 1, size=w.batch)]


@dataclasses.dataclass
class PageLayout:
    """Page tables of one batch (shared by all layers).

    int2_table / bf16_table: int32 [B, max_pages], logical page -> physical page
    of the INT2 / BF16 pool, -1 where the request keeps nothing in that pool.
    A logical page gets an INT2 page if it holds any position in
    [sink, context) (history, or recent positions that demotion will reach),
    and a BF16 page if it holds any position outside [sink, h_end - slack).
    Shared-prefix logical pages map to the same physical pages in every request.
    """
    int2_table: np.ndarray
    bf16_table: np.ndarray
    n_int2_pages: int
    n_bf16_pages: int
    seq_len: np.ndarray      # int32 [B]
    hist_end: np.ndarray     # int32 [B]  (context - recent, clamped to [min(sink, context), context])


def page_layout(w: Workload, seq_len: Sequence[int], bf16_slack: int = 1, shuffle: bool = True,
                hist_end: Optional[Sequence[int]] = None) -> PageLayout:
    ps = w.page_size
    B = len(seq_len)
    max_pages = max((t + ps - 1) // ps for t in seq_len)
    int2 = -np.ones((B, max_pages), dtype=np.int32)
    bf = -np.ones((B, max_pages), dtype=np.int32)
    n_int2 = n_bf = 0
    shared_pages = w.shared_prefix // ps
    if hist_end is None:
        hist_end = [min(t, max(w.sink, t - w.recent)) for t in seq_len]
    hist_end = np.asarray(hist_end, dtype=np.int32)
    for b, t in enumerate(seq_len):
        n_log = (t + ps - 1) // ps
        for lp in range(n_log):
            p0, p1 = lp * ps, min(t, (lp + 1) * ps)
            if b > 0 and lp < shared_pages:
                int2[b, lp] = int2[0, lp]
                bf[b, lp] = bf[0, lp]
                continue
            if p1 > w.sink:
                int2[b, lp] = n_int2
                n_int2 += 1
            lo_bf = max(w.sink, int(hist_end[b]) - bf16_slack)
            if p0 < w.sink or p1 > lo_bf:
                bf[b, lp] = n_bf
                n_bf += 1
    if shuffle:
        rng = np.random.default_rng(_seed("pages", w.seed, B))
        perm_i = rng.permutation(max(n_int2, 1)).astype(np.int32)
        perm_b = rng.permutation(max(n_bf, 1)).astype(np.int32)
        int2 = np.where(int2 >= 0, perm_i[np.maximum(int2, 0)], -1).astype(np.int32)
        bf = np.where(bf >= 0, perm_b[np.maximum(bf, 0)], -1).astype(np.int32)
    return PageLayout(int2, bf, n_int2, n_bf, np.asarray(seq_len, dtype=np.int32), hist_end)


def split_partials(seed: int, n_splits: int, head_dim: int = 128, empty: Sequence[int] = ()):
    """Random flash-decoding partials (m2, l, acc) for S history splits + 1 BF16 partial,
    float32, with some splits empty (m2 = -inf, l = 0, acc = 0)."""
    rng = np.random.default_rng(_seed("partials", seed, n_splits))
    S1 = n_splits + 1
    m2 = rng.normal(0.0, 8.0, size=S1).astype(np.float32)
    l = rng.uniform(1.0, 200.0, size=S1).astype(np.float32)
    acc = (rng.normal(0.0, 30.0, size=(S1, head_dim)) * l[:, None]).astype(np.float32)
    for i in empty:
        m2[i], l[i], acc[i] = -np.inf, 0.0, 0.0
    return m2, l, acc


def rotated_rows(seed: int, n: int, head_dim: int = 128, sigma: float = 3.0) -> np.ndarray:
    """float32 rows standing in for rotated keys/values (codec-only inputs), with a few
    exact ties and repeated values mixed in so that rounding edges are exercised."""
    rng = np.random.default_rng(_seed("rot", seed, n))
    x = (rng.normal(0.0, sigma, size=(n, head_dim))).astype(np.float32)
    if n > 2:
        x[1, :] = 1.5                                  # constant row
        x[2, ::2] = x[2, 0]                            # many equal values
    return x

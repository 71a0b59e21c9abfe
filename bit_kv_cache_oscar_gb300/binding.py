"""Thin ctypes binding of liboscar.so (include/oscar.h): argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors (device memory, caller-owned) and passes their addresses, sizes and the
current CUDA stream through.  No computation of the method happens here; if the
library is missing the calls raise instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liboscar.so")
_lib = None

i32 = ctypes.c_int32
vp = ctypes.c_void_p


class OscarError(RuntimeError):
    pass


class LayoutC(ctypes.Structure):
    _fields_ = [("head_dim", i32), ("n_kv_heads", i32), ("gqa", i32), ("page_size", i32),
                ("group", i32), ("sink", i32), ("recent", i32),
                ("levels_k", ctypes.c_float * 4), ("levels_v", ctypes.c_float * 4)]


class Int2PoolC(ctypes.Structure):
    _fields_ = [("codes_k", vp), ("codes_v", vp), ("scale_k", vp), ("zero_k", vp),
                ("scale_v", vp), ("zero_v", vp), ("n_pages", i32)]


class Bf16PoolC(ctypes.Structure):
    _fields_ = [("k", vp), ("v", vp), ("n_pages", i32)]


class PartialsC(ctypes.Structure):
    _fields_ = [("m", vp), ("l", vp), ("acc", vp), ("n_splits", i32)]


EXPORTS = [
    "oscar_partials_ml_floats", "oscar_partials_acc_floats", "oscar_suggest_splits", "oscar_demote",
    "oscar_quantize_rotated", "oscar_rotate_q", "oscar_decode_attention", "oscar_merge",
    "oscar_bf16_decode_attention", "oscar_get_device_status", "oscar_last_error_string", "oscar_version",
    "oscar_decode_attention_noalloc", "oscar_decode_attention_history", "oscar_decode_attention_window",
    "oscar_set_launch_overlap", "oscar_get_launch_overlap", "oscar_decode_attention_fused",
    "oscar_demote_range", "oscar_decode_attention_shared_prefix",
]


def lib():
    """Load liboscar.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OscarError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    st = ctypes.c_int
    L.oscar_partials_ml_floats.argtypes = [P(LayoutC), i32, i32]
    L.oscar_partials_ml_floats.restype = ctypes.c_size_t
    L.oscar_partials_acc_floats.argtypes = [P(LayoutC), i32, i32]
    L.oscar_partials_acc_floats.restype = ctypes.c_size_t
    L.oscar_suggest_splits.argtypes = [P(LayoutC), i32, i32, i32]
    L.oscar_suggest_splits.restype = i32
    L.oscar_demote.argtypes = [P(LayoutC), P(Bf16PoolC), vp, P(Int2PoolC), vp, i32, i32, vp, vp, i32, vp, vp,
                               ctypes.c_float, ctypes.c_float, vp, vp]
    L.oscar_demote.restype = st
    L.oscar_demote_range.argtypes = [P(LayoutC), P(Bf16PoolC), vp, P(Int2PoolC), vp, i32, i32, vp, vp, vp, vp,
                                     ctypes.c_float, ctypes.c_float, vp, vp]
    L.oscar_demote_range.restype = st
    L.oscar_quantize_rotated.argtypes = [P(LayoutC), vp, i32, ctypes.c_float, vp, vp, vp, vp]
    L.oscar_quantize_rotated.restype = st
    L.oscar_rotate_q.argtypes = [P(LayoutC), vp, vp, i32, vp, vp]
    L.oscar_rotate_q.restype = st
    L.oscar_decode_attention.argtypes = [P(LayoutC), vp, vp, P(Bf16PoolC), vp, P(Int2PoolC), vp, i32, vp, vp,
                                         i32, ctypes.c_float, P(PartialsC), vp]
    L.oscar_decode_attention.restype = st
    L.oscar_decode_attention_history.argtypes = [P(LayoutC), vp, P(Int2PoolC), vp, i32, vp, vp, i32,
                                                 ctypes.c_float, P(PartialsC), vp]
    L.oscar_decode_attention_history.restype = st
    L.oscar_decode_attention_window.argtypes = [P(LayoutC), vp, P(Bf16PoolC), vp, i32, vp, vp, i32,
                                                ctypes.c_float, P(PartialsC), vp]
    L.oscar_decode_attention_window.restype = st
    L.oscar_merge.argtypes = [P(LayoutC), P(PartialsC), vp, i32, vp, vp, vp, vp]
    L.oscar_merge.restype = st
    L.oscar_bf16_decode_attention.argtypes = [P(LayoutC), vp, P(Bf16PoolC), vp, i32, vp, i32, ctypes.c_float,
                                              P(PartialsC), vp]
    L.oscar_bf16_decode_attention.restype = st
    L.oscar_decode_attention_noalloc.argtypes = [P(LayoutC), vp, vp, P(Bf16PoolC), vp, P(Int2PoolC), vp, i32, vp,
                                                 vp, i32, ctypes.c_float, i32, vp, vp, vp, vp, vp]
    L.oscar_decode_attention_noalloc.restype = st
    L.oscar_get_device_status.argtypes = [P(i32), vp]
    L.oscar_get_device_status.restype = st
    L.oscar_last_error_string.argtypes = []
    L.oscar_last_error_string.restype = ctypes.c_char_p
    L.oscar_version.argtypes = []
    L.oscar_version.restype = ctypes.c_char_p
    L.oscar_decode_attention_fused.argtypes = [P(LayoutC), vp, vp, P(Bf16PoolC), vp, P(Int2PoolC), vp, i32, vp,
                                               vp, i32, ctypes.c_float, P(PartialsC), vp, vp, ctypes.c_float,
                                               ctypes.c_float, vp, vp, vp, vp, vp, vp]
    L.oscar_decode_attention_fused.restype = st
    L.oscar_decode_attention_shared_prefix.argtypes = [P(LayoutC), vp, vp, P(Bf16PoolC), vp, P(Int2PoolC), vp,
                                                        i32, vp, vp, i32, ctypes.c_float, i32, i32, P(PartialsC),
                                                        vp, vp]
    L.oscar_decode_attention_shared_prefix.restype = st
    L.oscar_set_launch_overlap.argtypes = [i32]
    L.oscar_set_launch_overlap.restype = st
    L.oscar_get_launch_overlap.argtypes = []
    L.oscar_get_launch_overlap.restype = i32
    _lib = L
    return L


def _check(name: str, status: int):
    if status != 0:
        raise OscarError(f"{name} failed ({status}): {lib().oscar_last_error_string().decode()}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise OscarError("tensor arguments must be contiguous")
    return vp(t.data_ptr())


def _stream(stream) -> vp:
    if stream is None:
        stream = torch.cuda.current_stream()
    return vp(stream.cuda_stream)


@dataclasses.dataclass(frozen=True)
class Layout:
    n_kv_heads: int
    gqa: int
    page_size: int
    group: int = 128
    sink: int = 64
    recent: int = 256
    head_dim: int = 128
    levels_k: Optional[tuple] = None    # key codebook (4 increasing levels), None = uniform
    levels_v: Optional[tuple] = None    # value codebook

    @property
    def n_q_heads(self) -> int:
        return self.n_kv_heads * self.gqa

    def c(self) -> LayoutC:
        lay = LayoutC(self.head_dim, self.n_kv_heads, self.gqa, self.page_size, self.group, self.sink,
                      self.recent)
        if self.levels_k is not None or self.levels_v is not None:
            lay.levels_k = (ctypes.c_float * 4)(*[float(x) for x in self.levels_k])
            lay.levels_v = (ctypes.c_float * 4)(*[float(x) for x in self.levels_v])
        return lay


@dataclasses.dataclass
class Int2Pool:
    """Paged INT2 pool of one layer; bf16 scale/zero stored as torch.bfloat16."""
    codes_k: torch.Tensor
    codes_v: torch.Tensor
    scale_k: torch.Tensor
    zero_k: torch.Tensor
    scale_v: torch.Tensor
    zero_v: torch.Tensor

    @property
    def n_pages(self) -> int:
        return self.codes_k.shape[0]

    @staticmethod
    def empty(layout: Layout, n_pages: int, device="cuda") -> "Int2Pool":
        ps, H, D, g = layout.page_size, layout.n_kv_heads, layout.head_dim, layout.group
        c = lambda: torch.zeros((n_pages, ps, H, D // 4), dtype=torch.uint8, device=device)
        s = lambda: torch.zeros((n_pages, ps, H, D // g), dtype=torch.bfloat16, device=device)
        return Int2Pool(c(), c(), s(), s(), s(), s())

    def c(self) -> Int2PoolC:
        return Int2PoolC(*(_ptr(t) for t in (self.codes_k, self.codes_v, self.scale_k, self.zero_k,
                                             self.scale_v, self.zero_v)), self.n_pages)


@dataclasses.dataclass
class Bf16Pool:
    k: torch.Tensor   # bf16 [n_pages, page_size, Hkv, D]
    v: torch.Tensor

    @property
    def n_pages(self) -> int:
        return self.k.shape[0]

    @staticmethod
    def empty(layout: Layout, n_pages: int, device="cuda") -> "Bf16Pool":
        shp = (n_pages, layout.page_size, layout.n_kv_heads, layout.head_dim)
        return Bf16Pool(torch.zeros(shp, dtype=torch.bfloat16, device=device),
                        torch.zeros(shp, dtype=torch.bfloat16, device=device))

    def c(self) -> Bf16PoolC:
        return Bf16PoolC(_ptr(self.k), _ptr(self.v), self.n_pages)


@dataclasses.dataclass
class Partials:
    m: torch.Tensor     # fp32 [B, Hq, S+1]
    l: torch.Tensor
    acc: torch.Tensor   # fp32 [B, Hq, S+1, D]
    n_splits: int

    @staticmethod
    def empty(layout: Layout, batch: int, n_splits: int, device="cuda") -> "Partials":
        shp = (batch, layout.n_q_heads, n_splits + 1)
        return Partials(torch.empty(shp, dtype=torch.float32, device=device),
                        torch.empty(shp, dtype=torch.float32, device=device),
                        torch.empty(shp + (layout.head_dim,), dtype=torch.float32, device=device), n_splits)

    def c(self) -> PartialsC:
        return PartialsC(_ptr(self.m), _ptr(self.l), _ptr(self.acc), self.n_splits)


def oscar_partials_ml_floats(layout: Layout, batch: int, n_splits: int) -> int:
    return int(lib().oscar_partials_ml_floats(ctypes.byref(layout.c()), batch, n_splits))


def oscar_partials_acc_floats(layout: Layout, batch: int, n_splits: int) -> int:
    return int(lib().oscar_partials_acc_floats(ctypes.byref(layout.c()), batch, n_splits))


def oscar_suggest_splits(layout: Layout, batch: int, max_hist_tokens: int, sm_count: int) -> int:
    return int(lib().oscar_suggest_splits(ctypes.byref(layout.c()), batch, max_hist_tokens, sm_count))


def oscar_demote(layout: Layout, src: Bf16Pool, bf16_page_table: torch.Tensor, dst: Int2Pool,
                 int2_page_table: torch.Tensor, req_idx: torch.Tensor, positions: torch.Tensor,
                 R_K: torch.Tensor, R_V: torch.Tensor, c_K: float, c_V: float,
                 rotated_out: Optional[torch.Tensor] = None, stream=None):
    if bf16_page_table.shape != int2_page_table.shape:
        raise OscarError("oscar_demote: both page tables must be [batch, max_pages]")
    batch, max_pages = int2_page_table.shape
    _check("oscar_demote", lib().oscar_demote(
        ctypes.byref(layout.c()), ctypes.byref(src.c()), _ptr(bf16_page_table), ctypes.byref(dst.c()),
        _ptr(int2_page_table), max_pages, batch, _ptr(req_idx), _ptr(positions), int(positions.numel()),
        _ptr(R_K), _ptr(R_V), float(c_K), float(c_V), _ptr(rotated_out), _stream(stream)))


def oscar_demote_range(layout: Layout, src: Bf16Pool, bf16_page_table: torch.Tensor, dst: Int2Pool,
                       int2_page_table: torch.Tensor, pos_begin: torch.Tensor, pos_end: torch.Tensor,
                       R_K: torch.Tensor, R_V: torch.Tensor, c_K: float, c_V: float,
                       rotated_out: Optional[torch.Tensor] = None, stream=None):
    if bf16_page_table.shape != int2_page_table.shape:
        raise OscarError("oscar_demote_range: both page tables must be [batch, max_pages]")
    batch, max_pages = int2_page_table.shape
    if pos_begin.numel() != batch or pos_end.numel() != batch:
        raise OscarError("oscar_demote_range: pos_begin and pos_end need one entry per request")
    _check("oscar_demote_range", lib().oscar_demote_range(
        ctypes.byref(layout.c()), ctypes.byref(src.c()), _ptr(bf16_page_table), ctypes.byref(dst.c()),
        _ptr(int2_page_table), max_pages, batch, _ptr(pos_begin), _ptr(pos_end), _ptr(R_K), _ptr(R_V),
        float(c_K), float(c_V), _ptr(rotated_out), _stream(stream)))


def oscar_quantize_rotated(layout: Layout, x_rot: torch.Tensor, clip: float, codes: torch.Tensor,
                           scale: torch.Tensor, zero: torch.Tensor, stream=None):
    n = x_rot.numel() // layout.head_dim
    _check("oscar_quantize_rotated", lib().oscar_quantize_rotated(
        ctypes.byref(layout.c()), _ptr(x_rot), n, float(clip), _ptr(codes), _ptr(scale), _ptr(zero),
        _stream(stream)))


def oscar_rotate_q(layout: Layout, q: torch.Tensor, R_K: torch.Tensor, q_rot: torch.Tensor, stream=None):
    _check("oscar_rotate_q", lib().oscar_rotate_q(
        ctypes.byref(layout.c()), _ptr(q), _ptr(R_K), int(q.shape[0]), _ptr(q_rot), _stream(stream)))


def oscar_decode_attention(layout: Layout, q: torch.Tensor, q_rot: torch.Tensor, bf16_pool: Bf16Pool,
                           bf16_page_table: torch.Tensor, int2_pool: Int2Pool, int2_page_table: torch.Tensor,
                           seq_len: torch.Tensor, hist_end: torch.Tensor, sm_scale: float, partials: Partials,
                           stream=None):
    _check("oscar_decode_attention", lib().oscar_decode_attention(
        ctypes.byref(layout.c()), _ptr(q), _ptr(q_rot), ctypes.byref(bf16_pool.c()), _ptr(bf16_page_table),
        ctypes.byref(int2_pool.c()), _ptr(int2_page_table), int(int2_page_table.shape[-1]), _ptr(seq_len),
        _ptr(hist_end), int(q.shape[0]), float(sm_scale), ctypes.byref(partials.c()), _stream(stream)))


def oscar_decode_attention_shared_prefix(layout: Layout, q: torch.Tensor, q_rot: torch.Tensor, bf16_pool: Bf16Pool,
                                         bf16_page_table: torch.Tensor, int2_pool: Int2Pool,
                                         int2_page_table: torch.Tensor, seq_len: torch.Tensor, hist_end: torch.Tensor,
                                         sm_scale: float, prefix_end: int, prefix_splits: int, partials: Partials,
                                         tile_counters: Optional[torch.Tensor] = None, stream=None):
    """Shared prefix [sink, prefix_end) once for the whole batch (slots 0 .. prefix_splits - 1), each
    request's own history after it (slots prefix_splits .. S - 1) and its BF16 window (slot S)."""
    _check("oscar_decode_attention_shared_prefix", lib().oscar_decode_attention_shared_prefix(
        ctypes.byref(layout.c()), _ptr(q), _ptr(q_rot), ctypes.byref(bf16_pool.c()), _ptr(bf16_page_table),
        ctypes.byref(int2_pool.c()), _ptr(int2_page_table), int(int2_page_table.shape[-1]), _ptr(seq_len),
        _ptr(hist_end), int(q.shape[0]), float(sm_scale), int(prefix_end), int(prefix_splits),
        ctypes.byref(partials.c()), _ptr(tile_counters), _stream(stream)))


def oscar_decode_attention_fused(layout: Layout, q: torch.Tensor, R_K: torch.Tensor, bf16_pool: Bf16Pool,
                                 bf16_page_table: torch.Tensor, int2_pool: Int2Pool, int2_page_table: torch.Tensor,
                                 seq_len: torch.Tensor, hist_end: torch.Tensor, sm_scale: float, partials: Partials,
                                 demote_pos: Optional[torch.Tensor] = None, R_V: Optional[torch.Tensor] = None,
                                 c_K: float = 0.0, c_V: float = 0.0, out: Optional[torch.Tensor] = None,
                                 out_f32: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                                 merge_counters: Optional[torch.Tensor] = None,
                                 tile_counters: Optional[torch.Tensor] = None, stream=None):
    """oscar_decode_attention with q . R_K computed inside the launch (same partials bits); with
    demote_pos ([batch] int32, -1 = none) also the per-step demotion of those positions; with
    out / out_f32 also oscar_merge's output, from a second launch that starts each request's
    merge on its arrival count when merge_counters (int32 zeros [2 * batch]) is given; with
    tile_counters (int32 zeros [2 * batch]) the history CTAs take 64-token units dynamically."""
    for name, t in (("merge_counters", merge_counters), ("tile_counters", tile_counters)):
        if t is not None and t.numel() < 2 * int(q.shape[0]):
            raise OscarError(f"oscar_decode_attention_fused: {name} needs 2 * batch int32 entries")
    _check("oscar_decode_attention_fused", lib().oscar_decode_attention_fused(
        ctypes.byref(layout.c()), _ptr(q), _ptr(R_K), ctypes.byref(bf16_pool.c()), _ptr(bf16_page_table),
        ctypes.byref(int2_pool.c()), _ptr(int2_page_table), int(int2_page_table.shape[-1]), _ptr(seq_len),
        _ptr(hist_end), int(q.shape[0]), float(sm_scale), ctypes.byref(partials.c()),
        _ptr(demote_pos) if demote_pos is not None else None, _ptr(R_V) if R_V is not None else None,
        float(c_K), float(c_V), _ptr(out) if out is not None else None,
        _ptr(out_f32) if out_f32 is not None else None, _ptr(lse) if lse is not None else None,
        _ptr(merge_counters) if merge_counters is not None else None,
        _ptr(tile_counters) if tile_counters is not None else None, _stream(stream)))


def oscar_decode_attention_history(layout: Layout, q_rot: torch.Tensor, int2_pool: Int2Pool,
                                   int2_page_table: torch.Tensor, seq_len: torch.Tensor, hist_end: torch.Tensor,
                                   sm_scale: float, partials: Partials, stream=None):
    _check("oscar_decode_attention_history", lib().oscar_decode_attention_history(
        ctypes.byref(layout.c()), _ptr(q_rot), ctypes.byref(int2_pool.c()), _ptr(int2_page_table),
        int(int2_page_table.shape[-1]), _ptr(seq_len), _ptr(hist_end), int(q_rot.shape[0]), float(sm_scale),
        ctypes.byref(partials.c()), _stream(stream)))


def oscar_decode_attention_window(layout: Layout, q: torch.Tensor, bf16_pool: Bf16Pool,
                                  bf16_page_table: torch.Tensor, seq_len: torch.Tensor, hist_end: torch.Tensor,
                                  sm_scale: float, partials: Partials, stream=None):
    _check("oscar_decode_attention_window", lib().oscar_decode_attention_window(
        ctypes.byref(layout.c()), _ptr(q), ctypes.byref(bf16_pool.c()), _ptr(bf16_page_table),
        int(bf16_page_table.shape[-1]), _ptr(seq_len), _ptr(hist_end), int(q.shape[0]), float(sm_scale),
        ctypes.byref(partials.c()), _stream(stream)))


def oscar_merge(layout: Layout, partials: Partials, R_V: Optional[torch.Tensor], out: Optional[torch.Tensor],
                out_f32: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None):
    batch = int((out if out is not None else out_f32).shape[0])
    _check("oscar_merge", lib().oscar_merge(
        ctypes.byref(layout.c()), ctypes.byref(partials.c()), _ptr(R_V), batch, _ptr(out), _ptr(out_f32),
        _ptr(lse), _stream(stream)))


def oscar_bf16_decode_attention(layout: Layout, q: torch.Tensor, pool: Bf16Pool, page_table: torch.Tensor,
                                seq_len: torch.Tensor, sm_scale: float, partials: Partials, stream=None):
    _check("oscar_bf16_decode_attention", lib().oscar_bf16_decode_attention(
        ctypes.byref(layout.c()), _ptr(q), ctypes.byref(pool.c()), _ptr(page_table), int(page_table.shape[-1]),
        _ptr(seq_len), int(q.shape[0]), float(sm_scale), ctypes.byref(partials.c()), _stream(stream)))


def oscar_decode_attention_noalloc(layout: Layout, q: torch.Tensor, q_rot: torch.Tensor, bf16_pool: Bf16Pool,
                                   bf16_page_table: torch.Tensor, int2_pool: Int2Pool,
                                   int2_page_table: torch.Tensor, seq_len: torch.Tensor, hist_end: torch.Tensor,
                                   sm_scale: float, n_splits: int, R_V: torch.Tensor,
                                   out: Optional[torch.Tensor], out_f32: Optional[torch.Tensor] = None,
                                   lse: Optional[torch.Tensor] = None, stream=None):
    """Decode attention + merge with the partials in the library's own device array (no caller scratch)."""
    _check("oscar_decode_attention_noalloc", lib().oscar_decode_attention_noalloc(
        ctypes.byref(layout.c()), _ptr(q), _ptr(q_rot), ctypes.byref(bf16_pool.c()), _ptr(bf16_page_table),
        ctypes.byref(int2_pool.c()), _ptr(int2_page_table), int(int2_page_table.shape[-1]), _ptr(seq_len),
        _ptr(hist_end), int(q.shape[0]), float(sm_scale), int(n_splits), _ptr(R_V), _ptr(out), _ptr(out_f32),
        _ptr(lse), _stream(stream)))


def oscar_get_device_status(stream=None) -> int:
    out = i32(0)
    _check("oscar_get_device_status", lib().oscar_get_device_status(ctypes.byref(out), _stream(stream)))
    return int(out.value)


def oscar_version() -> str:
    return lib().oscar_version().decode()


def oscar_set_launch_overlap(enabled: bool) -> None:
    """Programmatic dependent launch between consecutive decode kernels (see oscar.h for the
    caller's guarantee: the kernel before a decode call writes no pool, table, length or R)."""
    _check("oscar_set_launch_overlap", lib().oscar_set_launch_overlap(1 if enabled else 0))


def oscar_get_launch_overlap() -> bool:
    return bool(lib().oscar_get_launch_overlap())

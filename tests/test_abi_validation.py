"""Host-side argument checks of every entry point of the C ABI, without a GPU.

Each case below is rejected (or, with zero work, accepted as a no-op) before the
library makes any CUDA call, so it needs no device.  Most cases pass placeholder
addresses for the arrays that earlier checks want non-NULL and 16-byte aligned;
those cases run only where no GPU is visible, so that a reordering of the checks
could never hand such an address to a kernel.
"""
import ctypes

import pytest
import torch

from bit_kv_cache_oscar_gb300 import binding as ob
from bit_kv_cache_oscar_gb300 import build

OK, INVALID, UNSUPPORTED = 0, 1, 2
FAKE = 0x7F0000000000          # 16-byte aligned placeholder address (never dereferenced)
MISALIGNED = FAKE + 8

no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="placeholder addresses: host-only case")


@pytest.fixture(scope="module")
def L():
    build.build()
    return ob.lib()


def layout(n_kv=8, gqa=4):
    return ob.LayoutC(128, n_kv, gqa, 64, 128, 64, 256)


def int2_pool(n_pages=4, addr=FAKE):
    return ob.Int2PoolC(addr, addr, addr, addr, addr, addr, n_pages)


def bf16_pool(n_pages=4, addr=FAKE):
    return ob.Bf16PoolC(addr, addr, n_pages)


def partials(n_splits=4):
    return ob.PartialsC(FAKE, FAKE, FAKE, n_splits)


def err(L):
    return L.oscar_last_error_string().decode()


def demote(L, lay=None, src=None, dst=None, bpt=FAKE, ipt=FAKE, max_pages=4, batch=1, req=FAKE, pos=FAKE, n=1,
           RK=FAKE, RV=FAKE, cK=0.96, cV=0.92):
    lay = lay or layout()
    src = src or bf16_pool()
    dst = dst or int2_pool()
    return L.oscar_demote(ctypes.byref(lay), ctypes.byref(src), bpt, ctypes.byref(dst), ipt, max_pages, batch, req,
                          pos, n, RK, RV, cK, cV, None, None)


def test_null_layout_everywhere(L):
    assert L.oscar_demote(None, None, None, None, None, 1, 1, None, None, 1, None, None, 0.96, 0.92, None,
                          None) == INVALID
    assert "layout is NULL" in err(L)
    assert L.oscar_rotate_q(None, None, None, 1, None, None) == INVALID
    assert L.oscar_merge(None, None, None, 1, None, None, None, None) == INVALID
    assert L.oscar_decode_attention_noalloc(None, None, None, None, None, None, None, 1, None, None, 1, 0.1, 4,
                                            None, None, None, None, None) == INVALID
    assert "layout is NULL" in err(L)


@no_gpu
def test_null_pools_and_partials(L):
    lay = layout()
    assert L.oscar_demote(ctypes.byref(lay), None, None, None, None, 1, 1, None, None, 1, None, None, 0.96, 0.92,
                          None, None) == INVALID
    assert "BF16 pool is NULL" in err(L)
    src = bf16_pool()
    assert L.oscar_demote(ctypes.byref(lay), ctypes.byref(src), None, None, None, 1, 1, None, None, 1, None, None,
                          0.96, 0.92, None, None) == INVALID
    assert "INT2 pool is NULL" in err(L)
    i2 = int2_pool()
    assert L.oscar_decode_attention_history(ctypes.byref(lay), None, ctypes.byref(i2), None, 1, None, None, 1, 0.1,
                                            None, None) == INVALID
    assert "partials is NULL" in err(L)


@no_gpu
@pytest.mark.parametrize("pool,msg", [
    (lambda: ob.Int2PoolC(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4), "NULL array"),
    (lambda: int2_pool(addr=MISALIGNED), "16-byte aligned"),
    (lambda: int2_pool(n_pages=0), "n_pages"),
])
def test_int2_pool_checks(L, pool, msg):
    lay, src, dst = layout(), bf16_pool(), pool()
    assert L.oscar_demote(ctypes.byref(lay), ctypes.byref(src), None, ctypes.byref(dst), None, 1, 1, None, None, 1,
                          None, None, 0.96, 0.92, None, None) == INVALID
    assert msg in err(L)


@no_gpu
@pytest.mark.parametrize("pool,msg", [
    (lambda: ob.Bf16PoolC(FAKE, None, 4), "NULL array"),
    (lambda: bf16_pool(addr=MISALIGNED), "16-byte aligned"),
    (lambda: bf16_pool(n_pages=0), "n_pages"),
])
def test_bf16_pool_checks(L, pool, msg):
    lay, src = layout(), pool()
    assert L.oscar_bf16_decode_attention(ctypes.byref(lay), None, ctypes.byref(src), None, 1, None, 1, 0.1, None,
                                         None) == INVALID
    assert msg in err(L)


@no_gpu
@pytest.mark.parametrize("part,msg", [
    (lambda: ob.PartialsC(FAKE, None, FAKE, 4), "NULL array"),
    (lambda: ob.PartialsC(FAKE, FAKE, MISALIGNED, 4), "16-byte aligned"),
    (lambda: partials(0), "n_splits"),
    (lambda: partials(1025), "n_splits"),
])
def test_partials_checks(L, part, msg):
    lay, p = layout(), part()
    assert L.oscar_merge(ctypes.byref(lay), ctypes.byref(p), None, 1, FAKE, None, None, None) == INVALID
    assert msg in err(L)


@no_gpu
def test_zero_work_is_a_no_op(L):
    lay, src, dst, p = layout(), bf16_pool(), int2_pool(), partials()
    assert demote(L, n=0) == OK
    assert L.oscar_demote_range(ctypes.byref(lay), ctypes.byref(src), None, ctypes.byref(dst), None, 1, 0, None,
                                None, None, None, 0.96, 0.92, None, None) == OK
    assert L.oscar_rotate_q(ctypes.byref(lay), None, None, 0, None, None) == OK
    assert L.oscar_decode_attention(ctypes.byref(lay), None, None, ctypes.byref(src), None, ctypes.byref(dst), None,
                                    1, None, None, 0, 0.1, ctypes.byref(p), None) == OK
    assert L.oscar_decode_attention_fused(ctypes.byref(lay), None, None, ctypes.byref(src), None, ctypes.byref(dst),
                                          None, 1, None, None, 0, 0.1, ctypes.byref(p), None, None, 0.96, 0.92,
                                          None, None, None, None, None, None) == OK
    assert L.oscar_merge(ctypes.byref(lay), ctypes.byref(p), None, 0, None, None, None, None) == OK
    assert L.oscar_bf16_decode_attention(ctypes.byref(lay), None, ctypes.byref(src), None, 1, None, 0, 0.1,
                                         ctypes.byref(p), None) == OK
    assert L.oscar_decode_attention_noalloc(ctypes.byref(lay), None, None, None, None, None, None, 1, None, None, 0,
                                            0.1, 4, None, None, None, None, None) == OK


@no_gpu
def test_batch_and_count_ranges(L):
    lay, src, dst, p = layout(), bf16_pool(), int2_pool(), partials()
    assert demote(L, n=-1) == INVALID and "n -1" in err(L)
    assert demote(L, n=65535 * 256 + 1) == INVALID
    assert L.oscar_demote_range(ctypes.byref(lay), ctypes.byref(src), None, ctypes.byref(dst), None, 1, 65536, None,
                                None, None, None, 0.96, 0.92, None, None) == INVALID
    assert L.oscar_rotate_q(ctypes.byref(lay), None, None, -1, None, None) == INVALID
    assert L.oscar_merge(ctypes.byref(lay), ctypes.byref(p), None, 65536, FAKE, None, None, None) == INVALID
    assert L.oscar_bf16_decode_attention(ctypes.byref(lay), None, ctypes.byref(src), None, 1, None, -1, 0.1,
                                         ctypes.byref(p), None) == INVALID
    assert L.oscar_decode_attention_fused(ctypes.byref(lay), None, None, ctypes.byref(src), None, ctypes.byref(dst),
                                          None, 1, None, None, 65536, 0.1, ctypes.byref(p), None, None, 0.96, 0.92,
                                          None, None, None, None, None, None) == INVALID
    for n_splits in (0, 1025):
        assert L.oscar_decode_attention_noalloc(ctypes.byref(lay), None, None, None, None, None, None, 1, None,
                                                None, 1, 0.1, n_splits, None, None, None, None, None) == INVALID


@no_gpu
def test_null_arguments_after_the_pools(L):
    lay, src, dst, p = layout(), bf16_pool(), int2_pool(), partials()
    assert demote(L, bpt=None) == INVALID and "NULL page table" in err(L)
    assert L.oscar_demote_range(ctypes.byref(lay), ctypes.byref(src), None, ctypes.byref(dst), FAKE, 1, 1, FAKE,
                                FAKE, FAKE, None, 0.96, 0.92, None, None) == INVALID
    assert L.oscar_rotate_q(ctypes.byref(lay), FAKE, None, 1, FAKE, None) == INVALID
    assert L.oscar_decode_attention(ctypes.byref(lay), None, FAKE, ctypes.byref(src), FAKE, ctypes.byref(dst), FAKE,
                                    1, FAKE, FAKE, 1, 0.1, ctypes.byref(p), None) == INVALID
    assert L.oscar_decode_attention_window(ctypes.byref(lay), FAKE, ctypes.byref(src), FAKE, 1, None, FAKE, 1, 0.1,
                                           ctypes.byref(p), None) == INVALID
    assert L.oscar_merge(ctypes.byref(lay), ctypes.byref(p), None, 1, None, None, None, None) == INVALID
    assert "both NULL" in err(L)
    assert L.oscar_get_device_status(None, None) == INVALID


@no_gpu
def test_late_checks_of_oscar_demote(L):
    assert demote(L, max_pages=0) == INVALID and "max_pages_per_req" in err(L)
    assert demote(L, batch=0) == INVALID and "batch 0" in err(L)
    assert demote(L, RK=MISALIGNED) == INVALID and "R_K/R_V" in err(L)
    assert demote(L, RV=MISALIGNED) == INVALID and "R_K/R_V" in err(L)
    assert demote(L, cK=0.0) == INVALID and "clip" in err(L)
    assert demote(L, cV=-1.0) == INVALID and "clip" in err(L)
    assert demote(L, cK=float("nan")) == INVALID


@no_gpu
def test_late_checks_of_the_decode_calls(L):
    lay, src, dst, p = layout(), bf16_pool(), int2_pool(), partials()
    # misaligned q_rot / q
    assert L.oscar_decode_attention(ctypes.byref(lay), FAKE, MISALIGNED, ctypes.byref(src), FAKE, ctypes.byref(dst),
                                    FAKE, 1, FAKE, FAKE, 1, 0.1, ctypes.byref(p), None) == INVALID
    assert "not 16-byte aligned" in err(L)
    assert L.oscar_decode_attention(ctypes.byref(lay), FAKE, FAKE, ctypes.byref(src), FAKE, ctypes.byref(dst), FAKE,
                                    0, FAKE, FAKE, 1, 0.1, ctypes.byref(p), None) == INVALID
    assert "max_pages_per_req" in err(L)
    assert L.oscar_decode_attention_history(ctypes.byref(lay), MISALIGNED, ctypes.byref(dst), FAKE, 1, FAKE, FAKE,
                                            1, 0.1, ctypes.byref(p), None) == INVALID
    # the fused launch: kv head counts outside 1, 2, 4, 8, and a misaligned R_V
    lay3 = layout(n_kv=3)
    assert L.oscar_decode_attention_fused(ctypes.byref(lay3), FAKE, FAKE, ctypes.byref(src), FAKE,
                                          ctypes.byref(dst), FAKE, 1, FAKE, FAKE, 1, 0.1, ctypes.byref(p), None,
                                          None, 0.96, 0.92, None, None, None, None, None, None) == UNSUPPORTED
    assert L.oscar_decode_attention_fused(ctypes.byref(lay), FAKE, FAKE, ctypes.byref(src), FAKE, ctypes.byref(dst),
                                          FAKE, 1, FAKE, FAKE, 1, 0.1, ctypes.byref(p), None, MISALIGNED, 0.96,
                                          0.92, None, None, None, None, None, None) == INVALID
    assert "R_V" in err(L)
    # bulk demotion: a misaligned rotated_out
    assert L.oscar_demote_range(ctypes.byref(lay), ctypes.byref(src), FAKE, ctypes.byref(dst), FAKE, 1, 1, FAKE,
                                FAKE, FAKE, FAKE, 0.96, 0.92, MISALIGNED, None) == INVALID
    assert "rotated_out" in err(L)
    assert L.oscar_demote_range(ctypes.byref(lay), ctypes.byref(src), FAKE, ctypes.byref(dst), FAKE, 1, 1, FAKE,
                                FAKE, FAKE, FAKE, 0.0, 0.92, None, None) == INVALID


def test_launch_overlap_switch(L):
    before = L.oscar_get_launch_overlap()
    try:
        assert L.oscar_set_launch_overlap(1) == OK and L.oscar_get_launch_overlap() == 1
        assert L.oscar_set_launch_overlap(0) == OK and L.oscar_get_launch_overlap() == 0
    finally:
        L.oscar_set_launch_overlap(before)

"""OSCAR INT2 KV-cache decode path for GB300 (sm_103a).

The compute lives in liboscar.so (hand-written CUDA behind the C ABI of
include/oscar.h); ``binding`` is the ctypes layer with the same entry-point
names.  Build the library with ``__graft_entry__.build()`` or
``python -m bit_kv_cache_oscar_gb300.build``.
"""
from .binding import (  # noqa: F401
    Bf16Pool, Int2Pool, Layout, OscarError, Partials, oscar_bf16_decode_attention, oscar_decode_attention,
    oscar_demote, oscar_get_device_status, oscar_merge, oscar_partials_acc_floats, oscar_partials_ml_floats,
    oscar_quantize_rotated, oscar_rotate_q, oscar_suggest_splits, oscar_version,
)

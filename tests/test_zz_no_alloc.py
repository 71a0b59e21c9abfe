"""oscar_decode_attention_noalloc: decode attention + merge without caller scratch.

Some callers cannot allocate device memory (a host framework that owns every
allocation and offers no workspace, or a loop that must never call an
allocator).  This entry point keeps the split partials in a device array owned
by the library.  The test calls it through the C ABI twice in a row, on two
different inputs, and compares each output with the regular path
(oscar_decode_attention into caller-allocated partials, then oscar_merge),
within the attention-output tolerance used by the other parity tests.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_oscar_gb300 import binding as ob
from tests import scenario as sc

pytestmark = pytest.mark.gpu
D = 128


def _regular_and_noalloc(case, n_splits):
    L, dev = case.layout, case.dev
    B = len(case.seq)
    q_rot = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    ob.oscar_rotate_q(L, dev["q"], dev["RK"], q_rot)
    part = ob.Partials.empty(L, B, n_splits)
    ob.oscar_decode_attention(L, dev["q"], q_rot, dev["bf16"], dev["bf16_table"], dev["int2"], dev["int2_table"],
                              dev["seq_len"], dev["hist_end"], case.sm_scale, part)
    ref = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    ob.oscar_merge(L, part, dev["RV"], None, ref)
    got = torch.full((B, L.n_q_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    got_bf = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    ob.oscar_decode_attention_noalloc(L, dev["q"], q_rot, dev["bf16"], dev["bf16_table"], dev["int2"],
                                      dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, n_splits,
                                      dev["RV"], got_bf, got)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), got.cpu().numpy(), got_bf


def test_noalloc_matches_regular_path_twice():
    cases = [sc.make_case(n_kv=2, gqa=4, page_size=16, seq=(1024, 640)),
             sc.make_case(n_kv=8, gqa=4, page_size=64, seq=(3000,), seed=1)]
    for case, S in zip(cases, (5, 12)):
        sc.upload(case)
        ref, got, got_bf = _regular_and_noalloc(case, S)
        ok, r, m = sc.tolerance_ok(got.reshape(-1, D), ref.reshape(-1, D).astype(np.float64))
        assert ok, f"rel-L2 {r:.3e}, max-abs frac {m:.3e}"
        assert torch.equal(got_bf.float().cpu(), torch.from_numpy(got).to(torch.bfloat16).float())
        assert ob.oscar_get_device_status() == 0


def test_noalloc_rejects_oversized_request():
    case = sc.make_case(n_kv=8, gqa=8, page_size=64, seq=(1024,))
    sc.upload(case, demote_history=False)
    L, dev = case.layout, case.dev
    B = 16
    q = torch.zeros((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    q_rot = torch.zeros((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    out = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ob.OscarError, match="too large for the no-alloc scratch"):
        ob.oscar_decode_attention_noalloc(L, q, q_rot, dev["bf16"], dev["bf16_table"], dev["int2"],
                                          dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, 256,
                                          dev["RV"], out)

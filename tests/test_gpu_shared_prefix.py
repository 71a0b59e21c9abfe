"""Shared-prefix (cascade) decode attention against the oracle.

Requests share the INT2 pages of a prefix through their page tables (oscar_synthetic draws the
same prefix rows for every request and page_layout points the prefix pages of every request at
request 0's).  oscar_decode_attention_shared_prefix reads the prefix once for the batch on the
tensor cores (slots 0 .. prefix_splits - 1), each request's own history after it and its BF16
window; merged, the outputs must meet the attention bar against the oracle's attention over the
whole context, and each prefix slot must equal the oracle's partial over its token range.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_oscar_gb300 import binding as ob
from tests import scenario as sc
from tests.helpers import bf16_bits
from tests.test_gpu_parity import _check_outputs

pytestmark = pytest.mark.gpu

D = 128


def _run(case, prefix, S, prefix_splits, dynamic):
    L, dev = case.layout, case.dev
    B = len(case.seq)
    q_rot = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    ob.oscar_rotate_q(L, dev["q"], dev["RK"], q_rot)
    part = ob.Partials.empty(L, B, S)
    tiles = torch.zeros(2 * B, dtype=torch.int32, device="cuda") if dynamic else None
    ob.oscar_decode_attention_shared_prefix(L, dev["q"], q_rot, dev["bf16"], dev["bf16_table"], dev["int2"],
                                            dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale,
                                            prefix, prefix_splits, part, tile_counters=tiles)
    out = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, L.n_q_heads), dtype=torch.float32, device="cuda")
    ob.oscar_merge(L, part, dev["RV"], out, out32, lse)
    torch.cuda.synchronize()
    assert tiles is None or not tiles.any()
    assert ob.oscar_get_device_status() == 0
    return out, out32, lse, part


@pytest.mark.parametrize("n_kv,gqa,ps,seq,prefix,S,ps_splits,dynamic", [
    (8, 4, 64, (3000, 2500, 2200, 2900), 1024, 6, 2, False),    # the batch-32 shape's heads, 4 requests
    (8, 4, 64, (2600, 3100, 2400), 1536, 5, 3, True),
    (2, 8, 16, (1500,) * 20, 768, 4, 3, False),                 # 160 query rows: two request groups
    (4, 2, 32, (2000, 1800, 2600), 960, 5, 1, True),            # prefix end not on a page of 64
])
def test_shared_prefix_matches_oracle(n_kv, gqa, ps, seq, prefix, S, ps_splits, dynamic):
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=128, seq=seq, shared_prefix=prefix)
    sc.upload(case)
    assert all(int(h) >= prefix for h in case.hist_end)
    out, out32, lse, part = _run(case, prefix, S, ps_splits, dynamic)
    _check_outputs(case, out, out32, lse)


def test_shared_prefix_slots_are_the_prefix_partials():
    """Each prefix slot is the partial over its 128-token-tile range of [sink, prefix_end)."""
    n_kv, gqa, prefix, S, ps_splits = 8, 4, 1024, 6, 3
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=64, group=128, seq=(2200, 1900), shared_prefix=prefix)
    sc.upload(case)
    _, _, _, part = _run(case, prefix, S, ps_splits, False)
    L = case.layout
    m, l, acc = part.m.cpu().numpy(), part.l.cpu().numpy(), part.acc.cpu().numpy()
    qb = bf16_bits(case.q)
    first, n = L.sink // 128, -(-prefix // 128) - L.sink // 128
    for b in range(2):
        for h in (0, 5):
            cache = sc.oracle_head_cache(case, b, h)
            for g in range(gqa):
                hq = h * gqa + g
                for s in range(ps_splits):
                    lo = max(L.sink, (first + s * n // ps_splits) * 128)
                    hi = min(prefix, (first + (s + 1) * n // ps_splits) * 128)
                    rm, rl, racc = oracle.partial(qb[b, hq], case.RK[h], cache, case.sm_scale, [(lo, hi)])
                    assert abs(m[b, hq, s] - rm) <= 1e-4 * max(1.0, abs(rm))
                    assert abs(l[b, hq, s] - rl) <= 1e-4 * rl
                    err = np.linalg.norm(acc[b, hq, s] - racc) / np.linalg.norm(racc)
                    assert err <= 1e-4, (b, hq, s, err)


def test_shared_prefix_rejects_bad_arguments():
    case = sc.make_case(n_kv=8, gqa=4, page_size=64, group=128, seq=(1600, 1500), shared_prefix=512)
    sc.upload(case, demote_history=False)
    L, dev = case.layout, case.dev
    q_rot = torch.zeros((2, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    part = ob.Partials.empty(L, 2, 4)
    args = (dev["q"], q_rot, dev["bf16"], dev["bf16_table"], dev["int2"], dev["int2_table"], dev["seq_len"],
            dev["hist_end"], case.sm_scale)
    with pytest.raises(ob.OscarError, match="prefix_end"):
        ob.oscar_decode_attention_shared_prefix(L, *args, 520, 2, part)        # not a multiple of 16
    with pytest.raises(ob.OscarError, match="prefix_end"):
        ob.oscar_decode_attention_shared_prefix(L, *args, 64, 2, part)         # not above the sink
    with pytest.raises(ob.OscarError, match="prefix_splits"):
        ob.oscar_decode_attention_shared_prefix(L, *args, 512, 4, part)        # no slot left for the suffix
    L32 = ob.Layout(8, 4, 64, 32)
    with pytest.raises(ob.OscarError, match="group 128"):
        ob.oscar_decode_attention_shared_prefix(L32, *args, 512, 2, ob.Partials.empty(L32, 2, 4))

"""The value rotation folded into the model's projections (estelledc notes, "核心要点" item 3:
the value rotation can be absorbed into the projection weights): with R_V = NULL the values
arrive already rotated, every demotion path stores them as they are, and the merge does not
rotate back.  Checked against R_V = identity (bit for bit) and against the oracle with R_V = I.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_oscar_gb300 import binding as ob
from tests import scenario as sc
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu
D = 128


def _bytes(i2):
    return [t.clone() for t in (i2.codes_k, i2.codes_v, i2.scale_k, i2.zero_k, i2.scale_v, i2.zero_v)]


def _reset(i2, saved):
    for t, s in zip((i2.codes_k, i2.codes_v, i2.scale_k, i2.zero_k, i2.scale_v, i2.zero_v), saved):
        t.copy_(s)


def _equal(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq", [
    (8, 4, 64, 128, (1500, 900)),
    (2, 4, 16, 32, (1200,)),
    (4, 2, 32, 64, (1100, 700)),
])
def test_null_RV_stores_values_as_they_are(n_kv, gqa, ps, group, seq):
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq)
    dev = sc.upload(case, demote_history=False)
    L, B = case.layout, len(seq)
    i2 = dev["int2"]
    blank = _bytes(i2)
    eye = torch.eye(D, dtype=torch.float32, device="cuda").expand(n_kv, D, D).contiguous()
    req = torch.tensor([b for b in range(B) for _ in range(L.sink, int(case.hist_end[b]))], dtype=torch.int32,
                       device="cuda")
    pos = torch.tensor([p for b in range(B) for p in range(L.sink, int(case.hist_end[b]))], dtype=torch.int32,
                       device="cuda")
    results = {}
    for name, rv in (("eye", eye), ("null", None)):
        # the fp32-chain list path
        _reset(i2, blank)
        ob.oscar_demote(L, dev["stage"], dev["stage_table"], i2, dev["int2_table"], req, pos, dev["RK"], rv,
                        oracle.C_K, oracle.C_V)
        torch.cuda.synchronize()
        results[("list", name)] = _bytes(i2)
        # the tensor-core range path
        _reset(i2, blank)
        ob.oscar_demote_range(L, dev["stage"], dev["stage_table"], i2, dev["int2_table"],
                              torch.full((B,), L.sink, dtype=torch.int32, device="cuda"), dev["hist_end"],
                              dev["RK"], rv, oracle.C_K, oracle.C_V)
        torch.cuda.synchronize()
        results[("range", name)] = _bytes(i2)
        # the per-step demotion inside the decode launch (position hist_end of each request)
        _reset(i2, blank)
        part = ob.Partials.empty(L, B, 3)
        ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], i2,
                                        dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part,
                                        demote_pos=dev["hist_end"], R_V=rv, c_K=oracle.C_K, c_V=oracle.C_V)
        torch.cuda.synchronize()
        results[("fused", name)] = _bytes(i2)
    assert ob.oscar_get_device_status() == 0
    for path in ("list", "range", "fused"):
        assert _equal(results[(path, "eye")], results[(path, "null")]), path
    # V . I is exact on both rotation paths: the value codes agree across them, and with the oracle
    for k in (1, 4, 5):                        # codes_v, scale_v, zero_v
        assert torch.equal(results[("list", "null")][k], results[("range", "null")][k])
    for b in range(B):
        he = int(case.hist_end[b])
        for h in range(n_kv):
            vb = bf16_bits(case.V[b][L.sink:he, h])
            _, pv, zv, sv = oracle.demote_rows(vb, np.eye(D, dtype=np.float32), group, oracle.C_V)
            case.dev["int2"] = ob.Int2Pool(*results[("list", "null")])
            _, cv, _, _, zv_g, sv_g = sc.gather_int2(case, b, h)
            assert np.array_equal(cv[L.sink:he], pv) and np.array_equal(zv_g[L.sink:he], zv)
            assert np.array_equal(sv_g[L.sink:he], sv)


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq,S", [
    (8, 4, 64, 128, (2000, 1300), 5),
    (2, 8, 16, 32, (1400,), 3),
])
def test_folded_value_rotation_decode_matches_oracle(n_kv, gqa, ps, group, seq, S):
    """History values demoted with R_V = NULL, decode + merge with R_V = NULL: the output in the
    values' basis equals the oracle's attention with R_V = I (the attention-output bar)."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq)
    case.RV = np.stack([np.eye(D, dtype=np.float32)] * n_kv)
    dev = sc.upload(case, demote_history=False)
    L, B = case.layout, len(seq)
    # (the fp32-chain demotion: its key codes are the oracle's own, bit for bit)
    req = torch.tensor([b for b in range(B) for _ in range(L.sink, int(case.hist_end[b]))], dtype=torch.int32,
                       device="cuda")
    pos = torch.tensor([p for b in range(B) for p in range(L.sink, int(case.hist_end[b]))], dtype=torch.int32,
                       device="cuda")
    ob.oscar_demote(L, dev["stage"], dev["stage_table"], dev["int2"], dev["int2_table"], req, pos, dev["RK"], None,
                    oracle.C_K, oracle.C_V)
    part = ob.Partials.empty(L, B, S)
    out = torch.empty((B, L.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty((B, L.n_q_heads, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, L.n_q_heads), dtype=torch.float32, device="cuda")
    ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                    dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale, part,
                                    out=out, out_f32=out32, lse=lse)
    torch.cuda.synchronize()
    assert ob.oscar_get_device_status() == 0
    ref = sc.oracle_outputs(case)
    o32, lse_g = out32.cpu().numpy(), lse.cpu().numpy()
    for (b, hq), (o, l) in ref.items():
        ok, r, m = sc.tolerance_ok(o32[b, hq], o)
        assert ok, ((b, hq), r, m)
        assert abs(lse_g[b, hq] - l) <= 1e-4 * max(1.0, abs(l))

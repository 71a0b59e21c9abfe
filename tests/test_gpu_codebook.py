"""The non-uniform (Lloyd-Max) codebook on the GPU against the oracle: codes, scale and zero of
the quantizer and of the demotion bit for bit, decode attention (its INT2 part on the CUDA cores)
within the attention bar, and the tensor-core-only paths refusing the layout."""
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


def _levels():
    return oracle.lloyd_max_codebook(oracle.C_K), oracle.lloyd_max_codebook(oracle.C_V)


@pytest.mark.parametrize("group", [128, 64, 32])
def test_quantize_rotated_codebook_bit_exact(group):
    lk, lv = _levels()
    L = ob.Layout(2, 4, 16, group, levels_k=tuple(map(float, lk)), levels_v=tuple(map(float, lv)))
    rng = np.random.default_rng(4)
    x = rng.normal(0, 2.0, size=(300, D)).astype(np.float32)
    x[:, rng.integers(0, D, size=4)] *= 6
    x[0, :] = 1.25                                         # a constant row: scale 0, code 0
    xd = torch.from_numpy(x).cuda()
    codes = torch.empty((300, D // 4), dtype=torch.uint8, device="cuda")
    scale = torch.empty((300, D // group), dtype=torch.bfloat16, device="cuda")
    zero = torch.empty_like(scale)
    ob.oscar_quantize_rotated(L, xd, oracle.C_K, codes, scale, zero)
    torch.cuda.synchronize()
    packed, z, s = oracle.quantize_rows(x, group, oracle.C_K, levels=lk)
    assert np.array_equal(codes.cpu().numpy(), packed)
    assert np.array_equal(bf16_bits(zero), z) and np.array_equal(bf16_bits(scale), s)


@pytest.mark.parametrize("n_kv,gqa,ps,group,seq,S", [
    (8, 4, 64, 128, (3000, 1700), 6),       # the benchmark's shape
    (2, 8, 16, 32, (1400,), 3),
    (4, 2, 32, 64, (1800, 900), 4),
])
def test_demote_and_decode_with_codebook(n_kv, gqa, ps, group, seq, S):
    """oscar_demote writes the oracle's codebook codes, scale and zero for every history row;
    oscar_decode_attention + oscar_merge then match the oracle's attention over those codes read
    through the codebook."""
    case = sc.make_case(n_kv=n_kv, gqa=gqa, page_size=ps, group=group, seq=seq, levels=_levels())
    sc.upload(case)
    torch.cuda.synchronize()
    L = case.layout
    for b in range(len(seq)):
        he = int(case.hist_end[b])
        for h in range(n_kv):
            _, pk, zk, sk = oracle.demote_rows(bf16_bits(case.K[b][L.sink:he, h]), case.RK[h], group, oracle.C_K,
                                               levels=L.levels_k)
            _, pv, zv, sv = oracle.demote_rows(bf16_bits(case.V[b][L.sink:he, h]), case.RV[h], group, oracle.C_V,
                                               levels=L.levels_v)
            ck, cv, gzk, gsk, gzv, gsv = sc.gather_int2(case, b, h)
            assert np.array_equal(ck[L.sink:he], pk) and np.array_equal(cv[L.sink:he], pv)
            assert np.array_equal(gzk[L.sink:he], zk) and np.array_equal(gsk[L.sink:he], sk)
            assert np.array_equal(gzv[L.sink:he], zv) and np.array_equal(gsv[L.sink:he], sv)
    out, out32, lse, _ = sc.run_decode(case, S)
    _check_outputs(case, out, out32, lse)
    assert ob.oscar_get_device_status() == 0


def test_codebook_refused_by_tensor_core_only_paths():
    case = sc.make_case(n_kv=8, gqa=4, page_size=64, group=128, seq=(1200,), levels=_levels())
    sc.upload(case, demote_history=False)
    L, dev = case.layout, case.dev
    with pytest.raises(ob.OscarError, match="codebook"):
        ob.oscar_decode_attention_fused(L, dev["q"], dev["RK"], dev["bf16"], dev["bf16_table"], dev["int2"],
                                        dev["int2_table"], dev["seq_len"], dev["hist_end"], case.sm_scale,
                                        ob.Partials.empty(L, 1, 2))
    begin = torch.tensor([L.sink], dtype=torch.int32, device="cuda")
    with pytest.raises(ob.OscarError, match="uniform levels"):
        ob.oscar_demote_range(L, dev["stage"], dev["stage_table"], dev["int2"], dev["int2_table"], begin,
                              dev["hist_end"], dev["RK"], dev["RV"], oracle.C_K, oracle.C_V)

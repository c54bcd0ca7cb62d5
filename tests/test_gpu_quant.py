"""GPU parity of the 8-bit write that derives block scales from the data
(pkv_kv_cache_write_rescale), bit-exact against the oracle."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import bf16_dev, dev_bits, to_dev, torch_cache_dtype, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


@pytest.mark.parametrize("cfg", [5, 7, 9])
def test_rescale_write_bit_exact_then_partial_rewrite(cfg):
    torch = torch_mod()
    wl = W.make(cfg, small=True)
    d = W.host_data(wl)
    req, pos = W.token_rows_order(wl)
    bt = to_dev(wl.block_table)
    # oracle
    slots_o = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    kc_o = np.zeros(wl.cache_shape, wl.cache_np_dtype)
    vc_o = np.zeros_like(kc_o)
    ks_o = np.full((wl.NB, wl.Hkv), 123.0, np.float32)
    vs_o = ks_o.copy()
    oracle.kv_cache_write_rescale(d["k_rows"], d["v_rows"], slots_o, kc_o, vc_o, ks_o, vs_o)
    # library (garbage workspace: it needs no clearing)
    kc = torch.zeros(wl.cache_shape, dtype=torch_cache_dtype(wl), device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.full((wl.NB, wl.Hkv), 123.0, dtype=torch.float32, device="cuda")
    vs = ks.clone()
    ws = torch.full((8 * wl.NB * wl.Hkv,), 0x7F, dtype=torch.uint8, device="cuda")
    slots = pkv.compute_slot_mapping(bt, to_dev(pos), wl.BS, req_idx=to_dev(req))
    pkv.kv_cache_write_rescale(bf16_dev(d["k_rows"]), bf16_dev(d["v_rows"]), slots, kc, vc, ks, vs,
                               workspace=ws)
    assert np.array_equal(ks.cpu().numpy(), ks_o) and np.array_equal(vs.cpu().numpy(), vs_o)
    assert np.array_equal(dev_bits(kc), kc_o) and np.array_equal(dev_bits(vc), vc_o)
    # a second call over the step's new tokens only: their blocks are re-scaled from
    # those rows alone, every other scale stays
    req2, pos2 = wl.new_token_rows()
    s2 = oracle.slot_mapping(wl.block_table, req2, pos2, wl.BS)
    oracle.kv_cache_write_rescale(d["k_new"], d["v_new"], s2, kc_o, vc_o, ks_o, vs_o)
    slots2 = pkv.compute_slot_mapping(bt, to_dev(pos2), wl.BS, req_idx=to_dev(req2))
    pkv.kv_cache_write_rescale(bf16_dev(d["k_new"]), bf16_dev(d["v_new"]), slots2, kc, vc, ks, vs,
                               workspace=ws)
    assert np.array_equal(ks.cpu().numpy(), ks_o) and np.array_equal(vs.cpu().numpy(), vs_o)
    assert np.array_equal(dev_bits(kc), kc_o) and np.array_equal(dev_bits(vc), vc_o)


def test_rescale_write_rejects_bf16_and_small_workspace():
    torch_mod()
    L = pkv.lib()
    assert L.pkv_kv_cache_write_rescale(16, 16, 16, 4, 2, 128, 16, 8, 0, 16, 16, 16, 16, 16, 1 << 20,
                                        None) == -2
    assert L.pkv_kv_cache_write_rescale(16, 16, 16, 4, 2, 128, 16, 8, 1, 16, 16, 16, 16, 16, 8,
                                        None) == -3

"""The allocation-free decode entry point (pkv_paged_decode_attn_noalloc).

Some callers cannot call cudaMalloc: a plugin inside an engine that owns all device
memory and offers no workspace hook, or a latency-critical path that must not risk
cudaMalloc's implicit device synchronisation.  For them the library keeps the decode
scratch in a static device array.  These tests call that entry point through the C ABI
and check, on two calls in a row, that it returns what the workspace entry point
returns, and that a shape too large for the static array is refused.

The file name makes pytest collect it after every other test file.
"""
import ctypes

import numpy as np
import pytest

import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import bf16_dev, compare, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _inputs(cfg):
    torch = torch_mod()
    wl = W.make(cfg, small=True)
    d = W.host_data(wl)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    if wl.quant:
        kc = torch.zeros((wl.NB, wl.Hkv, wl.BS, wl.D), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        ks, vs = to_dev(d["k_scale"]), to_dev(d["v_scale"])
        req, pos = W.token_rows_order(wl)
        slots = pkv.compute_slot_mapping(bt, to_dev(pos), wl.BS, req_idx=to_dev(req))
        pkv.kv_cache_write(bf16_dev(d["k_rows"]), bf16_dev(d["v_rows"]), slots, kc, vc, ks, vs)
    else:
        kc, vc, ks, vs = bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"]), None, None
    return wl, bf16_dev(d["q"]), kc, vc, ks, vs, bt, sl


@pytest.mark.parametrize("cfg", [2, 5])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cfg):
    torch = torch_mod()
    wl, q, kc, vc, ks, vs, bt, sl = _inputs(cfg)
    ref = pkv.paged_decode_attn(q, kc, vc, bt, sl, wl.scale, k_scale=ks, v_scale=vs)
    ref64 = out_to_f64(ref)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        pkv.paged_decode_attn_noalloc(q, kc, vc, bt, sl, wl.scale, out=out, k_scale=ks,
                                      v_scale=vs)
        torch.cuda.synchronize()
        compare(out_to_f64(out), ref64, wl.quant)
        # same kernels, same launch plan: the bits agree as well
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_refuses_shapes_beyond_its_static_scratch():
    torch_mod()
    L = pkv.lib()
    # 16384 requests x 8 kv heads need far more than 16 MiB of scratch; the fake
    # pointers are never touched because the size check comes first
    st = L.pkv_paged_decode_attn_noalloc(16, 16, 16, None, None, 16, 4, 16, 16384, 64, 8, 128,
                                         16, 8, 0, 0.1, 16, None)
    assert st == -3  # PKV_ERR_WORKSPACE
    assert L.pkv_paged_decode_attn_noalloc(16, 16, 16, None, None, 16, 4, 16, 4, 64, 8, 96, 16,
                                           8, 0, 0.1, 16, None) == -2

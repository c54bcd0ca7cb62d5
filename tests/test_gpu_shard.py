"""A decode batch split over ranks, each shard run through the library on one GPU.

Splitting by requests, or by KV heads with their query heads, needs no exchange
(shard.py).  Each shard runs pkv_paged_decode_attn on its own inputs; the
concatenation of the shards' outputs must match the whole batch's oracle output within
the attention tolerance, as must the unsharded call.  Bit equality between the sharded
and unsharded GPU outputs is not expected: the decode kernel splits the batch's flat
page list evenly over its warps, so a shard's units can be cut at other pages than in
the whole batch, and their partial results are then merged in another grouping."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import shard
from paged_kv_cache_289_gb300 import workloads as W
from helpers import HostCase, bf16_dev, compare, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _dev_pages(case, h0=None, h1=None):
    wl = case.wl
    kc, vc = case.kc, case.vc
    ks, vs = case.d.get("k_scale"), case.d.get("v_scale")
    if h0 is not None:
        kc = np.ascontiguousarray(kc[:, h0:h1])
        vc = np.ascontiguousarray(vc[:, h0:h1])
        if wl.quant:
            ks = np.ascontiguousarray(ks[:, h0:h1])
            vs = np.ascontiguousarray(vs[:, h0:h1])
    if wl.quant:
        return to_dev(kc), to_dev(vc), to_dev(ks), to_dev(vs)
    return bf16_dev(kc), bf16_dev(vc), None, None


def _run(q, kc, vc, ks, vs, bt, sl, scale):
    out = pkv.paged_decode_attn(bf16_dev(q), kc, vc, to_dev(bt), to_dev(sl), scale, k_scale=ks,
                                v_scale=vs)
    return out_to_f64(out)


@pytest.mark.parametrize("cfg,world", [(2, 2), (2, 3), (5, 2), (3, 4)])
def test_request_and_kv_head_shards_reassemble_the_batch(cfg, world):
    wl = W.make(cfg, small=True)
    case = HostCase(wl)
    q = case.d["q"]
    ks_h, vs_h = case.d.get("k_scale"), case.d.get("v_scale")
    whole_ref = oracle.decode_attn(q, case.kc, case.vc, wl.block_table, wl.seq_lens, wl.scale,
                                   ks_h, vs_h)
    kc, vc, ks, vs = _dev_pages(case)
    whole_gpu = _run(q, kc, vc, ks, vs, wl.block_table, wl.seq_lens, wl.scale)
    compare(whole_gpu, whole_ref, wl.quant)

    # data parallel: whole requests per rank
    parts = []
    for a, b in shard.plan_requests(wl.seq_lens, world):
        if a == b:
            continue
        parts.append(_run(q[a:b], kc, vc, ks, vs, wl.block_table[a:b], wl.seq_lens[a:b],
                          wl.scale))
        compare(parts[-1], whole_ref[a:b], wl.quant)
    by_req = np.concatenate(parts, axis=0)
    compare(by_req, whole_ref, wl.quant)
    compare(by_req, whole_gpu, wl.quant)

    # tensor parallel over KV heads: each rank holds its heads' pages only
    G = wl.G
    parts = []
    for h0, h1 in shard.plan_kv_heads(wl.Hkv, world):
        if h0 == h1:
            continue
        kc_s, vc_s, ks_s, vs_s = _dev_pages(case, h0, h1)
        qs = np.ascontiguousarray(q[:, h0 * G:h1 * G])
        parts.append(_run(qs, kc_s, vc_s, ks_s, vs_s, wl.block_table, wl.seq_lens, wl.scale))
        compare(parts[-1], whole_ref[:, h0 * G:h1 * G], wl.quant)
    by_head = np.concatenate(parts, axis=1)
    compare(by_head, whole_ref, wl.quant)
    compare(by_head, whole_gpu, wl.quant)

"""GPU parity at the full workload sizes, in the launch configuration the benchmark
times.  Inputs are drawn on the device from a seeded generator; the oracle checks a
sample of (request, query head) rows one by one from the same bytes."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import compare, dev_bits, out_to_f64, torch_cache_dtype, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _sample_rows(wl, rng, n):
    rows = set()
    # always include the longest and the shortest requests, first and last heads
    rmax, rmin = int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens))
    for r in (rmax, rmin):
        rows.update({r * wl.Hq, r * wl.Hq + wl.Hq - 1})
    while len(rows) < n:
        rows.add(int(rng.integers(0, wl.N * wl.Hq)))
    return np.array(sorted(rows), np.int64)


def _compact(wl, reqs):
    """Compact block table over the pages of `reqs` (new ids 0..n-1) and the old ids."""
    old = []
    bt = np.zeros((len(reqs), wl.MB), np.int32)
    seen = {}
    for i, r in enumerate(reqs):
        for j, b in enumerate(wl.blocks_of(r)):
            b = int(b)
            if b not in seen:
                seen[b] = len(old)
                old.append(b)
            bt[i, j] = seen[b]
    return bt, np.array(old, np.int64)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5, 7, 9])
def test_fullsize_decode_step_sampled(cfg):
    torch = torch_mod()
    wl = W.make(cfg)
    dd = W.device_data(wl, "cuda")
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    if wl.quant:
        kc = torch.zeros(wl.cache_shape, dtype=torch_cache_dtype(wl), device="cuda")
        vc = torch.zeros_like(kc)
        req, pos = W.token_rows_order(wl)
        slots_all = pkv.compute_slot_mapping(bt, torch.from_numpy(pos).cuda(), wl.BS,
                                             req_idx=torch.from_numpy(req).cuda())
        pkv.kv_cache_write(dd["k_rows"], dd["v_rows"], slots_all, kc, vc, dd["k_scale"],
                           dd["v_scale"])
        ks, vs = dd["k_scale"], dd["v_scale"]
    else:
        kc, vc, ks, vs = dd["k_cache"], dd["v_cache"], None, None
    rng = np.random.default_rng(100 + cfg)
    rows = _sample_rows(wl, rng, 24 if cfg != 3 else 12)
    reqs = sorted({int(r) // wl.Hq for r in rows})
    cbt, old = _compact(wl, reqs)
    old_t = torch.from_numpy(old).cuda()
    # pages of the sampled requests before the step (bf16: drawn by torch on the device)
    kc_pre = dev_bits(kc.index_select(0, old_t))
    vc_pre = dev_bits(vc.index_select(0, old_t))

    # the decode step: new token of every request at seq_len - 1, then attention
    pos_new = torch.from_numpy(wl.new_token_positions()).cuda()
    slots = pkv.compute_slot_mapping(bt, pos_new, wl.BS)
    pkv.kv_cache_write(dd["k_new"], dd["v_new"], slots, kc, vc, ks, vs)
    ws = pkv.alloc_decode_workspace(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS,
                                    wl.kv_kind)
    out = pkv.paged_decode_attn(dd["q"], kc, vc, bt, sl, wl.scale, k_scale=ks, v_scale=vs,
                                workspace=ws)
    torch.cuda.synchronize()
    assert pkv.read_device_error(ws) == 0

    kc_s = dev_bits(kc.index_select(0, old_t))
    vc_s = dev_bits(vc.index_select(0, old_t))
    q_s = dev_bits(dd["q"][torch.tensor(reqs).cuda()])
    sl_s = wl.seq_lens[reqs]
    ks_s = vs_s = None
    newpos = (sl_s.astype(np.int64) - 1).astype(np.int32)
    k_new_s = dev_bits(dd["k_new"][torch.tensor(reqs).cuda()])
    v_new_s = dev_bits(dd["v_new"][torch.tensor(reqs).cuda()])
    if not wl.quant:
        # the oracle applies the step's write to the pre-step pages itself
        kc_o, vc_o = kc_pre.copy(), vc_pre.copy()
        sm = oracle.slot_mapping(cbt, np.arange(len(reqs), dtype=np.int32), newpos, wl.BS)
        oracle.kv_cache_write(k_new_s, v_new_s, sm, kc_o, vc_o)
        assert np.array_equal(kc_s, kc_o) and np.array_equal(vc_s, vc_o)
    else:
        ks_s = ks.index_select(0, old_t).cpu().numpy()
        vs_s = vs.index_select(0, old_t).cpu().numpy()
        # the oracle quantises the sampled requests' source rows (then the step's new rows)
        # itself; its pages must equal the library's bytes
        kc_o = np.zeros_like(kc_s)
        vc_o = np.zeros_like(vc_s)
        offs = wl.token_offsets
        for i, r in enumerate(reqs):
            S = int(wl.seq_lens[r])
            rows_k = dev_bits(dd["k_rows"][offs[r]:offs[r] + S])
            rows_v = dev_bits(dd["v_rows"][offs[r]:offs[r] + S])
            sm = oracle.slot_mapping(cbt, np.full(S, i, np.int32), np.arange(S, dtype=np.int32),
                                     wl.BS)
            oracle.kv_cache_write(rows_k, rows_v, sm, kc_o, vc_o, ks_s, vs_s)
        sm = oracle.slot_mapping(cbt, np.arange(len(reqs), dtype=np.int32), newpos, wl.BS)
        oracle.kv_cache_write(k_new_s, v_new_s, sm, kc_o, vc_o, ks_s, vs_s)
        for i, r in enumerate(reqs):
            S = int(wl.seq_lens[r])
            for j in range(len(wl.blocks_of(r))):
                n = min(wl.BS, S - j * wl.BS)
                b = cbt[i, j]
                assert np.array_equal(kc_s[b, :, :n], kc_o[b, :, :n])
                assert np.array_equal(vc_s[b, :, :n], vc_o[b, :, :n])
    local_rows = np.array([reqs.index(int(r) // wl.Hq) * wl.Hq + int(r) % wl.Hq for r in rows],
                          np.int64)
    ref = oracle.decode_rows(q_s, kc_o, vc_o, cbt, sl_s, wl.scale, local_rows, ks_s, vs_s)
    got = out_to_f64(out).reshape(wl.N * wl.Hq, wl.D)[rows]
    compare(got, ref, wl.quant)

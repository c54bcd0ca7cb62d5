"""GPU parity of multi-query paged attention (several new query tokens per request,
as when a speculative draft is verified): the library through the C ABI against the
fp64 oracle's causal multi-query attention on the same seeded inputs."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import (HostCase, bf16_dev, compare, dev_bits, out_to_f64, to_dev, torch_mod,
                     torch_cache_dtype)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _device_caches(case):
    torch = torch_mod()
    wl = case.wl
    if not wl.quant:
        return bf16_dev(case.d["k_cache"]), bf16_dev(case.d["v_cache"]), None, None
    kc = torch.zeros(wl.cache_shape, dtype=torch_cache_dtype(wl), device="cuda")
    vc = torch.zeros_like(kc)
    ks, vs = to_dev(case.d["k_scale"]), to_dev(case.d["v_scale"])
    slots = pkv.compute_slot_mapping(to_dev(wl.block_table), to_dev(case.pos_all), wl.BS,
                                     req_idx=to_dev(case.req_all))
    pkv.kv_cache_write(bf16_dev(case.d["k_rows"]), bf16_dev(case.d["v_rows"]), slots, kc, vc, ks,
                       vs)
    return kc, vc, ks, vs


def _gpu_step(case, kc, vc, ks, vs, q_offsets=None, max_q_len=None):
    wl = case.wl
    bt = to_dev(wl.block_table)
    req, pos = wl.new_token_rows()
    slots = pkv.compute_slot_mapping(bt, to_dev(pos), wl.BS, req_idx=to_dev(req))
    pkv.kv_cache_write(bf16_dev(case.d["k_new"]), bf16_dev(case.d["v_new"]), slots, kc, vc, ks, vs)
    qo = wl.q_offsets() if q_offsets is None else q_offsets
    mq = wl.q_len if max_q_len is None else max_q_len
    dt = wl.kv_kind
    torch = torch_mod()
    ws = torch.zeros(pkv.multiquery_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, dt, mq),
                     dtype=torch.uint8, device="cuda")
    out = pkv.paged_multiquery_attn(bf16_dev(case.d["q"]), to_dev(qo), mq, kc, vc, bt,
                                    to_dev(wl.seq_lens), wl.scale, k_scale=ks, v_scale=vs,
                                    workspace=ws)
    return slots, out, ws


def test_spec_verify_step_small():
    wl = W.make(6, small=True)
    case = HostCase(wl)
    kc, vc, ks, vs = _device_caches(case)
    slots_d, out_d, ws = _gpu_step(case, kc, vc, ks, vs)
    slots_o, out_o = case.oracle_step()
    assert np.array_equal(slots_d.cpu().numpy(), slots_o)
    assert np.array_equal(dev_bits(kc), case.kc)
    compare(out_to_f64(out_d), out_o, False)
    assert pkv.read_device_error(ws) == 0


@pytest.mark.parametrize("G,D,BS,kind,qmax", [(8, 128, 16, "bf16", 4), (8, 128, 32, "bf16", 2),
                                              (4, 64, 16, "bf16", 4), (1, 64, 32, "bf16", 4),
                                              (8, 128, 32, "fp8", 2), (4, 128, 16, "fp8", 2),
                                              (8, 128, 32, "int8", 2), (3, 128, 16, "bf16", 3),
                                              (8, 128, 32, "int4", 2), (4, 128, 16, "int4", 2)])
def test_multiquery_shapes_variable_qlen(G, D, BS, kind, qmax):
    """Every supported shape; each request has its own q_len in 1..qmax; short requests
    have fewer tokens than queries (their first queries see nothing: zero rows)."""
    rng = np.random.default_rng(G * 1000 + D + BS + qmax)
    Hkv = 2
    lens = [1, 2, BS - 1, BS, BS + 1, 3 * BS + 5, 700, 37]
    qlens = [int(rng.integers(1, qmax + 1)) for _ in lens]
    qlens[0], qlens[1] = qmax, qmax          # q_len > seq_len for the 1- and 2-token requests
    fp8 = kind != "bf16"
    wl = W.custom(len(lens), G * Hkv, Hkv, D, BS, lens, fp8=kind == "fp8", int8=kind == "int8",
                  int4=kind == "int4",
                  seed=G + D + BS)
    qoffs = np.zeros(len(lens) + 1, np.int32)
    np.cumsum(qlens, out=qoffs[1:])
    case = HostCase(wl)
    q = W.f32_to_bf16_bits(rng.standard_normal((int(qoffs[-1]), wl.Hq, D)).astype(np.float32))
    kc, vc, ks, vs = _device_caches(case)
    torch = torch_mod()
    dt = wl.kv_kind
    ws = torch.zeros(pkv.multiquery_workspace_size(wl.N, wl.Hq, Hkv, D, BS, dt, qmax),
                     dtype=torch.uint8, device="cuda")
    out = pkv.paged_multiquery_attn(bf16_dev(q), to_dev(qoffs), qmax, kc, vc,
                                    to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale,
                                    k_scale=ks, v_scale=vs, workspace=ws)
    ref = oracle.multiquery_attn(q, qoffs, case.kc, case.vc, wl.block_table, wl.seq_lens,
                                 wl.scale, case.d.get("k_scale"), case.d.get("v_scale"))
    got = out_to_f64(out)
    compare(got, ref, fp8)
    assert np.all(got[ref.reshape(len(ref), -1).any(axis=1) == 0] == 0)
    assert pkv.read_device_error(ws) == 0


def test_multiquery_with_one_query_equals_decode_bitwise():
    wl = W.make(2, small=True)
    d = W.host_data(wl)
    q = bf16_dev(d["q"])
    kc, vc = bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"])
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    a = dev_bits(pkv.paged_decode_attn(q, kc, vc, bt, sl, wl.scale))
    b = dev_bits(pkv.paged_multiquery_attn(q, to_dev(np.arange(wl.N + 1, dtype=np.int32)), 1,
                                           kc, vc, bt, sl, wl.scale))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("qmax", [2, 4])
def test_multiquery_long_request_split_over_every_warp(qmax):
    wl = W.custom(1, 8, 1, 128, 16, [20000], seed=9, q_len=qmax)
    case = HostCase(wl)
    kc, vc, ks, vs = _device_caches(case)
    _, out_d, ws = _gpu_step(case, kc, vc, ks, vs)
    _, out_o = case.oracle_step()
    compare(out_to_f64(out_d), out_o, False)
    assert pkv.read_device_error(ws) == 0


def test_multiquery_qlen_past_the_limit_is_clamped_and_flagged():
    torch = torch_mod()
    wl = W.custom(2, 8, 2, 128, 16, [100, 200], seed=10)
    d = W.host_data(wl)
    q = bf16_dev(W.f32_to_bf16_bits(np.ones((7, 8, 128), np.float32)))
    qoffs = np.array([0, 2, 7], np.int32)       # the second request asks for 5 > max 4
    ws = torch.zeros(pkv.multiquery_workspace_size(2, 8, 2, 128, 16, pkv.BF16, 4),
                     dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(q)
    pkv.paged_multiquery_attn(q, to_dev(qoffs), 4, bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"]),
                              to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale, out=out,
                              workspace=ws)
    err = pkv.read_device_error(ws)
    assert err & pkv.DEVERR_QLEN_CLAMPED and not (err & pkv.DEVERR_WAIT_TIMEOUT)
    assert np.all(np.isfinite(out_to_f64(out)))


def test_spec_verify_fullsize_sampled_requests():
    """Workload 6 at full size (64 requests x 4 new tokens, lengths U[1024, 8192]) in the
    benchmark's launch configuration; the oracle applies the step's write to the sampled
    requests' pre-step pages itself and computes all their query rows."""
    torch = torch_mod()
    wl = W.make(6)
    dd = W.device_data(wl, "cuda")
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    kc, vc = dd["k_cache"], dd["v_cache"]
    reqs = sorted({int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens)), 7, 40})
    old, seen = [], {}
    cbt = np.zeros((len(reqs), wl.MB), np.int32)
    for i, r in enumerate(reqs):
        for j, b in enumerate(wl.blocks_of(r)):
            if int(b) not in seen:
                seen[int(b)] = len(old)
                old.append(int(b))
            cbt[i, j] = seen[int(b)]
    old_t = torch.tensor(old, dtype=torch.int64, device="cuda")
    kc_o = dev_bits(kc.index_select(0, old_t))
    vc_o = dev_bits(vc.index_select(0, old_t))
    req, pos = wl.new_token_rows()
    slots = pkv.compute_slot_mapping(bt, to_dev(pos), wl.BS, req_idx=to_dev(req))
    pkv.kv_cache_write(dd["k_new"], dd["v_new"], slots, kc, vc)
    ws = torch.zeros(pkv.multiquery_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, pkv.BF16, 4),
                     dtype=torch.uint8, device="cuda")
    out = pkv.paged_multiquery_attn(dd["q"], to_dev(wl.q_offsets()), 4, kc, vc, bt, sl, wl.scale,
                                    workspace=ws)
    torch.cuda.synchronize()
    assert pkv.read_device_error(ws) == 0
    rows = np.concatenate([np.arange(r * 4, r * 4 + 4) for r in reqs])
    rows_t = torch.from_numpy(rows).cuda()
    sl_s = wl.seq_lens[reqs]
    sreq = np.repeat(np.arange(len(reqs), dtype=np.int32), 4)
    spos = (np.repeat(sl_s.astype(np.int64), 4) - 4 + np.tile(np.arange(4), len(reqs))).astype(np.int32)
    sm = oracle.slot_mapping(cbt, sreq, spos, wl.BS)
    oracle.kv_cache_write(dev_bits(dd["k_new"][rows_t]), dev_bits(dd["v_new"][rows_t]), sm, kc_o,
                          vc_o)
    assert np.array_equal(dev_bits(kc.index_select(0, old_t)), kc_o)
    qo = (np.arange(len(reqs) + 1) * 4).astype(np.int32)
    ref = oracle.multiquery_attn(dev_bits(dd["q"][rows_t]), qo, kc_o, vc_o, cbt, sl_s, wl.scale)
    compare(out_to_f64(out)[rows], ref, False)

"""The allocation-free decode entry point (pkv_paged_decode_attn_noalloc).

Some callers cannot call cudaMalloc: a plugin inside an engine that owns all device
memory and offers no workspace hook, or a latency-critical path that must not risk
cudaMalloc's implicit device synchronisation.  For them the library keeps the decode
scratch in a static device array.  These tests call that entry point through the C ABI
and check, on two calls in a row, that it agrees with the fp64 oracle within the
attention tolerances and with the workspace entry point bit for bit; that the largest
shape its 16 MiB array holds runs and agrees as well; and that the next larger shape is
refused.

The file name makes pytest collect it after every other test file.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import HostCase, bf16_dev, compare, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20          # the static array's size, as the header states


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _device_case(wl):
    """The oracle's own caches (each side sees the same page bytes and scales) and the
    same inputs on the device."""
    hc = HostCase(wl)
    if wl.quant:
        kc, vc = to_dev(hc.kc), to_dev(hc.vc)
        ks, vs = to_dev(hc.d["k_scale"]), to_dev(hc.d["v_scale"])
    else:
        kc, vc = bf16_dev(hc.kc), bf16_dev(hc.vc)
        ks = vs = None
    dev = dict(q=bf16_dev(hc.d["q"]), kc=kc, vc=vc, ks=ks, vs=vs,
               bt=to_dev(wl.block_table), sl=to_dev(wl.seq_lens))
    return hc, dev


def _oracle(hc):
    wl = hc.wl
    return oracle.decode_attn(hc.d["q"], hc.kc, hc.vc, wl.block_table, wl.seq_lens, wl.scale,
                              hc.d.get("k_scale"), hc.d.get("v_scale"))


@pytest.mark.parametrize("cfg", [2, 5])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_consecutive_calls(cfg):
    torch = torch_mod()
    wl = W.make(cfg, small=True)
    hc, d = _device_case(wl)
    ref64 = _oracle(hc).reshape(wl.N, wl.Hq, wl.D)
    ws_out = pkv.paged_decode_attn(d["q"], d["kc"], d["vc"], d["bt"], d["sl"], wl.scale,
                                   k_scale=d["ks"], v_scale=d["vs"])
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        pkv.paged_decode_attn_noalloc(d["q"], d["kc"], d["vc"], d["bt"], d["sl"], wl.scale,
                                      out=out, k_scale=d["ks"], v_scale=d["vs"])
        torch.cuda.synchronize()
        compare(out_to_f64(out), ref64, wl.quant)
        # same kernels, same launch plan: the bits agree with the workspace call
        assert torch.equal(out.view(torch.int16), ws_out.view(torch.int16))


def _largest_batch(Hq, Hkv, D, BS, kind, sms):
    """Largest batch whose decode workspace fits the static array (bisection; the size
    grows with the batch)."""
    lo, hi = 1, 16384
    assert pkv.decode_workspace_size(lo, Hq, Hkv, D, BS, kind, sms) <= SCRATCH_BYTES
    while lo < hi:
        mid = (lo + hi + 1) // 2
        n = pkv.decode_workspace_size(mid, Hq, Hkv, D, BS, kind, sms)
        if 0 < n <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_runs_at_its_size_limit_and_refuses_one_more_request():
    torch = torch_mod()
    Hq, Hkv, D, BS = 16, 8, 128, 16
    sms = pkv.device_num_sms()
    N = _largest_batch(Hq, Hkv, D, BS, 0, sms)
    assert pkv.decode_workspace_size(N + 1, Hq, Hkv, D, BS, 0, sms) > SCRATCH_BYTES
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 41, size=N).astype(np.int32)     # short requests, a small pool
    wl = W.custom(N, Hq, Hkv, D, BS, lens, seed=12, name="noalloc_limit")
    hc, d = _device_case(wl)
    ws_out = pkv.paged_decode_attn(d["q"], d["kc"], d["vc"], d["bt"], d["sl"], wl.scale)
    out = torch.full_like(d["q"], float("nan"))
    pkv.paged_decode_attn_noalloc(d["q"], d["kc"], d["vc"], d["bt"], d["sl"], wl.scale, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ws_out.view(torch.int16))
    rows = rng.choice(N * Hq, size=64, replace=False).astype(np.int64)
    ref = oracle.decode_rows(hc.d["q"], hc.kc, hc.vc, wl.block_table, wl.seq_lens, wl.scale,
                             rows)
    compare(out_to_f64(out).reshape(-1, D)[rows], ref, False)
    # one more request does not fit: refused before anything is launched
    L = pkv.lib()
    q1 = torch.zeros((N + 1, Hq, D), dtype=torch.bfloat16, device="cuda")
    bt1 = torch.zeros((N + 1, d["bt"].shape[1]), dtype=torch.int32, device="cuda")
    sl1 = torch.ones(N + 1, dtype=torch.int32, device="cuda")
    st = L.pkv_paged_decode_attn_noalloc(
        q1.data_ptr(), d["kc"].data_ptr(), d["vc"].data_ptr(), None, None, bt1.data_ptr(),
        bt1.shape[1], sl1.data_ptr(), N + 1, Hq, Hkv, D, BS, wl.NB, 0, wl.scale,
        q1.data_ptr(), None)
    assert st == -3  # PKV_ERR_WORKSPACE


def test_noalloc_statuses_match_the_workspace_entry_point():
    torch_mod()
    L = pkv.lib()
    # 16384 requests x 8 kv heads need far more than 16 MiB of scratch; the fake
    # pointers are never touched because the size check comes first
    st = L.pkv_paged_decode_attn_noalloc(16, 16, 16, None, None, 16, 4, 16, 16384, 64, 8, 128,
                                         16, 8, 0, 0.1, 16, None)
    assert st == -3  # PKV_ERR_WORKSPACE
    # unsupported head_dim, a negative batch, an empty batch with an unsupported shape and
    # an empty valid batch: the same status from both entry points
    for args in [(4, 64, 8, 96), (-1, 64, 8, 128), (0, 64, 8, 96), (0, 64, 8, 128)]:
        N, Hq, Hkv, D = args
        a = L.pkv_paged_decode_attn_noalloc(16, 16, 16, None, None, 16, 4, 16, N, Hq, Hkv, D,
                                            16, 8, 0, 0.1, 16, None)
        b = L.pkv_paged_decode_attn(16, 16, 16, None, None, 16, 4, 16, N, Hq, Hkv, D, 16, 8, 0,
                                    0.1, 16, None, 0, None)
        assert a == b, (args, a, b)
    assert L.pkv_paged_decode_attn_noalloc(16, 16, 16, None, None, 16, 4, 16, 4, 64, 8, 96, 16,
                                           8, 0, 0.1, 16, None) == -2

"""GPU parity of paged prefill attention (pkv_paged_prefill_attn, tcgen05 tensor cores):
chunks of new prompt tokens attending causally to each request's paged cache, against
the fp64 oracle's causal multi-query attention on the same seeded inputs.

"深入LLM推理：从KV Cache到PD分离的Serving全景解析": 推理的两阶段计算形态 (prefill),
KV Cache：Transformer的循环状态 (causal attention), PagedAttention与Cache管理 (block table).
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import HostCase, bf16_dev, compare, dev_bits, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _prefill(wl, q_bits, kc, vc, max_q_len=None, q_offsets=None, bt=None, out=None):
    torch = torch_mod()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qo = wl.q_offsets() if q_offsets is None else q_offsets
    out = pkv.paged_prefill_attn(bf16_dev(q_bits), to_dev(qo),
                                 wl.max_q_len if max_q_len is None else max_q_len, kc, vc,
                                 to_dev(wl.block_table if bt is None else bt),
                                 to_dev(wl.seq_lens), wl.scale, out=out, error_word=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def test_prefill_chunks_small_vs_oracle():
    """Ragged chunks (1 .. 300 tokens after contexts of up to 700) on the 70B-shaped layer:
    several query tiles per request, partial last tiles, one chunk with no context."""
    wl = W.make(8, small=True)
    case = HostCase(wl)
    out, err = _prefill(wl, case.d["q"], bf16_dev(case.kc), bf16_dev(case.vc))
    ref = oracle.multiquery_attn(case.d["q"], wl.q_offsets(), case.kc, case.vc, wl.block_table,
                                 wl.seq_lens, wl.scale)
    assert err == 0
    compare(out_to_f64(out), ref, False)


SHAPES = [(Hq, Hkv, D, BS) for (Hq, Hkv) in ((8, 8), (8, 4), (16, 4), (32, 4))
          for D in (64, 128) for BS in (16, 32)]


@pytest.mark.parametrize("Hq,Hkv,D,BS", SHAPES)
def test_prefill_shapes(Hq, Hkv, D, BS):
    seq = np.array([1, 17, 129, 300, 517, 64], np.int32)
    qls = np.array([1, 17, 5, 200, 140, 0], np.int32)
    wl = W.custom(len(seq), Hq, Hkv, D, BS, seq, seed=Hq * 100 + D + BS)
    wl.q_lens = qls
    case = HostCase(wl)
    out, err = _prefill(wl, case.d["q"], bf16_dev(case.kc), bf16_dev(case.vc))
    ref = oracle.multiquery_attn(case.d["q"], wl.q_offsets(), case.kc, case.vc, wl.block_table,
                                 wl.seq_lens, wl.scale)
    assert err == 0
    compare(out_to_f64(out), ref, False)


def test_prefill_matches_multiquery_kernel_for_short_chunks():
    """For q_len <= 4 the decode-family multi-query kernel covers the same rows: both
    paths agree with each other within the attention tolerance."""
    torch = torch_mod()
    wl = W.make(6, small=True)
    case = HostCase(wl)
    kc, vc = bf16_dev(case.kc), bf16_dev(case.vc)
    out_p, err = _prefill(wl, case.d["q"], kc, vc)
    ws = torch.zeros(pkv.multiquery_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, 0, 4),
                     dtype=torch.uint8, device="cuda")
    out_m = pkv.paged_multiquery_attn(bf16_dev(case.d["q"]), to_dev(wl.q_offsets()), 4, kc, vc,
                                      to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale,
                                      workspace=ws)
    torch.cuda.synchronize()
    assert err == 0
    compare(out_to_f64(out_p), out_to_f64(out_m), False)


def test_prefill_nan_poisoned_pool_and_context_shorter_than_chunk():
    """Every cache row no query may see (past each request's length, unused blocks) is
    NaN; requests whose chunk is longer than their cache have rows that see nothing
    (zero rows)."""
    seq = np.array([40, 300, 7], np.int32)
    qls = np.array([50, 180, 7], np.int32)        # request 0: 10 rows see no token
    wl = W.custom(len(seq), 32, 8, 128, 16, seq, seed=9)
    wl.q_lens = qls
    case = HostCase(wl)
    kc, vc = case.kc.copy(), case.vc.copy()
    keep = np.zeros((wl.NB, wl.Hkv, wl.BS), bool)
    for r in range(wl.N):
        for t in range(int(seq[r])):
            keep[wl.block_table[r, t // wl.BS], :, t % wl.BS] = True
    kc[~keep] = 0x7FC0
    vc[~keep] = 0x7FC0
    out, err = _prefill(wl, case.d["q"], bf16_dev(kc), bf16_dev(vc))
    ref = oracle.multiquery_attn(case.d["q"], wl.q_offsets(), kc, vc, wl.block_table,
                                 wl.seq_lens, wl.scale)
    got = out_to_f64(out)
    assert err == 0
    assert np.all(ref[:10] == 0) and np.all(got[:10] == 0)
    compare(got, ref, False)


def test_prefill_flags_bad_ids_and_clamped_chunks():
    torch = torch_mod()
    seq = np.array([200, 100], np.int32)
    qls = np.array([150, 60], np.int32)
    wl = W.custom(2, 16, 4, 128, 16, seq, seed=3)
    wl.q_lens = qls
    case = HostCase(wl)
    kc, vc = bf16_dev(case.kc), bf16_dev(case.vc)
    bt = wl.block_table.copy()
    bt[1, 2] = wl.NB + 5                         # out of range: read as zeros, flagged
    out, err = _prefill(wl, case.d["q"], kc, vc, bt=bt)
    assert err & pkv.DEVERR_BLOCK_RANGE
    assert np.all(np.isfinite(out_to_f64(out)))
    # max_q_len below a chunk: rows past it stay untouched, flagged
    sentinel = torch.full((wl.total_q, wl.Hq, wl.D), 3.0, dtype=torch.bfloat16, device="cuda")
    out, err = _prefill(wl, case.d["q"], kc, vc, max_q_len=100, out=sentinel)
    assert err & pkv.DEVERR_QLEN_CLAMPED
    got = out_to_f64(out)
    assert np.all(got[100:150] == 3.0)
    ref = oracle.multiquery_attn(case.d["q"], wl.q_offsets(), case.kc, case.vc, wl.block_table,
                                 wl.seq_lens, wl.scale)
    compare(got[:100], ref[:100], False)
    compare(got[150:], ref[150:], False)


def test_prefill_deterministic():
    wl = W.make(8, small=True)
    case = HostCase(wl)
    kc, vc = bf16_dev(case.kc), bf16_dev(case.vc)
    a, _ = _prefill(wl, case.d["q"], kc, vc)
    b, _ = _prefill(wl, case.d["q"], kc, vc)
    assert np.array_equal(dev_bits(a), dev_bits(b))


def test_prefill_rejects():
    torch = torch_mod()
    L = pkv.lib()
    z = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = z.data_ptr()

    def call(q=None, total_q=1, max_q_len=1, Hq=8, Hkv=8, D=128, BS=16, dt=0, scale=1.0,
             ks=None, ws=None, ws_bytes=0):
        return L.pkv_paged_prefill_attn(p if q is None else q, p, total_q, max_q_len, p, p, ks,
                                        ks, p, 1, p, 1, Hq, Hkv, D, BS, 4, dt, scale, p, ws,
                                        ws_bytes, None, None)
    assert call(dt=5) == -2                       # not a page kind
    assert call(Hq=12, Hkv=4) == -2               # G = 3
    assert call(D=96) == -2                       # head_dim 96
    assert call(q=p + 2) == -1                    # misaligned q
    assert call(total_q=0, max_q_len=0) == 0      # nothing to do
    for bad in (0.0, -1.0, float("nan"), float("inf")):    # scale must be finite and > 0
        assert call(scale=bad) == -1
    assert call(dt=1) == -1                       # quantised pages need their scales
    assert call(dt=1, ks=p) == -3                 # ... and a workspace
    n = L.pkv_prefill_workspace_size(1, 1, 8, 128, 16, 1)
    assert n > 0 and L.pkv_prefill_workspace_size(1, 1, 8, 128, 16, 0) == 0
    assert call(dt=1, ks=p, ws=p, ws_bytes=n - 1) == -3


@pytest.mark.parametrize("kind", ["fp8", "int8", "int4"])
def test_prefill_over_quantised_pages(kind):
    """Ragged prefill chunks over E4M3 / int8 / int4 pages (the oracle quantises the same
    source rows with its own write): the pages are expanded to bf16, then the tensor-core
    kernel runs; the result is within the quantised-page tolerance of the oracle fed the
    exact dequantised values."""
    torch = torch_mod()
    wl = W.make(8, small=True)
    wl.fp8, wl.int8, wl.int4 = kind == "fp8", kind == "int8", kind == "int4"
    case = HostCase(wl)
    kc = torch.zeros(wl.cache_shape, dtype=torch.int8 if wl.int8 else torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks, vs = to_dev(case.d["k_scale"]), to_dev(case.d["v_scale"])
    slots = pkv.compute_slot_mapping(to_dev(wl.block_table), to_dev(case.pos_all), wl.BS,
                                     req_idx=to_dev(case.req_all))
    pkv.kv_cache_write(bf16_dev(case.d["k_rows"]), bf16_dev(case.d["v_rows"]), slots, kc, vc,
                       ks, vs)
    assert np.array_equal(dev_bits(kc), case.kc) and np.array_equal(dev_bits(vc), case.vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.paged_prefill_attn(bf16_dev(case.d["q"]), to_dev(wl.q_offsets()), wl.max_q_len, kc,
                                 vc, to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale,
                                 k_scale=ks, v_scale=vs, error_word=err)
    torch.cuda.synchronize()
    ref = oracle.multiquery_attn(case.d["q"], wl.q_offsets(), case.kc, case.vc, wl.block_table,
                                 wl.seq_lens, wl.scale, case.d["k_scale"], case.d["v_scale"])
    assert int(err.item()) == 0
    compare(out_to_f64(out), ref, True)


def test_prefill_full_size_sampled():
    """Workload 8 at full size (8 requests x 2048-token chunks after contexts of up to
    6144 tokens) in the bench's launch configuration; 48 sampled (token, head) rows
    against the oracle, including every request's last token (the longest rows)."""
    torch = torch_mod()
    wl = W.make(8)
    dd = W.device_data(wl, torch.device("cuda"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.paged_prefill_attn(dd["q"], to_dev(wl.q_offsets()), wl.max_q_len, dd["k_cache"],
                                 dd["v_cache"], to_dev(wl.block_table), to_dev(wl.seq_lens),
                                 wl.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(8)
    qo = wl.q_offsets()
    toks = [int(qo[r + 1]) - 1 for r in range(wl.N)] + \
        [int(x) for x in rng.integers(0, wl.total_q, size=40)]
    heads = [int(x) for x in rng.integers(0, wl.Hq, size=len(toks))]
    rows = np.array([t * wl.Hq + h for t, h in zip(toks, heads)], np.int64)
    q = dev_bits(dd["q"])
    kc, vc = dev_bits(dd["k_cache"]), dev_bits(dd["v_cache"])
    ref = oracle.multiquery_rows(q, qo, kc, vc, wl.block_table, wl.seq_lens, wl.scale, rows)
    got = out_to_f64(out).reshape(-1, wl.D)[rows]
    compare(got, ref, False)

"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Slot mapping, cache writes and block hashes must match
bit-exactly; attention within the stated tolerances."""
import math

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
    ks = to_dev(case.d["k_scale"])
    vs = to_dev(case.d["v_scale"])
    slots = pkv.compute_slot_mapping(to_dev(wl.block_table), to_dev(case.pos_all), wl.BS,
                                     req_idx=to_dev(case.req_all))
    pkv.kv_cache_write(bf16_dev(case.d["k_rows"]), bf16_dev(case.d["v_rows"]), slots, kc, vc, ks,
                       vs)
    # the library's fp8 pages equal the oracle's byte for byte before the step
    assert np.array_equal(dev_bits(kc), case.kc)
    assert np.array_equal(dev_bits(vc), case.vc)
    return kc, vc, ks, vs


def _gpu_step(case, kc, vc, ks, vs):
    wl = case.wl
    bt = to_dev(wl.block_table)
    sl = to_dev(wl.seq_lens)
    slots = pkv.compute_slot_mapping(bt, to_dev(wl.new_token_positions()), wl.BS)
    pkv.kv_cache_write(bf16_dev(case.d["k_new"]), bf16_dev(case.d["v_new"]), slots, kc, vc, ks, vs)
    ws = pkv.alloc_decode_workspace(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS,
                                    wl.kv_kind)
    out = pkv.paged_decode_attn(bf16_dev(case.d["q"]), kc, vc, bt, sl, wl.scale, k_scale=ks,
                                v_scale=vs, workspace=ws)
    return slots, out, ws


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, 7, 9])
def test_decode_step_small(cfg):
    """Workloads 1..5 at oracle-friendly sizes: slots and cache bytes bit-exact,
    attention within tolerance, device error word clear."""
    wl = W.make(cfg, small=True)
    case = HostCase(wl)
    kc, vc, ks, vs = _device_caches(case)
    slots_d, out_d, ws = _gpu_step(case, kc, vc, ks, vs)
    slots_o, out_o = case.oracle_step()
    assert np.array_equal(slots_d.cpu().numpy(), slots_o)
    assert np.array_equal(dev_bits(kc), case.kc)
    assert np.array_equal(dev_bits(vc), case.vc)
    compare(out_to_f64(out_d), out_o, wl.quant)
    assert pkv.read_device_error(ws) == 0


@pytest.mark.parametrize("G,D,BS,kind", [(1, 64, 16, "bf16"), (2, 128, 32, "bf16"),
                                         (4, 128, 16, "bf16"), (8, 64, 32, "bf16"),
                                         (3, 128, 16, "bf16"), (1, 128, 32, "fp8"),
                                         (4, 128, 16, "fp8"), (8, 128, 32, "fp8"),
                                         (8, 128, 32, "int8"), (2, 128, 16, "int8"),
                                         (8, 128, 32, "int4"), (4, 128, 16, "int4"),
                                         (1, 128, 32, "int4"), (3, 128, 16, "int4")])
def test_decode_shapes_ragged(G, D, BS, kind):
    """Every supported shape on ragged lengths: 1 token, BS-1, BS, BS+1, long tails."""
    Hkv = 2
    lens = [1, BS - 1, BS, BS + 1, 7 * BS + 3, 1000, 37]
    fp8 = kind != "bf16"
    wl = W.custom(len(lens), G * Hkv, Hkv, D, BS, lens, fp8=kind == "fp8", int8=kind == "int8",
                  int4=kind == "int4", seed=G * 100 + D + BS)
    case = HostCase(wl)
    kc, vc, ks, vs = _device_caches(case)
    _, out_d, ws = _gpu_step(case, kc, vc, ks, vs)
    _, out_o = case.oracle_step()
    compare(out_to_f64(out_d), out_o, fp8)
    assert pkv.read_device_error(ws) == 0


def test_decode_empty_and_zero_length_requests():
    """seq_len 0 gives a zero output row; other rows unaffected."""
    torch = torch_mod()
    lens = [0, 5, 0, 300, 0]
    wl = W.custom(len(lens), 8, 2, 128, 16, lens, seed=3)
    wl.block_table[wl.seq_lens == 0] = 0
    d = W.host_data(wl)
    kc, vc = bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"])
    out = pkv.paged_decode_attn(bf16_dev(d["q"]), kc, vc, to_dev(wl.block_table),
                                to_dev(wl.seq_lens), wl.scale)
    ref = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                             wl.scale)
    got = out_to_f64(out)
    assert np.all(got[wl.seq_lens == 0] == 0)
    compare(got, ref, False)
    # batch of all-empty requests
    wl0 = W.custom(3, 8, 2, 128, 16, [0, 0, 0], seed=4)
    out0 = pkv.paged_decode_attn(bf16_dev(W.host_data(wl0)["q"]), kc, vc, to_dev(wl0.block_table),
                                 to_dev(wl0.seq_lens), 0.1)
    assert torch.count_nonzero(out0).item() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_ignores_poisoned_rows(fp8):
    """Rows past a request's length and unused pages hold NaN patterns: outputs stay finite
    and equal the oracle's (which never reads them)."""
    lens = [17, 33, 64, 100, 250]
    wl = W.custom(len(lens), 32, 4, 128, 32, lens, fp8=fp8, seed=11)
    case = HostCase(wl)
    nan_code = 0x7F if fp8 else 0x7FC0
    valid = np.zeros((wl.NB, wl.BS), bool)
    for r in range(wl.N):
        for j, b in enumerate(wl.blocks_of(r)):
            valid[b, :min(wl.BS, int(wl.seq_lens[r]) - j * wl.BS)] = True
    for c in (case.kc, case.vc):
        c.transpose(0, 2, 1, 3)[~valid] = nan_code
    torch = torch_mod()
    if fp8:
        kc, vc = to_dev(case.kc), to_dev(case.vc)
    else:
        kc = to_dev(case.kc.view(np.int16), torch.bfloat16)
        vc = to_dev(case.vc.view(np.int16), torch.bfloat16)
    ks = to_dev(case.d["k_scale"]) if fp8 else None
    vs = to_dev(case.d["v_scale"]) if fp8 else None
    out = pkv.paged_decode_attn(bf16_dev(case.d["q"]), kc, vc, to_dev(wl.block_table),
                                to_dev(wl.seq_lens), wl.scale, k_scale=ks, v_scale=vs)
    ref = oracle.decode_attn(case.d["q"], case.kc, case.vc, wl.block_table, wl.seq_lens, wl.scale,
                             case.d.get("k_scale"), case.d.get("v_scale"))
    compare(out_to_f64(out), ref, fp8)


def test_decode_single_long_request_split_everywhere():
    """One request longer than the grid: every warp holds a slice, the reduce merges
    up to a few hundred partials per unit."""
    lens = [20000]
    wl = W.custom(1, 8, 1, 128, 16, lens, seed=5)
    case = HostCase(wl)
    kc, vc, ks, vs = _device_caches(case)
    _, out_d, ws = _gpu_step(case, kc, vc, ks, vs)
    _, out_o = case.oracle_step()
    compare(out_to_f64(out_d), out_o, False)
    assert pkv.read_device_error(ws) == 0


def test_decode_is_deterministic():
    wl = W.make(2, small=True)
    case = HostCase(wl)
    kc, vc, ks, vs = _device_caches(case)
    q = bf16_dev(case.d["q"])
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    a = dev_bits(pkv.paged_decode_attn(q, kc, vc, bt, sl, wl.scale))
    b = dev_bits(pkv.paged_decode_attn(q, kc, vc, bt, sl, wl.scale))
    assert np.array_equal(a, b)


def test_decode_invariant_under_block_relabel():
    """Relabelling physical blocks (pool and table together) changes no output bit."""
    torch = torch_mod()
    wl = W.make(2, small=True)
    d = W.host_data(wl)
    q = bf16_dev(d["q"])
    out1 = dev_bits(pkv.paged_decode_attn(q, bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"]),
                                          to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale))
    perm = np.random.default_rng(1).permutation(wl.NB)
    kc2 = np.empty_like(d["k_cache"]); kc2[perm] = d["k_cache"]
    vc2 = np.empty_like(d["v_cache"]); vc2[perm] = d["v_cache"]
    bt2 = perm[wl.block_table].astype(np.int32)
    out2 = dev_bits(pkv.paged_decode_attn(q, bf16_dev(kc2), bf16_dev(vc2), to_dev(bt2),
                                          to_dev(wl.seq_lens), wl.scale))
    assert np.array_equal(out1, out2)


def test_decode_bad_block_ids_and_lengths_are_flagged_not_read():
    """Out-of-range block ids read as zeros and set PKV_DEVERR_BLOCK_RANGE; a length past
    the table is clamped and sets PKV_DEVERR_SEQ_CLAMPED.  Nothing faults."""
    wl = W.custom(3, 8, 2, 128, 16, [40, 40, 40], seed=8)
    d = W.host_data(wl)
    bt = wl.block_table.copy()
    bt[1, 1] = wl.NB + 5
    bt[2, 0] = -3
    sl = wl.seq_lens.copy()
    sl[0] = 10 ** 6
    ws = pkv.alloc_decode_workspace(3, 8, 2, 128, 16, pkv.BF16)
    out = pkv.paged_decode_attn(bf16_dev(d["q"]), bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"]),
                                to_dev(bt), to_dev(sl), wl.scale, workspace=ws)
    err = pkv.read_device_error(ws)
    assert err & pkv.DEVERR_BLOCK_RANGE and err & pkv.DEVERR_SEQ_CLAMPED
    assert not (err & pkv.DEVERR_WAIT_TIMEOUT)
    assert np.all(np.isfinite(out_to_f64(out)))


# ---------------------------------------------------------------- write / slots
def test_fp8_write_exhaustive_bf16_patterns():
    """Every bf16 bit pattern through the FP8 write, scale 1 and random scales: the
    library's bytes equal the oracle's (NaN inputs: both give a NaN code)."""
    torch = torch_mod()
    bits = np.arange(65536, dtype=np.uint16).reshape(512, 1, 128)
    T, BS, NB = 512, 16, 32
    slots = np.arange(T, dtype=np.int64)
    rng = np.random.default_rng(2)
    for scales in (np.ones((NB, 1), np.float32),
                   rng.uniform(0.001, 3.0, (NB, 1)).astype(np.float32),
                   (2.0 ** rng.integers(-8, 8, (NB, 1))).astype(np.float32)):
        kc_o = np.zeros((NB, 1, BS, 128), np.uint8)
        vc_o = np.zeros_like(kc_o)
        oracle.kv_cache_write(bits, bits[::-1].copy(), slots, kc_o, vc_o, scales, scales)
        kc = torch.zeros((NB, 1, BS, 128), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        pkv.kv_cache_write(bf16_dev(bits), bf16_dev(bits[::-1].copy()), to_dev(slots), kc, vc,
                           to_dev(scales), to_dev(scales))
        for got, ref in ((dev_bits(kc), kc_o), (dev_bits(vc), vc_o)):
            nan_ref = (ref & 0x7F) == 0x7F
            nan_got = (got & 0x7F) == 0x7F
            assert np.array_equal(nan_ref, nan_got)
            assert np.array_equal(got[~nan_ref], ref[~nan_ref])


def test_int8_write_exhaustive_bf16_patterns():
    """Every bf16 bit pattern through the int8 write with scale 1 and random scales:
    the library's bytes equal the oracle's."""
    torch = torch_mod()
    bits = np.arange(65536, dtype=np.uint16).reshape(512, 1, 128)
    T, BS, NB = 512, 16, 32
    slots = np.arange(T, dtype=np.int64)
    rng = np.random.default_rng(3)
    for scales in (np.ones((NB, 1), np.float32),
                   rng.uniform(0.001, 3.0, (NB, 1)).astype(np.float32)):
        kc_o = np.zeros((NB, 1, BS, 128), np.int8)
        vc_o = np.zeros_like(kc_o)
        oracle.kv_cache_write(bits, bits[::-1].copy(), slots, kc_o, vc_o, scales, scales)
        kc = torch.zeros((NB, 1, BS, 128), dtype=torch.int8, device="cuda")
        vc = torch.zeros_like(kc)
        pkv.kv_cache_write(bf16_dev(bits), bf16_dev(bits[::-1].copy()), to_dev(slots), kc, vc,
                           to_dev(scales), to_dev(scales))
        assert np.array_equal(dev_bits(kc), kc_o)
        assert np.array_equal(dev_bits(vc), vc_o)


def test_int4_write_exhaustive_bf16_patterns():
    """Every bf16 bit pattern through the int4 write (two codes per byte) with scale 1 and
    random scales: the library's bytes equal the oracle's."""
    torch = torch_mod()
    bits = np.arange(65536, dtype=np.uint16).reshape(512, 1, 128)
    T, BS, NB = 512, 16, 32
    slots = np.arange(T, dtype=np.int64)
    rng = np.random.default_rng(4)
    for scales in (np.ones((NB, 1), np.float32),
                   rng.uniform(0.001, 3.0, (NB, 1)).astype(np.float32)):
        kc_o = np.zeros((NB, 1, BS, 64), np.uint8)
        vc_o = np.zeros_like(kc_o)
        oracle.kv_cache_write(bits, bits[::-1].copy(), slots, kc_o, vc_o, scales, scales)
        kc = torch.zeros((NB, 1, BS, 64), dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        pkv.kv_cache_write(bf16_dev(bits), bf16_dev(bits[::-1].copy()), to_dev(slots), kc, vc,
                           to_dev(scales), to_dev(scales))
        assert np.array_equal(dev_bits(kc), kc_o)
        assert np.array_equal(dev_bits(vc), vc_o)


def test_slot_mapping_padding_and_req_idx():
    rng = np.random.default_rng(12)
    wl = W.make(4, small=True)
    T = 500
    req = rng.integers(0, wl.N, T).astype(np.int32)
    pos = np.array([rng.integers(-2, int(wl.seq_lens[r])) for r in req], np.int32)
    ref = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    got = pkv.compute_slot_mapping(to_dev(wl.block_table), to_dev(pos), wl.BS,
                                   req_idx=to_dev(req)).cpu().numpy()
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- hash
def _hash_both(tokens, offsets, B, seed):
    ref, ho = oracle.prefix_block_hash(tokens, offsets, B, seed)
    torch = torch_mod()
    tok = to_dev(tokens if tokens.size else np.zeros(1, np.int32))
    got = pkv.prefix_block_hash(tok, to_dev(offsets), B, to_dev(ho), int(ho[-1]), seed=seed)
    return got.cpu().numpy().view(np.uint64), ref


@pytest.mark.parametrize("cfg,small", [(1, False), (4, False), (3, True), (2, True)])
def test_prefix_hash_bit_exact(cfg, small):
    wl = W.make(cfg, small=small)
    got, ref = _hash_both(wl.tokens, wl.token_offsets, wl.hash_block, 0x5EED)
    assert np.array_equal(got, ref)
    if cfg == 4:
        npre = wl.notes["shared_prefix_blocks"]
        ho = oracle.hash_offsets(wl.token_offsets, wl.hash_block)
        first = got[ho[0]:ho[0] + npre]
        for r in range(wl.N):
            assert np.array_equal(got[ho[r]:ho[r] + npre], first)


def test_prefix_hash_long_sequence_and_odd_block_sizes():
    rng = np.random.default_rng(31)
    lens = [131072, 0, 5, 4097, 33]
    toks = rng.integers(0, 128000, sum(lens)).astype(np.int32)
    offs = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(lens, out=offs[1:])
    for B in (16, 32, 7, 1):
        got, ref = _hash_both(toks, offs, B, B)
        assert np.array_equal(got, ref)


def _resume_both(tokens, offsets, B, prev, first, ho):
    ref, _ = oracle.prefix_block_hash_resume(tokens, offsets, B, prev, first, ho)
    torch = __import__("torch")
    tok = to_dev(tokens if tokens.size else np.zeros(1, np.int32))
    n = int(ho[-1])
    out = torch.full((max(n, 1),), 0x5A5A5A5A, dtype=torch.int64, device="cuda")
    got = pkv.prefix_block_hash_resume(tok, to_dev(offsets), B,
                                       to_dev(np.asarray(prev, np.uint64).view(np.int64)),
                                       to_dev(np.asarray(first, np.int64)), to_dev(ho), n, out=out)
    g = out.cpu().numpy().view(np.uint64)
    return g, ref, got


@pytest.mark.parametrize("B", [16, 32, 7])
def test_prefix_hash_resume_bit_exact(B):
    """Resumed chains equal the oracle's bit for bit: every sequence cut at its own point
    (none hashed, some, all, past the end, negative), the previous hash taken from the
    full chain; a 131,072-token sequence resumed near its start (several digest chunks)
    and at its last block (one block, the decode-step case)."""
    rng = np.random.default_rng(41)
    lens = [131072, 131072, 0, 5, 4097, 33, 16 * 40, 16 * 40 + 9, 3000]
    toks = rng.integers(0, 128000, sum(lens)).astype(np.int32)
    offs = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(lens, out=offs[1:])
    full, fho = oracle.prefix_block_hash(toks, offs, B, 0xC0FFEE)
    nfull = np.diff(offs) // B
    first = np.array([3, nfull[1] - 1, 0, 0, nfull[4] // 2, nfull[5], nfull[6] + 4, -2, 1],
                     np.int64)
    prev = np.array([full[fho[s] + min(max(int(first[s]), 0), int(nfull[s])) - 1]
                     if min(max(int(first[s]), 0), int(nfull[s])) > 0 else 0xC0FFEE
                     for s in range(len(lens))], np.uint64)
    n = np.maximum(nfull - np.clip(first, 0, None), 0)
    ho = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(n, out=ho[1:])
    got, ref, _ = _resume_both(toks, offs, B, prev, first, ho)
    assert np.array_equal(got[:int(ho[-1])], ref)
    # the resumed hashes are the full chain's suffixes
    for s in range(len(lens)):
        k = min(max(int(first[s]), 0), int(nfull[s]))
        assert np.array_equal(ref[ho[s]:ho[s + 1]], full[fho[s] + k:fho[s + 1]])


def test_prefix_hash_resume_room_limits_and_untouched_tail():
    rng = np.random.default_rng(42)
    B = 16
    lens = [16 * 9, 16 * 5 + 1, 16 * 3000]
    toks = rng.integers(0, 128000, sum(lens)).astype(np.int32)
    offs = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(lens, out=offs[1:])
    full, fho = oracle.prefix_block_hash(toks, offs, B, 7)
    first = np.array([3, 0, 10], np.int64)
    prev = np.array([full[fho[0] + 2], 7, full[fho[2] + 9]], np.uint64)
    ho = np.array([0, 2, 12, 12 + 2500], np.int64)      # rooms 2 (needs 6), 10 (5), 2500 (2990)
    got, ref, _ = _resume_both(toks, offs, B, prev, first, ho)
    assert np.array_equal(got[:2], ref[:2]) and np.array_equal(got[:2], full[3:5])
    assert np.array_equal(got[2:7], full[fho[1]:fho[2]])
    assert np.all(got[7:12] == 0x5A5A5A5A)                # past the chain's end: untouched
    assert np.array_equal(got[12:], full[fho[2] + 10:fho[2] + 10 + 2500])
    assert np.array_equal(got[12:], ref[12:])


def test_decode_workspace_reuse_and_garbage_contents():
    """One workspace shared by successive calls of different shapes, starting from
    garbage bytes: the page prefix and the partial slots are written before they are
    read, so nothing in the workspace needs clearing."""
    torch = torch_mod()
    cases = [W.custom(3, 16, 2, 128, 16, [40, 5000, 700], seed=41),     # pages > warps
             W.custom(5, 16, 2, 128, 16, [3, 17, 1, 33, 64], seed=42),  # pages < warps
             W.make(2, small=True)]
    n = max(pkv.decode_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, pkv.BF16) for wl in cases)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:4] = 0   # the error word
    for rep in range(2):
        for wl in cases:
            d = W.host_data(wl)
            out = pkv.paged_decode_attn(bf16_dev(d["q"]), bf16_dev(d["k_cache"]),
                                        bf16_dev(d["v_cache"]), to_dev(wl.block_table),
                                        to_dev(wl.seq_lens), wl.scale, workspace=ws)
            ref = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table,
                                     wl.seq_lens, wl.scale)
            compare(out_to_f64(out), ref, False)
    assert pkv.read_device_error(ws) == 0

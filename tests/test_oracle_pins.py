"""Pins of the CPU oracle to facts other than itself (no GPU).

Each test anchors one oracle function to something independent: numbers the
sources print, published test vectors, library codecs (torch CPU dtypes),
closed forms, brute force, or invariants a plausible bug would break.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_289_gb300 import workloads as W
from conftest import golden_rows


# ---------------------------------------------------------------- KV size
def test_kv_size_formula_matches_printed_values():
    rows = golden_rows("kv_size.txt")
    assert rows
    for L, Hkv, d, S, b, expect in rows:
        assert oracle.kv_bytes(int(L), int(Hkv), int(d), int(S), int(b)) == int(expect)


def test_kv_size_fp8_halves_bytes():
    # "ai-infra-7", 传输量化: FP8 halves the bytes of FP16
    assert 2 * oracle.kv_bytes(80, 8, 128, 4096, 1) == oracle.kv_bytes(80, 8, 128, 4096, 2)


# ---------------------------------------------------------------- codecs
def test_bf16_decode_matches_torch_for_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_e4m3_decode_spec_points():
    for code, val in golden_rows("e4m3_spec.txt"):
        got = oracle.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_encode_matches_torch_below_saturation():
    # every finite bf16 value with |x| < 448: round to nearest, ties to even
    bits = np.arange(65536, dtype=np.uint16)
    x = W.bf16_bits_to_f32(bits)
    keep = np.isfinite(x) & (np.abs(x) < 448.0)
    xs = x[keep]
    ref = torch.from_numpy(xs.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(v)) for v in xs], dtype=np.uint8)
    # +0 / -0 both fine for values that round to zero only if the sign matches torch's
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates_and_nan():
    for v in (448.0, 448.5, 463.9, 464.0, 500.0, 1e30, float("inf")):
        assert oracle.e4m3_from_float(v) == 0x7E
        assert oracle.e4m3_from_float(-v) == 0xFE
    assert oracle.e4m3_from_float(float("nan")) & 0x7F == 0x7F


def _brute_e4m3(x):
    """Nearest finite E4M3 value by exhaustive search over the decoded codes;
    ties to the even code; saturate beyond the largest finite value."""
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0x00
    # rounding acts on the magnitude; the sign of x is kept (so -tiny -> -0)
    codes = np.array([sign | c for c in range(0x7F)], dtype=np.int64)
    vals = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if abs(x) >= 448.0:
        return sign | 0x7E
    dist = np.abs(vals - x)
    cand = codes[dist == dist.min()]
    even = [c for c in cand if c % 2 == 0]     # ties: even mantissa
    return int(even[0] if even else cand[0])


def test_e4m3_encode_brute_force_on_binary32_inputs():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 100,
        rng.standard_normal(2000).astype(np.float32) * 0.01,
        np.float32([0.0625 * k for k in range(-80, 81)]),          # many exact ties
        np.float32([2.0 ** -10 * k for k in range(-40, 41)]),      # subnormal ties
        np.float32([440.0, 447.99, -447.99, 0.0009765625, 0.00146484375]),
    ])
    for x in xs:
        assert oracle.e4m3_from_float(float(x)) == _brute_e4m3(float(x)), x


# ---------------------------------------------------------------- slot mapping / write
def test_slot_mapping_worked_example():
    rows = golden_rows("slot_mapping_example.txt")
    bt = np.array([[5, 2, 7], [3, 0, 0]], dtype=np.int32)
    req = np.array([int(r[0]) for r in rows], np.int32)
    pos = np.array([int(r[1]) for r in rows], np.int32)
    expect = np.array([int(r[2]) for r in rows], np.int64)
    assert np.array_equal(oracle.slot_mapping(bt, req, pos, 16), expect)


def _bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_write_leaves_other_bytes_and_copies_bf16_bytes():
    wl = W.make(1)
    d = W.host_data(wl)
    kc, vc = d["k_cache"].copy(), d["v_cache"].copy()
    req = np.arange(wl.N, dtype=np.int32)
    slots = oracle.slot_mapping(wl.block_table, req, wl.new_token_positions(), wl.BS)
    slots[1] = -1  # a padding token is skipped
    oracle.kv_cache_write(d["k_new"], d["v_new"], slots, kc, vc)
    changed = np.zeros(kc.shape[:3], bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), wl.BS)
        changed[b, :, o] = True
        assert np.array_equal(kc[b, :, o], d["k_new"][t])
        assert np.array_equal(vc[b, :, o], d["v_new"][t])
    assert changed.sum() == (wl.N - 1) * wl.Hkv
    assert np.array_equal(kc[~changed], d["k_cache"][~changed])
    assert np.array_equal(vc[~changed], d["v_cache"][~changed])


def test_write_then_attend_returns_the_written_value():
    # Links slot mapping + write to the attention gather: make the new token's key the
    # only non-zero key, aligned with q and large, so softmax is one-hot on it and the
    # output equals the new value row (closed form).
    wl = W.make(1)
    D = wl.D
    kc = np.zeros((wl.NB, wl.Hkv, wl.BS, D), np.uint16)
    vc = _bf16(np.random.default_rng(3).standard_normal((wl.NB, wl.Hkv, wl.BS, D)))
    q = _bf16(np.ones((wl.N, wl.Hq, D)))
    k_new = _bf16(np.full((wl.N, wl.Hkv, D), 8.0))
    v_new = _bf16(np.random.default_rng(4).standard_normal((wl.N, wl.Hkv, D)))
    req = np.arange(wl.N, dtype=np.int32)
    slots = oracle.slot_mapping(wl.block_table, req, wl.new_token_positions(), wl.BS)
    oracle.kv_cache_write(k_new, v_new, slots, kc, vc)
    out = oracle.decode_attn(q, kc, vc, wl.block_table, wl.seq_lens, 1.0)
    vref = W.bf16_bits_to_f32(v_new).astype(np.float64)
    for r in range(wl.N):
        for hq in range(wl.Hq):
            np.testing.assert_allclose(out[r, hq], vref[r, hq // wl.G], atol=1e-12)


def test_fp8_write_error_within_half_spacing():
    wl = W.make(5, small=True)
    d = W.host_data(wl)
    req, pos = W.token_rows_order(wl)
    slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    kc = np.zeros((wl.NB, wl.Hkv, wl.BS, wl.D), np.uint8)
    vc = np.zeros_like(kc)
    oracle.kv_cache_write(d["k_rows"], d["v_rows"], slots, kc, vc, d["k_scale"], d["v_scale"])
    table = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    x = W.bf16_bits_to_f32(d["k_rows"]).astype(np.float64)
    b = slots // wl.BS
    o = slots % wl.BS
    codes = kc[b, :, o]                                  # [T, Hkv, D]
    s = d["k_scale"][b].astype(np.float64)[:, :, None]   # [T, Hkv, 1]
    y = x / s                                            # the value before rounding
    got = table[codes]
    # spacing of E4M3 around |y|: 2^(e-3) for normals (e = floor log2 |y| >= -6), 2^-9 below
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
    half = np.where(np.abs(y) < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
    # the binary32 division adds at most one binary32 rounding of y
    assert np.all(np.abs(got - y) <= half * (1 + 1e-6) + np.abs(y) * 2.0 ** -24)
    # amax/448 scaling: every block's largest magnitude lands on +-448 (or one ulp below it
    # if the binary32 divide rounds under 448)
    assert np.abs(got).max() == 448.0


# ---------------------------------------------------------------- attention
def _paged_from_dense(rng, K, V, BS, NB_extra=3):
    """Scatter dense per-request K/V [S_r, Hkv, D] into a paged bf16 cache, block ids
    drawn from a random permutation (test-side scatter, independent of the oracle)."""
    N = len(K)
    Hkv, D = K[0].shape[1], K[0].shape[2]
    nblk = [-(-k.shape[0] // BS) for k in K]
    NB = sum(nblk) + NB_extra
    ids = rng.permutation(NB)
    kc = _bf16(rng.standard_normal((NB, Hkv, BS, D)))   # garbage everywhere else
    vc = _bf16(rng.standard_normal((NB, Hkv, BS, D)))
    bt = np.zeros((N, max(nblk)), np.int32)
    o = 0
    for r in range(N):
        for j in range(nblk[r]):
            bt[r, j] = ids[o]
            rows = K[r][j * BS:(j + 1) * BS]
            kc[ids[o], :, :rows.shape[0]] = rows.transpose(1, 0, 2)
            vc[ids[o], :, :rows.shape[0]] = V[r][j * BS:(j + 1) * BS].transpose(1, 0, 2)
            o += 1
    return kc, vc, bt


def _dense_reference(q, K, V, scale, G):
    """softmax(scale q K^T) V with numpy/scipy library routines, fp64."""
    out = []
    for r in range(len(K)):
        Kr = W.bf16_bits_to_f32(K[r]).astype(np.float64)   # [S, Hkv, D]
        Vr = W.bf16_bits_to_f32(V[r]).astype(np.float64)
        qr = W.bf16_bits_to_f32(q[r]).astype(np.float64)   # [Hq, D]
        o = []
        for hq in range(qr.shape[0]):
            s = scale * (Kr[:, hq // G, :] @ qr[hq])
            p = scipy.special.softmax(s)
            o.append(p @ Vr[:, hq // G, :])
        out.append(np.stack(o))
    return np.stack(out)


@pytest.mark.parametrize("BS,G,D", [(16, 4, 64), (32, 8, 128), (16, 1, 32)])
def test_decode_matches_dense_bruteforce(BS, G, D):
    rng = np.random.default_rng(11 + BS + G)
    Hkv = 2
    lens = [1, BS - 1, BS, 3 * BS + 5]
    K = [_bf16(rng.standard_normal((S, Hkv, D))) for S in lens]
    V = [_bf16(rng.standard_normal((S, Hkv, D))) for S in lens]
    q = _bf16(rng.standard_normal((len(lens), Hkv * G, D)))
    kc, vc, bt = _paged_from_dense(rng, K, V, BS)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode_attn(q, kc, vc, bt, np.array(lens, np.int32), scale)
    ref = _dense_reference(q, K, V, scale, G)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_decode_invariant_under_physical_block_relabel():
    wl = W.make(1)
    d = W.host_data(wl)
    out = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                             wl.scale)
    perm = np.random.default_rng(5).permutation(wl.NB)     # new id of old block b = perm[b]
    kc2 = np.empty_like(d["k_cache"])
    vc2 = np.empty_like(d["v_cache"])
    kc2[perm] = d["k_cache"]
    vc2[perm] = d["v_cache"]
    bt2 = perm[wl.block_table].astype(np.int32)
    out2 = oracle.decode_attn(d["q"], kc2, vc2, bt2, wl.seq_lens, wl.scale)
    assert np.array_equal(out, out2)


def test_gqa_equals_mha_with_replicated_kv_heads():
    wl = W.make(1)                                          # Hkv = 1, G = 4
    d = W.host_data(wl)
    out = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                             wl.scale)
    kc = np.repeat(d["k_cache"], wl.Hq, axis=1)             # Hkv' = Hq, G' = 1
    vc = np.repeat(d["v_cache"], wl.Hq, axis=1)
    out_mha = oracle.decode_attn(d["q"], kc, vc, wl.block_table, wl.seq_lens, wl.scale)
    assert np.array_equal(out, out_mha)


def test_probabilities_are_a_distribution():
    wl = W.make(2, small=True)
    d = W.host_data(wl)
    for r, hq in [(0, 0), (3, 17), (7, 63)]:
        o, p, lse = oracle.decode_row_detail(d["q"], d["k_cache"], d["v_cache"], wl.block_table,
                                             wl.seq_lens, wl.scale, r, hq)
        assert p.shape[0] == wl.seq_lens[r]
        assert np.all(p >= 0)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.isfinite(lse)


def test_closed_form_special_cases():
    rng = np.random.default_rng(9)
    BS, D, Hkv, G = 16, 64, 1, 2
    # (a) one token: output is that token's value row
    K = [_bf16(rng.standard_normal((1, Hkv, D)))]
    V = [_bf16(rng.standard_normal((1, Hkv, D)))]
    q = _bf16(rng.standard_normal((1, G, D)))
    kc, vc, bt = _paged_from_dense(rng, K, V, BS)
    out = oracle.decode_attn(q, kc, vc, bt, np.array([1], np.int32), 0.125)
    v0 = W.bf16_bits_to_f32(V[0][0, 0]).astype(np.float64)
    assert np.array_equal(out[0, 0], v0) and np.array_equal(out[0, 1], v0)
    # (b) identical keys, or (c) q = 0, or (d) scale 0: output is the mean of V
    S = 45
    Vs = [_bf16(rng.standard_normal((S, Hkv, D)))]
    vmean = W.bf16_bits_to_f32(Vs[0][:, 0]).astype(np.float64).mean(axis=0)
    same_k = np.repeat(_bf16(rng.standard_normal((1, Hkv, D))), S, axis=0)
    for Ks, qq, sc in [([same_k], q, 0.125),
                       ([_bf16(rng.standard_normal((S, Hkv, D)))], np.zeros_like(q), 0.125),
                       ([_bf16(rng.standard_normal((S, Hkv, D)))], q, 0.0)]:
        kc, vc, bt = _paged_from_dense(rng, Ks, Vs, BS)
        out = oracle.decode_attn(qq, kc, vc, bt, np.array([S], np.int32), sc)
        np.testing.assert_allclose(out[0, 0], vmean, atol=1e-13)


def test_split_lse_merge_equals_unsplit():
    # Online-softmax equivalence ("GPU推理深度拆解：KV Cache视角", 算子优化要点 and
    # 系统层：Context Parallel): attention over two disjoint token ranges merged by
    # log-sum-exp weights equals attention over the union.
    wl = W.make(3, small=True)
    d = W.host_data(wl)
    r, BS = 2, wl.BS
    S = int(wl.seq_lens[r])
    for cut_blocks in (1, 7, (S // BS) - 1):
        cut = cut_blocks * BS
        bt = np.zeros((3, wl.MB), np.int32)
        blocks = wl.blocks_of(r)
        bt[0, :len(blocks)] = blocks                      # the whole request
        bt[1, :cut_blocks] = blocks[:cut_blocks]          # first part
        bt[2, :len(blocks) - cut_blocks] = blocks[cut_blocks:]  # second part
        lens = np.array([S, cut, S - cut], np.int32)
        q = np.repeat(d["q"][r:r + 1], 3, axis=0)
        for hq in (0, 9, 63):
            res = [oracle.decode_row_detail(q, d["k_cache"], d["v_cache"], bt, lens, wl.scale, i,
                                            hq) for i in range(3)]
            (o, _, lse), (o1, _, l1), (o2, _, l2) = res
            m = max(l1, l2)
            w1, w2 = math.exp(l1 - m), math.exp(l2 - m)
            merged = (w1 * o1 + w2 * o2) / (w1 + w2)
            np.testing.assert_allclose(merged, o, atol=1e-12)
            assert abs(lse - (m + math.log(w1 + w2))) < 1e-12


def test_fp8_decode_uses_dequantised_values():
    # fp8 oracle == bf16-free fp64 computation on decode(code) * scale, done densely.
    wl = W.make(5, small=True)
    d = W.host_data(wl)
    req, pos = W.token_rows_order(wl)
    slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    kc = np.zeros((wl.NB, wl.Hkv, wl.BS, wl.D), np.uint8)
    vc = np.zeros_like(kc)
    oracle.kv_cache_write(d["k_rows"], d["v_rows"], slots, kc, vc, d["k_scale"], d["v_scale"])
    table = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    rows = np.array([0, 5 * wl.Hq + 33, (wl.N - 1) * wl.Hq + 63], np.int64)
    got = oracle.decode_rows(d["q"], kc, vc, wl.block_table, wl.seq_lens, wl.scale, rows,
                             d["k_scale"], d["v_scale"])
    for i, row in enumerate(rows):
        r, hq = divmod(int(row), wl.Hq)
        h = hq // wl.G
        blocks = wl.blocks_of(r)
        S = int(wl.seq_lens[r])
        Kd = np.concatenate([table[kc[b, h]] * float(d["k_scale"][b, h]) for b in blocks])[:S]
        Vd = np.concatenate([table[vc[b, h]] * float(d["v_scale"][b, h]) for b in blocks])[:S]
        qv = W.bf16_bits_to_f32(d["q"][r, hq]).astype(np.float64)
        p = scipy.special.softmax(wl.scale * (Kd @ qv))
        np.testing.assert_allclose(got[i], p @ Vd, atol=1e-12)


# ---------------------------------------------------------------- hash
def test_hash_primitives_published_vectors():
    for row in golden_rows("hash_vectors.txt"):
        if row[0] == "fnv1a64":
            s = row[1].strip('"').encode("ascii")
            assert oracle.fnv1a64(s) == int(row[2], 16)
        else:
            k = int(row[1])
            z = (k * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
            assert oracle.fmix64(z) == int(row[2], 16)


def _hash(seqs, B=16, seed=0x1234):
    toks = np.concatenate([np.asarray(s, np.int32) for s in seqs]) if seqs else np.zeros(0, np.int32)
    offs = np.zeros(len(seqs) + 1, np.int64)
    np.cumsum([len(s) for s in seqs], out=offs[1:])
    h, ho = oracle.prefix_block_hash(toks, offs, B, seed)
    return [h[ho[i]:ho[i + 1]] for i in range(len(seqs))]


def test_hash_token_exact_prefix_properties():
    rng = np.random.default_rng(21)
    B = 16
    base = rng.integers(0, 128000, 10 * B + 7).astype(np.int32)
    hs = _hash([base])[0]
    assert len(hs) == 10                                  # partial tail block: no hash
    # prefix consistency: a truncated sequence gets the same leading hashes
    for n in (B, 3 * B, 3 * B + 5, 10 * B):
        assert np.array_equal(_hash([base[:n]])[0], hs[: n // B])
    # changing one token in block j changes hashes j.. and none before
    for j in (0, 4, 9):
        for pos in (j * B, j * B + 7, j * B + B - 1):
            mod = base.copy()
            mod[pos] = (mod[pos] + 1) % 128000
            h2 = _hash([mod])[0]
            assert np.array_equal(h2[:j], hs[:j])
            assert np.all(h2[j:] != hs[j:])
    # a change in the partial tail changes nothing
    mod = base.copy()
    mod[-1] += 1
    assert np.array_equal(_hash([mod])[0], hs)
    # the seed enters every hash
    assert np.all(_hash([base], seed=1)[0] != _hash([base], seed=2)[0])
    # a block whose bytes are the same as another's but at another position differs
    rep = np.tile(base[:B], 4)
    hr = _hash([rep])[0]
    assert len(set(hr.tolist())) == 4


def test_hash_prefix_sharing_workload():
    wl = W.make(4, small=True)
    h, ho = oracle.prefix_block_hash(wl.tokens, wl.token_offsets, 16, 0)
    npre = wl.notes["shared_prefix_blocks"]
    first = h[ho[0]:ho[0] + npre]
    all_hashes = set()
    for r in range(wl.N):
        hr = h[ho[r]:ho[r + 1]]
        assert np.array_equal(hr[:npre], first)          # shared blocks: identical hashes
        all_hashes.update(hr[npre:].tolist())
    # tails are distinct random tokens: no collisions among distinct prefixes
    assert len(all_hashes) == int(ho[-1]) - wl.N * npre
    assert not (all_hashes & set(first.tolist()))


def test_hash_empty_and_short_sequences():
    out = _hash([[], [1, 2, 3], list(range(16))])
    assert len(out[0]) == 0 and len(out[1]) == 0 and len(out[2]) == 1


def test_hash_resume_continues_the_chain_at_every_cut():
    """h_i = H(h_{i-1}, block i): continuing from h_k over the same tokens gives exactly
    h_{k+1}, h_{k+2}, ... of the whole chain, for every cut k (the published-vector-pinned
    chain above is the reference).  Several sequences at once, each cut independently."""
    rng = np.random.default_rng(23)
    B, seed = 16, 0x1234
    seqs = [rng.integers(0, 128000, n).astype(np.int32) for n in (0, 5, 16, 16 * 7 + 3, 16 * 12)]
    whole = _hash(seqs, B, seed)
    toks = np.concatenate(seqs)
    offs = np.zeros(len(seqs) + 1, np.int64)
    np.cumsum([len(s) for s in seqs], out=offs[1:])
    for cut in range(0, 14):
        first = np.array([cut] * len(seqs), np.int64)
        prev = np.array([seed if min(cut, len(w)) == 0 else int(w[min(cut, len(w)) - 1])
                         for w in whole], np.uint64)
        got, ho = oracle.prefix_block_hash_resume(toks, offs, B, prev, first)
        for s, w in enumerate(whole):
            assert np.array_equal(got[ho[s]:ho[s + 1]], w[cut:]), (cut, s)
    # mixed cuts, one per sequence, including one past the last full block
    first = np.array([0, 0, 1, 3, 12], np.int64)
    prev = np.array([seed, seed, whole[2][0], whole[3][2], whole[4][11]], np.uint64)
    got, ho = oracle.prefix_block_hash_resume(toks, offs, B, prev, first)
    assert np.diff(ho).tolist() == [0, 0, 0, 4, 0]
    assert np.array_equal(got, whole[3][3:])
    # a negative count of blocks already hashed starts the chain at prev as h_0
    got, _ = oracle.prefix_block_hash_resume(toks, offs, B, [seed] * 5, [-3] * 5)
    assert np.array_equal(got, np.concatenate(whole))


def test_hash_resume_respects_the_room_per_sequence():
    """hash_offsets gives each sequence's room: a short room takes the first hashes of
    the continued chain and nothing is written past it."""
    rng = np.random.default_rng(24)
    B, seed = 16, 99
    seqs = [rng.integers(0, 128000, n).astype(np.int32) for n in (16 * 9, 16 * 5 + 1)]
    whole = _hash(seqs, B, seed)
    toks = np.concatenate(seqs)
    offs = np.array([0, len(seqs[0]), len(seqs[0]) + len(seqs[1])], np.int64)
    ho = np.array([0, 2, 2 + 10], np.int64)               # room 2 (needs 6), room 10 (needs 5)
    got, _ = oracle.prefix_block_hash_resume(toks, offs, B, [whole[0][2], seed], [3, 0], ho)
    assert np.array_equal(got[:2], whole[0][3:5])
    assert np.array_equal(got[2:7], whole[1])
    assert np.all(got[7:] == 0)                            # untouched past the chain's end


# ---------------------------------------------------------------- multi-query (verify) attention
def _dense_causal(q, qoffs, K, V, scale, G):
    """Query i of request r (its newest tokens) over positions 0..S-q_len+i, with scipy."""
    out = np.zeros((q.shape[0], q.shape[1], q.shape[2]))
    for r in range(len(K)):
        Kr = W.bf16_bits_to_f32(K[r]).astype(np.float64)
        Vr = W.bf16_bits_to_f32(V[r]).astype(np.float64)
        S = Kr.shape[0]
        ql = qoffs[r + 1] - qoffs[r]
        for i in range(ql):
            qv = W.bf16_bits_to_f32(q[qoffs[r] + i]).astype(np.float64)
            n = S - ql + i + 1
            if n <= 0:
                continue
            for hq in range(q.shape[1]):
                s = scale * (Kr[:n, hq // G, :] @ qv[hq])
                out[qoffs[r] + i, hq] = scipy.special.softmax(s) @ Vr[:n, hq // G, :]
    return out


def test_multiquery_matches_dense_causal_bruteforce():
    rng = np.random.default_rng(71)
    BS, Hkv, G, D = 16, 2, 4, 64
    lens = [1, 5, 16, 40, 77]
    qlens = [1, 2, 4, 3, 8]
    K = [_bf16(rng.standard_normal((S, Hkv, D))) for S in lens]
    V = [_bf16(rng.standard_normal((S, Hkv, D))) for S in lens]
    qoffs = np.zeros(len(lens) + 1, np.int32)
    np.cumsum(qlens, out=qoffs[1:])
    q = _bf16(rng.standard_normal((int(qoffs[-1]), Hkv * G, D)))
    kc, vc, bt = _paged_from_dense(rng, K, V, BS)
    got = oracle.multiquery_attn(q, qoffs, kc, vc, bt, np.array(lens, np.int32), 0.1)
    ref = _dense_causal(q, qoffs, K, V, 0.1, G)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_multiquery_rows_match_dense_causal_and_the_whole_output():
    """Selected rows re-derive each row's request on their own, so they are pinned
    separately: every row of every request, in shuffled order and with repeats, against
    the dense causal brute force, and bit for bit against the whole-batch output.  The
    batch has ragged q_lens, a request with more queries than cached tokens (its first
    queries see nothing), and requests with no queries in the middle and at the end."""
    rng = np.random.default_rng(72)
    BS, Hkv, G, D = 16, 2, 4, 64
    lens = [3, 5, 16, 9, 40, 77, 12]
    qlens = [5, 2, 0, 4, 3, 8, 0]
    K = [_bf16(rng.standard_normal((S, Hkv, D))) for S in lens]
    V = [_bf16(rng.standard_normal((S, Hkv, D))) for S in lens]
    qoffs = np.zeros(len(lens) + 1, np.int32)
    np.cumsum(qlens, out=qoffs[1:])
    Hq = Hkv * G
    q = _bf16(rng.standard_normal((int(qoffs[-1]), Hq, D)))
    kc, vc, bt = _paged_from_dense(rng, K, V, BS)
    sl = np.array(lens, np.int32)
    ref = _dense_causal(q, qoffs, K, V, 0.1, G).reshape(-1, D)
    whole = oracle.multiquery_attn(q, qoffs, kc, vc, bt, sl, 0.1).reshape(-1, D)
    rows = np.concatenate([rng.permutation(ref.shape[0]),
                           rng.integers(0, ref.shape[0], size=40)]).astype(np.int64)
    got = oracle.multiquery_rows(q, qoffs, kc, vc, bt, sl, 0.1, rows)
    np.testing.assert_allclose(got, ref[rows], rtol=0, atol=1e-12)
    assert np.array_equal(got, whole[rows])
    # the rows that see no token: request 0's first two queries
    zero = np.arange(2 * Hq)
    assert np.all(ref[zero] == 0) and np.all(got[np.isin(rows, zero)] == 0)
    # every other row saw at least one token
    assert np.all(np.any(ref[2 * Hq:] != 0, axis=-1))


def test_multiquery_single_query_is_decode_and_empty_rows_are_zero():
    wl = W.make(2, small=True)
    d = W.host_data(wl)
    qoffs = np.arange(wl.N + 1, dtype=np.int32)
    got = oracle.multiquery_attn(d["q"], qoffs, d["k_cache"], d["v_cache"], wl.block_table,
                                 wl.seq_lens, wl.scale)
    ref = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                             wl.scale)
    assert np.array_equal(got, ref)
    # more queries than cached tokens: the first queries see nothing
    q = np.repeat(d["q"][:1], 5, axis=0)
    lens = np.array([3], np.int32)
    got = oracle.multiquery_attn(q, np.array([0, 5], np.int32), d["k_cache"], d["v_cache"],
                                 wl.block_table[:1], lens, wl.scale)
    assert np.all(got[:2] == 0) and np.all(np.any(got[2:] != 0, axis=-1))


# ---------------------------------------------------------------- int8 pages
def test_int8_encode_matches_torch_round_half_even_and_clamp():
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 60,
                         np.float32([k + 0.5 for k in range(-130, 130)]),   # exact ties
                         np.float32([126.5, 127.5, -127.5, -128.0, 1e9, -1e9, 0.0, -0.0])])
    ref = torch.clamp(torch.round(torch.from_numpy(xs)), -127, 127).to(torch.int8).numpy()
    got = np.array([oracle.int8_from_float(float(x)) for x in xs], np.int8)
    assert np.array_equal(got, ref)
    assert oracle.int8_from_float(float("nan")) == 0


def test_int8_write_and_decode_use_code_times_scale():
    wl = W.make(7, small=True)
    d = W.host_data(wl)
    req, pos = W.token_rows_order(wl)
    slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    kc = np.zeros((wl.NB, wl.Hkv, wl.BS, wl.D), np.int8)
    vc = np.zeros_like(kc)
    oracle.kv_cache_write(d["k_rows"], d["v_rows"], slots, kc, vc, d["k_scale"], d["v_scale"])
    x = W.bf16_bits_to_f32(d["k_rows"]).astype(np.float64)
    b, o = slots // wl.BS, slots % wl.BS
    codes = kc[b, :, o].astype(np.float64)
    s = d["k_scale"][b].astype(np.float64)[:, :, None]
    # half a step, plus the one binary32 rounding of the quotient x / s
    assert np.all(np.abs(codes * s - x) <= 0.5 * s * (1 + 1e-6) + np.abs(x) * 2.0 ** -23)
    assert np.abs(codes).max() == 127                                 # amax/127 scaling
    rows = np.array([0, 3 * wl.Hq + 10], np.int64)
    got = oracle.decode_rows(d["q"], kc, vc, wl.block_table, wl.seq_lens, wl.scale, rows,
                             d["k_scale"], d["v_scale"])
    for i, row in enumerate(rows):
        r, hq = divmod(int(row), wl.Hq)
        h = hq // wl.G
        blocks = wl.blocks_of(r)
        S = int(wl.seq_lens[r])
        Kd = np.concatenate([kc[bb, h].astype(np.float64) * float(d["k_scale"][bb, h]) for bb in blocks])[:S]
        Vd = np.concatenate([vc[bb, h].astype(np.float64) * float(d["v_scale"][bb, h]) for bb in blocks])[:S]
        qv = W.bf16_bits_to_f32(d["q"][r, hq]).astype(np.float64)
        p = scipy.special.softmax(wl.scale * (Kd @ qv))
        np.testing.assert_allclose(got[i], p @ Vd, atol=1e-12)


# ---------------------------------------------------------------- int4 pages
def test_int4_code_is_nearest_integer_clamped_offset_binary():
    """Code = q + 8 with q the nearest integer to x (ties to even), clamped to [-7, 7]:
    checked against a brute-force search over the 15 candidate values."""
    rng = np.random.default_rng(9)
    xs = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 4,
                         np.float32([k + 0.5 for k in range(-9, 9)]),       # exact ties
                         np.float32([6.5, 7.5, -7.5, -8.0, 1e9, -1e9, 0.0, -0.0, 0.49999997])])
    for x in xs:
        cands = np.arange(-7, 8, dtype=np.float64)
        dist = np.abs(cands - float(x))
        best = cands[dist == dist.min()]
        q = best[0] if len(best) == 1 else [c for c in best if int(c) % 2 == 0][0]
        assert oracle.int4_code_from_float(float(x)) == int(q) + 8, x
    assert oracle.int4_code_from_float(float("nan")) == 8


def test_int4_write_packs_two_codes_per_byte_low_nibble_first():
    """A row of D values becomes D/2 bytes, value 2b in the low nibble of byte b; the
    attention reads value = (code - 8) * scale and equals a dense brute force."""
    D, BS, NB = 128, 16, 4
    vals = np.float32(np.tile(np.arange(-7, 9), D // 16))                 # -7 .. 8 repeated
    bits = W.f32_to_bf16_bits(vals).reshape(1, 1, D)
    kc = np.zeros((NB, 1, BS, D // 2), np.uint8)
    vc = np.zeros_like(kc)
    sc = np.ones((NB, 1), np.float32)
    oracle.kv_cache_write(bits, bits, np.array([BS + 3], np.int64), kc, vc, sc, sc)
    row = kc[1, 0, 3]
    q = np.clip(np.rint(vals), -7, 7).astype(np.int64) + 8
    assert np.array_equal(row & 0xF, q[0::2]) and np.array_equal(row >> 4, q[1::2])
    assert np.all(kc[0] == 0) and np.all(kc[1, 0, :3] == 0)          # nothing else written
    wl = W.make(9, small=True)
    d = W.host_data(wl)
    req, pos = W.token_rows_order(wl)
    slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    kc = np.zeros(wl.cache_shape, np.uint8)
    vc = np.zeros_like(kc)
    oracle.kv_cache_write(d["k_rows"], d["v_rows"], slots, kc, vc, d["k_scale"], d["v_scale"])
    x = W.bf16_bits_to_f32(d["k_rows"]).astype(np.float64)
    b, o = slots // wl.BS, slots % wl.BS
    packed = kc[b, :, o]
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(x.shape).astype(np.float64) - 8
    s = d["k_scale"][b].astype(np.float64)[:, :, None]
    assert np.all(np.abs(codes * s - x) <= 0.5 * s * (1 + 1e-6) + np.abs(x) * 2.0 ** -23)
    assert np.abs(codes).max() == 7                                   # amax/7 scaling
    rows = np.array([0, 2 * wl.Hq + 17], np.int64)
    got = oracle.decode_rows(d["q"], kc, vc, wl.block_table, wl.seq_lens, wl.scale, rows,
                             d["k_scale"], d["v_scale"])

    def deq(cache, scale, bb, h):
        p_ = cache[bb, h]
        c_ = np.stack([p_ & 0xF, p_ >> 4], axis=-1).reshape(wl.BS, wl.D).astype(np.float64) - 8
        return c_ * float(scale[bb, h])
    for i, row_ in enumerate(rows):
        r, hq = divmod(int(row_), wl.Hq)
        h = hq // wl.G
        blocks = wl.blocks_of(r)
        S = int(wl.seq_lens[r])
        Kd = np.concatenate([deq(kc, d["k_scale"], bb, h) for bb in blocks])[:S]
        Vd = np.concatenate([deq(vc, d["v_scale"], bb, h) for bb in blocks])[:S]
        qv = W.bf16_bits_to_f32(d["q"][r, hq]).astype(np.float64)
        p = scipy.special.softmax(wl.scale * (Kd @ qv))
        np.testing.assert_allclose(got[i], p @ Vd, atol=1e-12)


@pytest.mark.parametrize("cfg", [5, 7, 9])
def test_rescale_write_scales_equal_the_amax_recipe(cfg):
    """Writing every token of a workload in one rescaling call gives each used block the
    scale amax/QMAX of its rows: the same numbers as the generator's independent numpy
    recipe; blocks nobody writes keep their scale."""
    wl = W.make(cfg, small=True)
    d = W.host_data(wl)
    req, pos = W.token_rows_order(wl)
    slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
    kc = np.zeros(wl.cache_shape, wl.cache_np_dtype)
    vc = np.zeros_like(kc)
    ks = np.full((wl.NB, wl.Hkv), 123.0, np.float32)
    vs = np.full((wl.NB, wl.Hkv), 123.0, np.float32)
    oracle.kv_cache_write_rescale(d["k_rows"], d["v_rows"], slots, kc, vc, ks, vs)
    used = np.zeros(wl.NB, bool)
    used[np.unique(slots // wl.BS)] = True
    assert np.array_equal(ks[used], d["k_scale"][used])
    assert np.array_equal(vs[used], d["v_scale"][used])
    assert np.all(ks[~used] == 123.0) and np.all(vs[~used] == 123.0)
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    oracle.kv_cache_write(d["k_rows"], d["v_rows"], slots, kc2, vc2, d["k_scale"], d["v_scale"])
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


def test_thread_count_changes_no_result():
    """The single-core timing of the oracle computes the same bits as the all-core one."""
    wl = W.make(2, small=True)
    d = W.host_data(wl)
    n0 = oracle.num_threads()
    try:
        a = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                               wl.scale)
        oracle.set_num_threads(1)
        assert oracle.num_threads() == 1
        b = oracle.decode_attn(d["q"], d["k_cache"], d["v_cache"], wl.block_table, wl.seq_lens,
                               wl.scale)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(a, b)

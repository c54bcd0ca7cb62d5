"""GPU parity of the block copy (pkv_copy_blocks) and of a block-sharing step driven by
the native block manager: prefix reuse by chained hash, beam forks, copy-on-write
of the shared partial block, the new token's write and decode over the resulting
tables -- every cache byte bit-exact and the attention within tolerance of the oracle.

"深入LLM推理：从KV Cache到PD分离的Serving全景解析", PagedAttention与Cache管理 (sharing,
copy-on-write for beam search); "ai-infra-7", 优化一：Prefix Cache (hash-keyed reuse).
"""
import numpy as np
import pytest

import oracle
import oracle.block_manager as obm
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import bf16_dev, compare, dev_bits, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu

KINDS = {"bf16": (np.uint16, None), "fp8": (np.uint8, "uint8"), "int8": (np.int8, "int8")}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _tdtype(kind):
    torch = torch_mod()
    return {"bf16": torch.bfloat16, "fp8": torch.uint8, "int8": torch.int8}[kind]


def _random_pool(rng, kind, NB, Hkv, BS, D):
    if kind == "bf16":
        return W._randn_bf16(rng, (NB, Hkv, BS, D))
    if kind == "fp8":
        return rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    return rng.integers(-127, 128, size=(NB, Hkv, BS, D), dtype=np.int8)


def _dev_pool(a, kind):
    if kind == "bf16":
        return bf16_dev(a)
    return to_dev(a)


def _mapping(rng, NB, n_pairs):
    """Distinct destinations, none of them a source; plus skipped pairs."""
    ids = rng.permutation(NB)
    src = ids[:n_pairs]
    dst = ids[n_pairs:2 * n_pairs]
    src = rng.choice(src, size=n_pairs)          # a source may be copied several times
    pairs = np.stack([src, dst], axis=1).astype(np.int32)
    extra = np.array([[3, 3], [-1, 5], [NB, 7], [2, NB + 4]], dtype=np.int32)
    return np.concatenate([pairs, extra])


@pytest.mark.parametrize("kind", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("shape", [(64, 8, 16, 128), (33, 2, 32, 64), (17, 1, 16, 8)])
def test_copy_blocks_bit_exact(kind, shape):
    torch = torch_mod()
    NB, Hkv, BS, D = shape
    if kind != "bf16" and D == 8:
        D = 16                                       # 8-bit blocks stay 16-byte multiples
    rng = np.random.default_rng(NB * 7 + D)
    kc = _random_pool(rng, kind, NB, Hkv, BS, D)
    vc = _random_pool(rng, kind, NB, Hkv, BS, D)
    ks = rng.random((NB, Hkv)).astype(np.float32)
    vs = rng.random((NB, Hkv)).astype(np.float32)
    mp = _mapping(rng, NB, NB // 3)
    kd, vd = _dev_pool(kc, kind), _dev_pool(vc, kind)
    ksd, vsd = to_dev(ks), to_dev(vs)
    q8 = kind != "bf16"
    pkv.copy_blocks(kd, vd, to_dev(mp), ksd if q8 else None, vsd if q8 else None)
    obm.copy_blocks(kc, vc, mp, ks if q8 else None, vs if q8 else None)
    torch.cuda.synchronize()
    assert np.array_equal(dev_bits(kd), kc)
    assert np.array_equal(dev_bits(vd), vc)
    if q8:
        assert np.array_equal(ksd.cpu().numpy(), ks) and np.array_equal(vsd.cpu().numpy(), vs)


def test_copy_blocks_empty_and_rejects():
    torch = torch_mod()
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pkv.copy_blocks(kc, vc, torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    L = pkv.lib()
    mp = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    assert L.pkv_copy_blocks(kc.data_ptr(), vc.data_ptr(), None, None, mp.data_ptr(), 1, 2, 64,
                             16, 4, 5, None) == -2          # dtype
    assert L.pkv_copy_blocks(kc.data_ptr(), vc.data_ptr(), None, None, mp.data_ptr(), 1, 1, 4,
                             1, 4, 0, None) == -2           # 8-byte blocks: no 16-byte multiple
    assert L.pkv_copy_blocks(kc.data_ptr() + 2, vc.data_ptr(), None, None, mp.data_ptr(), 1,
                             2, 64, 16, 4, 0, None) == -1   # alignment
    assert L.pkv_copy_blocks(kc.data_ptr(), vc.data_ptr(), None, None, mp.data_ptr(), 1, 2, 64,
                             16, 4, 1, None) == -1          # 8-bit without scales


def test_copy_blocks_full_pool_properties():
    """A 70B-layer-sized pool (8 KV heads x 16 tokens x 128 bf16 = 32 KB per block and
    cache, 1.3 GB for both caches): destinations equal their sources' original bytes,
    every other block is untouched."""
    torch = torch_mod()
    NB, Hkv, BS, D = 20480, 8, 16, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    kc = torch.randn((NB, Hkv, BS, D), generator=g, device="cuda", dtype=torch.bfloat16)
    vc = torch.randn((NB, Hkv, BS, D), generator=g, device="cuda", dtype=torch.bfloat16)
    rng = np.random.default_rng(78)
    mp = _mapping(rng, NB, 4096)
    k0, v0 = kc.clone(), vc.clone()
    pkv.copy_blocks(kc, vc, to_dev(mp))
    torch.cuda.synchronize()
    good = mp[:4096]
    src = torch.from_numpy(good[:, 0].astype(np.int64)).cuda()
    dst = torch.from_numpy(good[:, 1].astype(np.int64)).cuda()
    assert torch.equal(kc[dst], k0[src]) and torch.equal(vc[dst], v0[src])
    keep = torch.ones(NB, dtype=torch.bool, device="cuda")
    keep[dst] = False
    assert torch.equal(kc[keep], k0[keep]) and torch.equal(vc[keep], v0[keep])
    del k0, v0


# ----------------------------------------------------------------------------------
# block sharing driven by the native manager, both sides step by step
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("kind", ["bf16", "fp8", "int8"])
def test_prefix_reuse_fork_copy_on_write_decode(kind):
    torch = torch_mod()
    c = W.beam_case()
    BS, Hq, Hkv, D, NB = c["BS"], c["Hq"], c["Hkv"], c["D"], c["NB"]
    np_dt = KINDS[kind][0]
    q8 = kind != "bf16"
    # pools: zeros on both sides; 8-bit scales start at one fixed value on both sides
    kc_o = np.zeros((NB, Hkv, BS, D), np_dt)
    vc_o = np.zeros_like(kc_o)
    kd = torch.zeros((NB, Hkv, BS, D), dtype=_tdtype(kind), device="cuda")
    vd = torch.zeros_like(kd)
    ks_o = np.full((NB, Hkv), 0.05, np.float32) if q8 else None
    vs_o = ks_o.copy() if q8 else None
    ksd = to_dev(ks_o) if q8 else None
    vsd = to_dev(vs_o) if q8 else None

    # 1. chained block hashes of every prompt: library on the GPU == oracle
    prompts = c["prompts"]
    offs = np.zeros(len(prompts) + 1, np.int64)
    np.cumsum([len(p) for p in prompts], out=offs[1:])
    toks = np.concatenate(prompts).astype(np.int32)
    h_o, ho = oracle.prefix_block_hash(toks, offs, BS, seed=0x1234)
    h_d = pkv.prefix_block_hash(to_dev(toks), to_dev(offs), BS, to_dev(ho), int(ho[-1]),
                                seed=0x1234)
    h_g = h_d.cpu().numpy().view(np.uint64)
    assert np.array_equal(h_g, h_o)

    bm = pkv.BlockManager(NB, BS)
    model = obm.BlockManagerModel(NB, BS)
    lens = {}

    def write_rows(seq_ids, positions, k_rows, v_rows, rescale):
        tables = [model.block_table(s) for s in seq_ids]
        MB = max(len(t) for t in tables)
        bt = np.zeros((len(seq_ids), MB), np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        req = np.repeat(np.arange(len(seq_ids), dtype=np.int32),
                        [len(p) for p in positions])
        pos = np.concatenate(positions).astype(np.int32)
        slots_o = oracle.slot_mapping(bt, req, pos, BS)
        slots_d = pkv.compute_slot_mapping(to_dev(bt), to_dev(pos), BS, req_idx=to_dev(req))
        assert np.array_equal(slots_d.cpu().numpy(), slots_o)
        kr, vr = np.concatenate(k_rows), np.concatenate(v_rows)
        if rescale:
            oracle.kv_cache_write_rescale(kr, vr, slots_o, kc_o, vc_o, ks_o, vs_o)
            pkv.kv_cache_write_rescale(bf16_dev(kr), bf16_dev(vr), slots_d, kd, vd, ksd, vsd)
        else:
            oracle.kv_cache_write(kr, vr, slots_o, kc_o, vc_o, ks_o, vs_o)
            pkv.kv_cache_write(bf16_dev(kr), bf16_dev(vr), slots_d, kd, vd, ksd, vsd)

    # 2. prefill: each request takes its cached prefix blocks and writes only the rest
    hits_seen = []
    for r, p in enumerate(prompts):
        hs = [int(x) for x in h_o[ho[r]:ho[r + 1]]]
        got = bm.add_sequence(r, len(p), hs)
        assert got == model.add_sequence(r, len(p), hs)
        hits = got[1]
        hits_seen.append(hits)
        lens[r] = len(p)
        lo = hits * BS
        if lo < len(p):
            write_rows([r], [np.arange(lo, len(p))], [c["k_rows"][r][lo:]],
                       [c["v_rows"][r][lo:]], rescale=q8)
    fams = 2
    assert hits_seen[:fams] == [0] * fams and all(h == 4 for h in hits_seen[fams:])

    # 3. beams fork; every live sequence appends one token (copy-on-write first)
    for parent, child in c["forks"]:
        bm.fork(parent, child)
        model.fork(parent, child)
        lens[child] = lens[parent]
    pairs, positions = [], []
    for s in c["live"]:
        p = lens[s]
        assert bm.grow(s, p + 1) == model.grow(s, p + 1)
        got = bm.prepare_write(s, p // BS)
        assert got == model.prepare_write(s, p // BS)
        if got[0] >= 0:
            pairs.append(got)
        positions.append(np.array([p]))
        lens[s] = p + 1
    # request 0 and its two beams share one partial block: two copies, one in place
    assert len(pairs) == 4
    mp = np.array(pairs, np.int32)
    obm.copy_blocks(kc_o, vc_o, mp, ks_o, vs_o)
    pkv.copy_blocks(kd, vd, to_dev(mp), ksd, vsd)
    live = c["live"]
    write_rows(live, positions, [c["k_new"][i:i + 1] for i in range(len(live))],
               [c["v_new"][i:i + 1] for i in range(len(live))], rescale=False)
    torch.cuda.synchronize()
    assert np.array_equal(dev_bits(kd), kc_o) and np.array_equal(dev_bits(vd), vc_o)
    if q8:
        assert np.array_equal(ksd.cpu().numpy(), ks_o) and np.array_equal(vsd.cpu().numpy(), vs_o)

    # beams see the parent's tokens and their own new token only
    t0, t100 = model.block_table(0), model.block_table(100)
    j, off = (lens[0] - 1) // BS, (lens[0] - 1) % BS
    assert t0[:j] == t100[:j] and t0[j] != t100[j]
    assert np.array_equal(kc_o[t0[j], :, :off], kc_o[t100[j], :, :off])
    assert not np.array_equal(kc_o[t0[j], :, off], kc_o[t100[j], :, off])

    # 4. decode over the manager's tables
    tables = [model.block_table(s) for s in live]
    MB = max(len(t) for t in tables)
    bt = np.zeros((len(live), MB), np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    seq = np.array([lens[s] for s in live], np.int32)
    ref = oracle.decode_attn(c["q"], kc_o, vc_o, bt, seq, c["scale"], ks_o, vs_o)
    out = pkv.paged_decode_attn(bf16_dev(c["q"]), kd, vd, to_dev(bt), to_dev(seq), c["scale"],
                                k_scale=ksd, v_scale=vsd)
    torch.cuda.synchronize()
    compare(out_to_f64(out), ref, q8)

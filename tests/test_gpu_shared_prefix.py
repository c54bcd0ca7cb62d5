"""Decode over a shared prefix (pkv_paged_decode_attn_shared_prefix) against the fp64
oracle's plain decode over the full sequences.

The batch's requests all begin with the same tokens held in the same blocks; the call
attends the shared pages once for the whole batch (tensor-core pass over the stacked
queries), each request's private tail with the decode kernel, and merges the two with
log-sum-exp weights.  Its result must equal attention over prefix + tail."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import bf16_dev, compare, dev_bits, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _bits(rng, shape):
    return W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _case(N, Hq, Hkv, D, BS, prefix, tails, seed):
    """Block tables whose first prefix/BS entries are the same shared blocks, private
    tail blocks after them (ids from a permutation of a pool 10% larger than needed),
    and random bf16 caches (garbage in every row no request uses)."""
    rng = np.random.default_rng(seed)
    tails = np.asarray(tails, np.int64)
    npre = prefix // BS
    ntail = [-(-int(t) // BS) for t in tails]
    NB = int(np.ceil(1.1 * (npre + sum(ntail)))) + 2
    ids = rng.permutation(NB).astype(np.int32)
    MB = max(1, npre + max(ntail))
    bt = np.zeros((N, MB), np.int32)
    o = npre
    for r in range(N):
        bt[r, :npre] = ids[:npre]
        bt[r, npre:npre + ntail[r]] = ids[o:o + ntail[r]]
        o += ntail[r]
    seq = (prefix + tails).astype(np.int32)
    kc = _bits(rng, (NB, Hkv, BS, D))
    vc = _bits(rng, (NB, Hkv, BS, D))
    q = _bits(rng, (N, Hq, D))
    return q, kc, vc, bt, seq, 1.0 / np.sqrt(D)


def _run(q, kc, vc, bt, seq, scale, prefix):
    torch = torch_mod()
    N, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    ws = torch.full((pkv.shared_prefix_workspace_size(N, Hq, Hkv, D, BS, prefix),), 0x5A,
                    dtype=torch.uint8, device="cuda")   # garbage: nothing needs clearing
    ws[:4] = 0
    out = pkv.paged_decode_attn_shared_prefix(bf16_dev(q), bf16_dev(kc), bf16_dev(vc),
                                              to_dev(bt), to_dev(seq), scale, prefix,
                                              workspace=ws)
    torch.cuda.synchronize()
    assert pkv.read_device_error(ws) == 0
    return out


# ovl: the plan the call takes on a 152-SM device (checked first, so that both plans are
# known to be covered): True = the prefix pass on its own stream beside a tail decode sized
# to the remaining SMs (few prefix CTAs, long tails), False = prefix pass, then tails.
@pytest.mark.parametrize("N,Hq,Hkv,D,BS,prefix,tails,seed,ovl", [
    (12, 32, 8, 128, 16, 512, "u16-200", 1, False),   # the prefix-sharing shape, small
    (5, 64, 8, 128, 32, 160, [0, 1, 300, 31, 32], 2, True),   # G = 8, prefix not 256k
    (33, 8, 8, 64, 16, 1024, "u0-100", 3, False),     # G = 1: 33 rows over 128-row tiles
    (1, 16, 4, 128, 16, 4096, [37], 4, False),        # one request, a long shared prefix
    (130, 32, 8, 128, 16, 768, "u0-64", 5, False),    # two query tiles per KV head
    (7, 32, 8, 128, 32, 320, [0] * 7, 6, False),      # every tail empty: prefix partials only
    (40, 32, 8, 128, 16, 256, "u600-1200", 8, True),  # 2 tiles x 8 heads, long tails
    (64, 16, 8, 128, 32, 512, "u900-1500", 9, True),
])
def test_shared_prefix_matches_full_attention(N, Hq, Hkv, D, BS, prefix, tails, seed, ovl):
    if isinstance(tails, str):
        lo, hi = (int(x) for x in tails[1:].split("-"))
        tails = np.random.default_rng(seed + 100).integers(lo, hi + 1, size=N)
    q, kc, vc, bt, seq, scale = _case(N, Hq, Hkv, D, BS, prefix, tails, seed)
    sms = torch_mod().cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert pkv.shared_prefix_plan(N, Hq, Hkv, D, BS, bt.shape[1], prefix)[0] == ovl
    got = out_to_f64(_run(q, kc, vc, bt, seq, scale, prefix))
    ref = oracle.decode_attn(q, kc, vc, bt, seq, scale)
    compare(got, ref, False)
    # the plain decode of the same batch agrees as well (within the same tolerance)
    plain = pkv.paged_decode_attn(bf16_dev(q), bf16_dev(kc), bf16_dev(vc), to_dev(bt),
                                  to_dev(seq), scale)
    compare(got, out_to_f64(plain), False)


def test_shared_prefix_of_zero_is_the_plain_decode_bit_for_bit():
    torch = torch_mod()
    q, kc, vc, bt, seq, scale = _case(6, 32, 8, 128, 16, 0, [5, 90, 17, 300, 1, 64], 7)
    got = _run(q, kc, vc, bt, seq, scale, 0)
    plain = pkv.paged_decode_attn(bf16_dev(q), bf16_dev(kc), bf16_dev(vc), to_dev(bt),
                                  to_dev(seq), scale)
    assert torch.equal(got.view(torch.int16), plain.view(torch.int16))


def test_shared_prefix_rejects_bad_prefixes_before_launching():
    torch_mod()
    L = pkv.lib()
    f = L.pkv_paged_decode_attn_shared_prefix
    # (fake pointers: every call below fails its host checks first)
    assert f(16, 16, 16, 16, 8, 16, 4, 32, 8, 128, 16, 64, 24, 0.1, 16, 16, 1 << 30,
             None) == -1          # prefix not a block multiple
    assert f(16, 16, 16, 16, 8, 16, 4, 32, 8, 128, 16, 64, 16 * 9, 0.1, 16, 16, 1 << 30,
             None) == -1          # prefix past the block table
    assert f(16, 16, 16, 16, 8, 16, 4, 32, 8, 96, 16, 64, 32, 0.1, 16, 16, 1 << 30,
             None) == -2          # head_dim
    assert f(16, 16, 16, 16, 8, 16, 4, 24, 8, 128, 16, 64, 32, 0.1, 16, 16, 1 << 30,
             None) == -2          # G = 3 (the prefix pass takes 1, 2, 4, 8)
    assert f(16, 16, 16, 16, 8, 16, 4, 32, 8, 128, 16, 64, 32, 0.1, 16, 16, 16,
             None) == -3          # workspace too small


def test_shared_prefix_full_size_prefix_sharing_workload_sampled():
    """The prefix-sharing workload at full size (128 requests, 4096 shared tokens,
    private tails of 256-1024): sampled rows against the oracle."""
    torch = torch_mod()
    wl = W.make(4)
    dd = W.device_data(wl, "cuda")
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    prefix = wl.notes["shared_prefix_blocks"] * wl.BS
    out = pkv.paged_decode_attn_shared_prefix(dd["q"], dd["k_cache"], dd["v_cache"], bt, sl,
                                              wl.scale, prefix)
    torch.cuda.synchronize()
    rng = np.random.default_rng(41)
    rows = np.unique(np.concatenate([[0, wl.N * wl.Hq - 1],
                                     rng.integers(0, wl.N * wl.Hq, size=22)])).astype(np.int64)
    reqs = sorted({int(r) // wl.Hq for r in rows})
    old, seen = [], {}
    cbt = np.zeros((len(reqs), wl.MB), np.int32)
    for i, r in enumerate(reqs):
        for j, b in enumerate(wl.blocks_of(r)):
            b = int(b)
            if b not in seen:
                seen[b] = len(old)
                old.append(b)
            cbt[i, j] = seen[b]
    old_t = torch.tensor(old, dtype=torch.int64, device="cuda")
    kc_s = dev_bits(dd["k_cache"].index_select(0, old_t))
    vc_s = dev_bits(dd["v_cache"].index_select(0, old_t))
    q_s = dev_bits(dd["q"][torch.tensor(reqs).cuda()])
    local = np.array([reqs.index(int(r) // wl.Hq) * wl.Hq + int(r) % wl.Hq for r in rows],
                     np.int64)
    ref = oracle.decode_rows(q_s, kc_s, vc_s, cbt, wl.seq_lens[reqs], wl.scale, local)
    got = out_to_f64(out).reshape(wl.N * wl.Hq, wl.D)[rows]
    compare(got, ref, False)

"""The decode step captured once in a CUDA graph and replayed ("GPU推理深度拆解：KV Cache视角",
算子优化要点: CUDA Graph wants static shapes and addresses).  Every entry point takes
caller-owned buffers and never synchronises, so slot mapping, cache write, decode (with its
split-unit merges) and the prefix hash record into one graph.  Each replay, fed new values in
the same buffers, must equal the eager calls bit for bit, split units (merged by the
second kernel from the workspace's partial slots) included."""
import numpy as np
import pytest

import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import bf16_dev, dev_bits, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


@pytest.mark.parametrize("cfg", [2, 3])
def test_decode_step_graph_replay_equals_eager(cfg):
    torch = torch_mod()
    wl = W.make(cfg, small=True)
    d = W.host_data(wl)
    bt = to_dev(wl.block_table)
    sl = to_dev(wl.seq_lens)
    pos = to_dev(wl.new_token_positions())
    toks = to_dev(wl.tokens)
    toffs = to_dev(wl.token_offsets)
    ho = np.zeros(wl.N + 1, np.int64)
    np.cumsum(np.diff(wl.token_offsets) // wl.hash_block, out=ho[1:])
    hoffs = to_dev(ho)
    nh = int(ho[-1])
    # static buffers the graph reads and writes
    q = bf16_dev(d["q"])
    kn, vn = bf16_dev(d["k_new"]), bf16_dev(d["v_new"])
    kc, vc = bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"])
    slots = torch.empty(wl.N, dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    hashes = torch.empty(max(nh, 1), dtype=torch.int64, device="cuda")
    ws = pkv.alloc_decode_workspace(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, pkv.BF16)
    stream = torch.cuda.Stream()

    def step(st):
        pkv.compute_slot_mapping(bt, pos, wl.BS, out=slots, stream=st)
        pkv.kv_cache_write(kn, vn, slots, kc, vc, stream=st)
        pkv.paged_decode_attn(q, kc, vc, bt, sl, wl.scale, out=out, workspace=ws, stream=st)
        pkv.prefix_block_hash(toks, toffs, wl.hash_block, hoffs, nh, seed=7, out=hashes,
                              stream=st)

    # warm up on the side stream (first calls may set kernel attributes), then capture
    with torch.cuda.stream(stream):
        step(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(stream)
    torch.cuda.synchronize()

    rng = np.random.default_rng(cfg)
    kc0, vc0 = kc.clone(), vc.clone()
    for rep in range(3):
        # new inputs in the same buffers
        q.copy_(bf16_dev(W.f32_to_bf16_bits(
            rng.standard_normal(d["q"].shape).astype(np.float32))))
        kn.copy_(bf16_dev(W.f32_to_bf16_bits(
            rng.standard_normal(d["k_new"].shape).astype(np.float32))))
        kc.copy_(kc0)
        vc.copy_(vc0)
        graph.replay()
        torch.cuda.synchronize()
        got_out, got_k, got_h = dev_bits(out), dev_bits(kc), hashes[:nh].cpu().numpy()
        # eager reference on fresh copies of the same inputs
        kc.copy_(kc0)
        vc.copy_(vc0)
        out_e = torch.empty_like(q)
        ws_e = pkv.alloc_decode_workspace(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, pkv.BF16)
        sl_e = pkv.compute_slot_mapping(bt, pos, wl.BS)
        pkv.kv_cache_write(kn, vn, sl_e, kc, vc)
        pkv.paged_decode_attn(q, kc, vc, bt, sl, wl.scale, out=out_e, workspace=ws_e)
        h_e = pkv.prefix_block_hash(toks, toffs, wl.hash_block, hoffs, nh, seed=7)
        torch.cuda.synchronize()
        assert np.array_equal(got_out, dev_bits(out_e)), f"replay {rep}: output differs"
        assert np.array_equal(got_k, dev_bits(kc)), f"replay {rep}: cache differs"
        assert np.array_equal(got_h, h_e.cpu().numpy()), f"replay {rep}: hashes differ"
        assert pkv.read_device_error(ws) == 0


def test_shared_prefix_step_with_resumed_hash_graph_replay_equals_eager():
    """The serving-style step of the prefix-sharing workload (small): slot mapping, write,
    shared-prefix decode (prefix pass, tail decode, merge) and the resumed hash chains,
    captured once and replayed with new queries and new K rows; bit for bit the eager
    calls."""
    torch = torch_mod()
    wl = W.make(4, small=True)
    d = W.host_data(wl)
    prefix = wl.notes["shared_prefix_blocks"] * wl.BS
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    pos = to_dev(wl.new_token_positions())
    toks, toffs = to_dev(wl.tokens), to_dev(wl.token_offsets)
    lens = np.diff(wl.token_offsets)
    first = ((lens - 1) // wl.hash_block).astype(np.int64)   # blocks full before the step
    ho = np.zeros(wl.N + 1, np.int64)
    np.cumsum(lens // wl.hash_block - first, out=ho[1:])
    nh = int(ho[-1])
    fho = np.zeros(wl.N + 1, np.int64)
    np.cumsum(lens // wl.hash_block, out=fho[1:])
    chain = pkv.prefix_block_hash(toks, toffs, wl.hash_block, to_dev(fho), int(fho[-1]), seed=3)
    chain = chain.cpu().numpy().view(np.uint64)
    prev = np.array([chain[fho[s] + first[s] - 1] if first[s] > 0 else 3 for s in range(wl.N)],
                    np.uint64)
    prev_t, first_t, hoffs = to_dev(prev.view(np.int64)), to_dev(first), to_dev(ho)
    q = bf16_dev(d["q"])
    kn, vn = bf16_dev(d["k_new"]), bf16_dev(d["v_new"])
    kc, vc = bf16_dev(d["k_cache"]), bf16_dev(d["v_cache"])
    slots = torch.empty(wl.N, dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    hashes = torch.empty(max(nh, 1), dtype=torch.int64, device="cuda")
    nws = pkv.shared_prefix_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, prefix)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def step(st, o, w, h):
        pkv.compute_slot_mapping(bt, pos, wl.BS, out=slots, stream=st)
        pkv.kv_cache_write(kn, vn, slots, kc, vc, stream=st)
        pkv.paged_decode_attn_shared_prefix(q, kc, vc, bt, sl, wl.scale, prefix, out=o,
                                            workspace=w, stream=st)
        pkv.prefix_block_hash_resume(toks, toffs, wl.hash_block, prev_t, first_t, hoffs, nh,
                                     out=h, stream=st)

    with torch.cuda.stream(stream):
        step(stream, out, ws, hashes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(stream, out, ws, hashes)
    torch.cuda.synchronize()

    rng = np.random.default_rng(9)
    kc0, vc0 = kc.clone(), vc.clone()
    for rep in range(3):
        q.copy_(bf16_dev(W.f32_to_bf16_bits(
            rng.standard_normal(d["q"].shape).astype(np.float32))))
        kn.copy_(bf16_dev(W.f32_to_bf16_bits(
            rng.standard_normal(d["k_new"].shape).astype(np.float32))))
        kc.copy_(kc0)
        vc.copy_(vc0)
        graph.replay()
        torch.cuda.synchronize()
        got_out, got_h = dev_bits(out), hashes[:nh].cpu().numpy()
        kc.copy_(kc0)
        vc.copy_(vc0)
        out_e = torch.empty_like(q)
        ws_e = torch.zeros(nws, dtype=torch.uint8, device="cuda")
        h_e = torch.empty(max(nh, 1), dtype=torch.int64, device="cuda")
        step(torch.cuda.current_stream(), out_e, ws_e, h_e)
        torch.cuda.synchronize()
        assert np.array_equal(got_out, dev_bits(out_e)), f"replay {rep}: output differs"
        assert np.array_equal(got_h, h_e[:nh].cpu().numpy()), f"replay {rep}: hashes differ"
        assert pkv.read_device_error(ws) == 0


def test_overlapped_shared_prefix_call_graph_replay_equals_eager():
    """A batch whose shared-prefix call takes the overlapped plan (the prefix pass on the
    library's second stream beside the tail decode, joined before the merge), captured
    once: the fork and join become graph edges, and every replay with new queries equals
    the eager call bit for bit."""
    torch = torch_mod()
    rng = np.random.default_rng(31)
    N, Hq, Hkv, D, BS, prefix = 40, 32, 8, 128, 16, 256
    tails = rng.integers(600, 1201, size=N)
    npre = prefix // BS
    ntail = [-(-int(t) // BS) for t in tails]
    NB = npre + sum(ntail) + 4
    ids = rng.permutation(NB).astype(np.int32)
    MB = npre + max(ntail)
    bt = np.zeros((N, MB), np.int32)
    o = npre
    for r in range(N):
        bt[r, :npre] = ids[:npre]
        bt[r, npre:npre + ntail[r]] = ids[o:o + ntail[r]]
        o += ntail[r]
    seq = (prefix + tails).astype(np.int32)
    kc = bf16_dev(W.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, BS, D), dtype=np.float32)))
    vc = bf16_dev(W.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, BS, D), dtype=np.float32)))
    q = bf16_dev(W.f32_to_bf16_bits(rng.standard_normal((N, Hq, D), dtype=np.float32)))
    btd, sld = to_dev(bt), to_dev(seq)
    nws = pkv.shared_prefix_workspace_size(N, Hq, Hkv, D, BS, prefix)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    stream = torch.cuda.Stream()
    scale = 1.0 / np.sqrt(D)

    def call(st, o_, w_):
        pkv.paged_decode_attn_shared_prefix(q, kc, vc, btd, sld, scale, prefix, out=o_,
                                            workspace=w_, stream=st)

    with torch.cuda.stream(stream):
        call(stream, out, ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call(stream, out, ws)
    torch.cuda.synchronize()
    for rep in range(3):
        q.copy_(bf16_dev(W.f32_to_bf16_bits(
            rng.standard_normal((N, Hq, D)).astype(np.float32))))
        graph.replay()
        torch.cuda.synchronize()
        got = dev_bits(out)
        out_e = torch.empty_like(q)
        ws_e = torch.zeros(nws, dtype=torch.uint8, device="cuda")
        call(torch.cuda.current_stream(), out_e, ws_e)
        torch.cuda.synchronize()
        assert np.array_equal(got, dev_bits(out_e)), f"replay {rep}: output differs"
        assert pkv.read_device_error(ws) == 0

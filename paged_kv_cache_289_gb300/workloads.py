"""Seeded synthetic workloads for the paged-KV decode path.

This module is the ONLY thing shared between the CUDA path and the CPU oracle.
It holds the input recipe -- shapes, value distributions, block-table
permutations, token ids -- and none of the method's arithmetic: no slot
computation, no quantisation, no attention, no hashing.

The five workloads follow the shapes the sources discuss:
  1 tiny        -- 4 requests, GQA group 4, head_dim 64, 16-token blocks
  2 70B-shaped  -- a Llama-3.3-70B-like GQA layer (64 q heads / 8 kv heads, d=128),
                   the 320 KB/token model of "ai-infra-7" ("KV Cache 到底有多大？")
  3 long ctx    -- 32K..128K-token requests at batch 4 (32-token blocks)
  4 prefix      -- 128 requests sharing the pages of one 4096-token system prompt
                   ("ai-infra-7", "优化一：Prefix Cache")
  5 fp8         -- 256 requests, log-uniform lengths, E4M3 pages with one fp32 scale
                   per (block, kv head) = amax/448 of the source values
                   ("ai-infra-7", "优化三：KV 传输优化", 传输量化)

Every random draw comes from ``numpy.random.default_rng(seed)`` (metadata and
host tensors) or from a seeded ``torch.Generator`` on the device (large
tensors at full size).  bf16 values are N(0,1) float32 draws rounded to the
nearest bf16 (ties to even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

VOCAB_SMALL = 32000
VOCAB = 128000
E4M3_MAX = 448.0
INT8_MAX = 127.0
INT4_MAX = 7.0


@dataclass
class Workload:
    name: str
    cfg: int
    seed: int
    N: int
    Hq: int
    Hkv: int
    D: int
    BS: int
    NB: int
    fp8: bool
    scale: float
    seq_lens: np.ndarray          # int32 [N]
    block_table: np.ndarray       # int32 [N, MB]; entries past a request's blocks are 0
    tokens: np.ndarray            # int32 [sum seq_lens] (CSR by request)
    token_offsets: np.ndarray     # int64 [N + 1]
    hash_block: int = 16
    q_len: int = 1                # new query tokens per request (speculative verify: > 1)
    int8: bool = False            # int8 pages (symmetric, scale = amax/127)
    int4: bool = False            # int4 pages (two offset-binary codes per byte, amax/7)
    q_lens: np.ndarray | None = None   # int32 [N] per-request query counts (prefill chunks);
                                       # None: q_len for every request
    notes: dict = field(default_factory=dict)

    @property
    def query_lens(self) -> np.ndarray:
        """New query tokens of each request (int64 [N])."""
        if self.q_lens is not None:
            return np.asarray(self.q_lens, dtype=np.int64)
        return np.full(self.N, self.q_len, dtype=np.int64)

    @property
    def total_q(self) -> int:
        return int(self.query_lens.sum())

    @property
    def max_q_len(self) -> int:
        return int(self.query_lens.max()) if self.N else 0

    @property
    def quant(self) -> bool:
        """Quantised pages with one fp32 scale per (block, kv head) (E4M3, int8, int4)."""
        return self.fp8 or self.int8 or self.int4

    @property
    def kv_kind(self) -> int:
        """0: bf16 pages, 1: E4M3, 2: int8, 3: int4."""
        return 3 if self.int4 else (2 if self.int8 else (1 if self.fp8 else 0))

    @property
    def qmax(self) -> float:
        """Largest code magnitude of the 8-bit kind (the scale recipe divides amax by it)."""
        return INT4_MAX if self.int4 else (INT8_MAX if self.int8 else E4M3_MAX)

    @property
    def cache_np_dtype(self):
        return np.int8 if self.int8 else (np.uint8 if (self.fp8 or self.int4) else np.uint16)

    @property
    def cache_shape(self):
        """Shape of one cache tensor: [NB, Hkv, BS, D] elements, or [.., D / 2] bytes for
        int4 pages."""
        return (self.NB, self.Hkv, self.BS, self.D // 2 if self.int4 else self.D)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def MB(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    @property
    def elt(self) -> float:
        """Bytes per cached element: 2 (bf16), 1 (E4M3, int8), 0.5 (int4)."""
        return 0.5 if self.int4 else (1 if self.quant else 2)

    def blocks_of(self, r: int) -> np.ndarray:
        nb = -(-int(self.seq_lens[r]) // self.BS)
        return self.block_table[r, :nb]

    def new_token_positions(self) -> np.ndarray:
        """Decode step: each request's newest token sits at position seq_len - 1."""
        return (self.seq_lens.astype(np.int64) - 1).astype(np.int32)

    def q_offsets(self) -> np.ndarray:
        """Query rows of each request, request-major (int32 [N + 1])."""
        o = np.zeros(self.N + 1, dtype=np.int64)
        np.cumsum(self.query_lens, out=o[1:])
        return o.astype(np.int32)

    def new_token_rows(self):
        """(req_idx, positions) of the step's new tokens: the last q_len tokens of
        every request (positions seq_len - q_len .. seq_len - 1)."""
        ql = self.query_lens
        req = np.repeat(np.arange(self.N, dtype=np.int32), ql)
        pos = np.concatenate([np.arange(int(s) - int(n), int(s)) for s, n in
                              zip(self.seq_lens, ql)]) if self.N else np.zeros(0)
        return req, pos.astype(np.int32)

    def prefill_flops(self) -> int:
        """Causal-effective flops of attention over the new queries: every (query head,
        visible key) pair costs 2 D for Q K^T and 2 D for P V."""
        tot = 0
        for s, n in zip(self.seq_lens.astype(np.int64), self.query_lens):
            ctx = int(s) - int(n)
            i = np.arange(int(n), dtype=np.int64)
            vis = np.clip(ctx + i + 1, 0, int(s))
            tot += int(vis.sum())
        return tot * self.Hq * 4 * self.D

    def kv_read_bytes(self) -> int:
        """Logical K+V bytes one decode step reads: sum_r seq_len_r * Hkv * D * 2 * elt."""
        return int(self.total_tokens * self.Hkv * self.D * 2 * self.elt)

    def unique_kv_read_bytes(self) -> int:
        """K+V bytes of distinct physical token rows read (shared prefix pages once)."""
        rows = set()
        for r in range(self.N):
            S = int(self.seq_lens[r])
            blocks = self.blocks_of(r)
            for j, b in enumerate(blocks):
                rows.add((int(b), min(self.BS, S - j * self.BS)))
        n = sum(cnt for _, cnt in rows)
        return int(n * self.Hkv * self.D * 2 * self.elt)


# ----------------------------------------------------------------------------
# metadata
# ----------------------------------------------------------------------------
def _assign_blocks(rng, seq_lens, BS, NB=None, slack=1.1):
    nblk = [-(-int(s) // BS) for s in seq_lens]
    need = int(sum(nblk))
    if NB is None:
        NB = max(1, math.ceil(slack * need))
    ids = rng.permutation(NB)[:need].astype(np.int32)
    MB = max(1, max(nblk) if nblk else 1)
    bt = np.zeros((len(seq_lens), MB), dtype=np.int32)
    o = 0
    for r, n in enumerate(nblk):
        bt[r, :n] = ids[o:o + n]
        o += n
    return bt, NB


def _tokens(rng, seq_lens, vocab):
    offs = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    np.cumsum(np.asarray(seq_lens, dtype=np.int64), out=offs[1:])
    toks = rng.integers(0, vocab, size=int(offs[-1]), dtype=np.int64).astype(np.int32)
    return toks, offs


def make(cfg: int, seed: int | None = None, small: bool = False,
         batch: int | None = None) -> Workload:
    """Workload `cfg` (1..5).  `small=True` keeps the head/dim/block shape but
    shrinks batch and lengths so the fp64 oracle finishes in seconds.  `batch`
    overrides the number of requests of workloads 2, 4, 5 and 6 (same length law).
    Workload 6 is workload 2 with four new query tokens per request (speculative
    verify)."""
    seed = cfg if seed is None else seed
    rng = np.random.default_rng(seed)
    if cfg == 1:
        seq = np.array([17, 33, 64, 100], dtype=np.int32)
        N, Hq, Hkv, D, BS = 4, 4, 1, 64, 16
        NB = 32
        perm = rng.permutation(NB).astype(np.int32)
        nblk = [-(-int(s) // BS) for s in seq]
        bt = np.zeros((N, max(nblk)), dtype=np.int32)
        o = 0
        for r, n in enumerate(nblk):
            bt[r, :n] = perm[o:o + n]
            o += n
        toks, offs = _tokens(rng, seq, VOCAB_SMALL)
        return Workload("tiny", 1, seed, N, Hq, Hkv, D, BS, NB, False, 1.0 / 8.0, seq, bt, toks,
                        offs)
    if cfg == 2:
        if small:
            N, lo, hi = 8, 64, 700
        else:
            N, lo, hi = 64, 1024, 8192
        N = batch or N
        seq = rng.integers(lo, hi + 1, size=N).astype(np.int32)
        Hq, Hkv, D, BS = 64, 8, 128, 16
        bt, NB = _assign_blocks(rng, seq, BS)
        toks, offs = _tokens(rng, seq, VOCAB)
        return Workload("llama70b_decode" + ("_small" if small else ""), 2, seed, N, Hq, Hkv, D,
                        BS, NB, False, 1.0 / math.sqrt(D), seq, bt, toks, offs)
    if cfg == 3:
        if small:
            seq = np.array([1000, 3000, 5000, 6143], dtype=np.int32)
        else:
            seq = np.array([32768, 65536, 98304, 131072], dtype=np.int32)
        N, Hq, Hkv, D, BS = 4, 64, 8, 128, 32
        bt, NB = _assign_blocks(rng, seq, BS)
        toks, offs = _tokens(rng, seq, VOCAB)
        return Workload("long_context" + ("_small" if small else ""), 3, seed, N, Hq, Hkv, D,
                        BS, NB, False, 1.0 / math.sqrt(D), seq, bt, toks, offs)
    if cfg == 4:
        if small:
            N, prefix, tlo, thi = 12, 512, 16, 200
        else:
            N, prefix, tlo, thi = 128, 4096, 256, 1024
        N = batch or N
        Hq, Hkv, D, BS = 32, 8, 128, 16
        tails = rng.integers(tlo, thi + 1, size=N).astype(np.int32)
        seq = (prefix + tails).astype(np.int32)
        npre = prefix // BS
        ntail = [-(-int(t) // BS) for t in tails]
        need = npre + sum(ntail)
        NB = math.ceil(1.1 * need)
        ids = rng.permutation(NB).astype(np.int32)
        shared = ids[:npre]
        MB = npre + max(ntail)
        bt = np.zeros((N, MB), dtype=np.int32)
        o = npre
        for r in range(N):
            bt[r, :npre] = shared
            bt[r, npre:npre + ntail[r]] = ids[o:o + ntail[r]]
            o += ntail[r]
        prefix_tokens = rng.integers(0, VOCAB, size=prefix, dtype=np.int64).astype(np.int32)
        parts = []
        for r in range(N):
            parts.append(prefix_tokens)
            parts.append(rng.integers(0, VOCAB, size=int(tails[r]), dtype=np.int64).astype(np.int32))
        toks = np.concatenate(parts)
        offs = np.zeros(N + 1, dtype=np.int64)
        np.cumsum(seq.astype(np.int64), out=offs[1:])
        wl = Workload("prefix_sharing" + ("_small" if small else ""), 4, seed, N, Hq, Hkv, D, BS,
                      NB, False, 1.0 / math.sqrt(D), seq, bt, toks, offs)
        wl.notes["shared_prefix_blocks"] = npre
        return wl
    if cfg == 5:
        if small:
            N, lo, hi = 16, 128, 2048
        else:
            N, lo, hi = 256, 128, 16384
        N = batch or N
        seq = np.exp(rng.uniform(math.log(lo), math.log(hi), size=N)).astype(np.int64)
        seq = np.clip(seq, lo, hi).astype(np.int32)
        Hq, Hkv, D, BS = 64, 8, 128, 32
        bt, NB = _assign_blocks(rng, seq, BS)
        toks, offs = _tokens(rng, seq, VOCAB)
        return Workload("fp8_at_scale" + ("_small" if small else ""), 5, seed, N, Hq, Hkv, D, BS,
                        NB, True, 1.0 / math.sqrt(D), seq, bt, toks, offs)
    if cfg == 7:
        # int8 pages at scale: workload 5's requests with symmetric int8 codes
        wl = make(5, seed=seed, small=small, batch=batch)
        wl.name = "int8_at_scale" + ("_small" if small else "")
        wl.cfg = 7
        wl.fp8 = False
        wl.int8 = True
        return wl
    if cfg == 9:
        # int4 pages at scale: workload 5's requests with symmetric int4 codes
        wl = make(5, seed=seed, small=small, batch=batch)
        wl.name = "int4_at_scale" + ("_small" if small else "")
        wl.cfg = 9
        wl.fp8 = False
        wl.int4 = True
        return wl
    if cfg == 8:
        # chunked prefill on the 70B-shaped layer: a chunk of new prompt tokens per
        # request after a cached context; small: ragged chunks spanning several tiles
        Hq, Hkv, D, BS = 64, 8, 128, 16
        if small:
            qls = np.array([130, 257, 1, 64, 300], dtype=np.int32)
            ctx = rng.integers(0, 700, size=qls.shape[0]).astype(np.int32)
            ctx[2] = 0
        else:
            N = batch or 8
            qls = np.full(N, 2048, dtype=np.int32)
            ctx = rng.integers(0, 6144 + 1, size=N).astype(np.int32)
        seq = (ctx + qls).astype(np.int32)
        bt, NB = _assign_blocks(rng, seq, BS)
        toks, offs = _tokens(rng, seq, VOCAB)
        return Workload("prefill_chunk" + ("_small" if small else ""), 8, seed, int(seq.shape[0]),
                        Hq, Hkv, D, BS, NB, False, 1.0 / math.sqrt(D), seq, bt, toks, offs,
                        q_lens=qls)
    if cfg == 6:
        # speculative verify on the 70B-shaped layer: 4 new tokens per request
        # (3 drafted + 1), all checked in one attention pass
        wl = make(2, seed=seed, small=small, batch=batch)
        wl.name = "spec_verify_q4" + ("_small" if small else "")
        wl.cfg = 6
        wl.q_len = 4
        return wl
    raise ValueError(f"unknown workload {cfg}")


def custom(N, Hq, Hkv, D, BS, seq_lens, fp8=False, seed=0, slack=1.1, scale=None, name="custom",
           q_len=1, int8=False, int4=False):
    """A workload with explicit lengths (edge cases: empty, ragged, one-token requests)."""
    rng = np.random.default_rng(seed)
    seq = np.asarray(seq_lens, dtype=np.int32)
    bt, NB = _assign_blocks(rng, seq, BS, slack=slack)
    toks, offs = _tokens(rng, seq, VOCAB)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    return Workload(name, 0, seed, N, Hq, Hkv, D, BS, NB, fp8, sc, seq, bt, toks, offs,
                    q_len=q_len, int8=int8, int4=int4)


# ----------------------------------------------------------------------------
# value generation
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def _randn_bf16(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def token_rows_order(wl: Workload):
    """(req_idx, positions) of every cached token, request-major, position-minor."""
    req = np.repeat(np.arange(wl.N, dtype=np.int32), wl.seq_lens.astype(np.int64))
    pos = np.concatenate([np.arange(int(s), dtype=np.int32) for s in wl.seq_lens]) \
        if wl.N else np.zeros(0, np.int32)
    return req, pos


def fp8_scales_from_rows(wl: Workload, k_rows_bits: np.ndarray, v_rows_bits: np.ndarray):
    """Workloads 5 and 7: one fp32 scale per (physical block, kv head) = amax/448 (E4M3) or
    amax/127 (int8) of the source values of the block's tokens (1.0 for an all-zero or
    unused block)."""
    ks = np.ones((wl.NB, wl.Hkv), dtype=np.float32)
    vs = np.ones((wl.NB, wl.Hkv), dtype=np.float32)
    kf = np.abs(bf16_bits_to_f32(k_rows_bits)).max(axis=2)  # [T, Hkv]
    vf = np.abs(bf16_bits_to_f32(v_rows_bits)).max(axis=2)
    o = 0
    for r in range(wl.N):
        S = int(wl.seq_lens[r])
        for j, b in enumerate(wl.blocks_of(r)):
            lo, hi = o + j * wl.BS, o + min(S, (j + 1) * wl.BS)
            ka = np.float32(kf[lo:hi].max(axis=0)) if hi > lo else np.zeros(wl.Hkv, np.float32)
            va = np.float32(vf[lo:hi].max(axis=0)) if hi > lo else np.zeros(wl.Hkv, np.float32)
            ks[b] = np.where(ka > 0, ka / np.float32(wl.qmax), np.float32(1.0))
            vs[b] = np.where(va > 0, va / np.float32(wl.qmax), np.float32(1.0))
        o += S
    return ks, vs


def host_data(wl: Workload, seed_offset: int = 1000) -> dict:
    """Host (numpy) tensors for a workload small enough to hold in host memory.

    bf16 workloads: `k_cache`, `v_cache` uint16 [NB, Hkv, BS, D] filled with N(0,1)
    bf16 everywhere (rows past a request's length and unused blocks included).
    fp8 workloads: `k_rows`, `v_rows` uint16 [T, Hkv, D] source values of every
    cached token (order of `token_rows_order`) plus `k_scale`, `v_scale` fp32
    [NB, Hkv]; each side quantises them into its own cache with its own write.
    Both: `q` uint16 [N, Hq, D]; `k_new`, `v_new` uint16 [N, Hkv, D] (the decode
    step's new token of each request, written at position seq_len - 1)."""
    rng = np.random.default_rng(wl.seed + seed_offset)
    d = {"q": _randn_bf16(rng, (wl.total_q, wl.Hq, wl.D))}
    if not wl.quant:
        d["k_cache"] = _randn_bf16(rng, (wl.NB, wl.Hkv, wl.BS, wl.D))
        d["v_cache"] = _randn_bf16(rng, (wl.NB, wl.Hkv, wl.BS, wl.D))
    else:
        T = wl.total_tokens
        d["k_rows"] = _randn_bf16(rng, (T, wl.Hkv, wl.D))
        d["v_rows"] = _randn_bf16(rng, (T, wl.Hkv, wl.D))
        d["k_scale"], d["v_scale"] = fp8_scales_from_rows(wl, d["k_rows"], d["v_rows"])
    d["k_new"] = _randn_bf16(rng, (wl.total_q, wl.Hkv, wl.D))
    d["v_new"] = _randn_bf16(rng, (wl.total_q, wl.Hkv, wl.D))
    return d


def device_data(wl: Workload, device, seed_offset: int = 2000) -> dict:
    """Device (torch) tensors for full-size workloads, drawn from a seeded
    torch.Generator on `device`.  Same keys and layouts as `host_data`, as
    torch tensors (bf16 bit patterns stored as torch.bfloat16).  For fp8
    workloads the scales follow the same amax/448 recipe, reduced on the device."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(wl.seed + seed_offset)
    bf = torch.bfloat16
    d = {"q": torch.randn((wl.total_q, wl.Hq, wl.D), generator=g, device=device, dtype=bf)}
    if not wl.quant:
        d["k_cache"] = torch.randn((wl.NB, wl.Hkv, wl.BS, wl.D), generator=g, device=device,
                                   dtype=bf)
        d["v_cache"] = torch.randn((wl.NB, wl.Hkv, wl.BS, wl.D), generator=g, device=device,
                                   dtype=bf)
    else:
        T = wl.total_tokens
        d["k_rows"] = torch.randn((T, wl.Hkv, wl.D), generator=g, device=device, dtype=bf)
        d["v_rows"] = torch.randn((T, wl.Hkv, wl.D), generator=g, device=device, dtype=bf)
        # segment (request, logical block) of every token row, and its physical block
        seg = np.zeros(T, dtype=np.int64)
        phys = []
        o = 0
        s_id = 0
        for r in range(wl.N):
            S = int(wl.seq_lens[r])
            blocks = wl.blocks_of(r)
            for j, b in enumerate(blocks):
                lo, hi = o + j * wl.BS, o + min(S, (j + 1) * wl.BS)
                seg[lo:hi] = s_id
                phys.append(int(b))
                s_id += 1
            o += S
        seg_t = torch.from_numpy(seg).to(device)
        phys_t = torch.tensor(phys, dtype=torch.int64, device=device)
        for key, skey in (("k_rows", "k_scale"), ("v_rows", "v_scale")):
            amax_rows = d[key].abs().amax(dim=2).float()            # [T, Hkv]
            amax = torch.zeros((s_id, wl.Hkv), dtype=torch.float32, device=device)
            amax.scatter_reduce_(0, seg_t[:, None].expand(T, wl.Hkv), amax_rows, "amax")
            sc = torch.where(amax > 0, amax / wl.qmax, torch.ones_like(amax))
            full = torch.ones((wl.NB, wl.Hkv), dtype=torch.float32, device=device)
            full[phys_t] = sc
            d[skey] = full
    d["k_new"] = torch.randn((wl.total_q, wl.Hkv, wl.D), generator=g, device=device, dtype=bf)
    d["v_new"] = torch.randn((wl.total_q, wl.Hkv, wl.D), generator=g, device=device, dtype=bf)
    return d


def beam_case(seed: int = 31, BS: int = 16, Hq: int = 32, Hkv: int = 8, D: int = 128,
              families: int = 2, prefix_blocks: int = 4, requests: int = 6, NB: int = 128,
              vocab: int = 32000) -> dict:
    """Inputs of a block-sharing scenario: `requests` prompts, request r opening with the
    system prompt of family r % families (prefix_blocks full blocks, identical tokens and
    identical K/V rows across the family) followed by a private tail; requests 0 and 1
    each fork two beams (sequence ids 100 + 2r and 101 + 2r); then every live sequence
    appends one new token.  Tails of requests 0 and 1 end inside a block, so their beams
    share a partial block.  Everything is drawn from one seeded generator; bf16 values
    are N(0, 1) bit patterns (uint16)."""
    rng = np.random.default_rng(seed)
    P = prefix_blocks * BS
    fam_tok = rng.integers(0, vocab, size=(families, P), dtype=np.int32)
    fam_k = _randn_bf16(rng, (families, P, Hkv, D))
    fam_v = _randn_bf16(rng, (families, P, Hkv, D))
    tails = rng.integers(5, 40, size=requests)
    tails[0], tails[1] = 7, BS + 3
    prompts, k_rows, v_rows = [], [], []
    for r in range(requests):
        f = r % families
        t = int(tails[r])
        prompts.append(np.concatenate([fam_tok[f], rng.integers(0, vocab, size=t,
                                                                dtype=np.int32)]))
        k_rows.append(np.concatenate([fam_k[f], _randn_bf16(rng, (t, Hkv, D))]))
        v_rows.append(np.concatenate([fam_v[f], _randn_bf16(rng, (t, Hkv, D))]))
    forks = [(0, 100), (0, 101), (1, 102), (1, 103)]
    live = list(range(requests)) + [c for _, c in forks]
    n = len(live)
    return {"BS": BS, "Hq": Hq, "Hkv": Hkv, "D": D, "NB": NB, "prompts": prompts,
            "k_rows": k_rows, "v_rows": v_rows, "forks": forks, "live": live,
            "q": _randn_bf16(rng, (n, Hq, D)), "k_new": _randn_bf16(rng, (n, Hkv, D)),
            "v_new": _randn_bf16(rng, (n, Hkv, D)), "scale": 1.0 / float(np.sqrt(D))}

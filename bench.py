#!/usr/bin/env python3
"""Benchmark of the paged-KV decode step (libpagedkv on GB300).

One step = the whole hot path over one batch: slot mapping of each request's new
token, KV cache write, paged GQA decode attention (the decode kernel, then a merge
kernel for requests split across warps), and the chained prefix block hash of every
request's tokens (on a side stream).

Workload: the Llama-3.3-70B-shaped decode layer -- batch 64, 64 query / 8 KV heads,
head_dim 128, bf16, 16-token blocks, lengths U[1024, 8192], blocks randomly permuted
in a pool 10% larger than needed.  Pages (~1.33 GB) exceed the 129 MB L2, so no flush
is needed between steps.

Prints ONE JSON line (rank 0).  With the default workload, the line also carries
`per_workload`: decode-launch rooflines of workloads 3 (long context), 5 (E4M3 pages)
and 4 (prefix sharing, logical and unique bytes, with and without an L2 flush), and
workload 3's step with the full and the resumed prefix hash.  `--impl reference` times
the fp64 CPU oracle instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attention: KV-read HBM GB/s (% of GB300 peak), query tokens/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=2, help="workload id (2 = the metric's)")
    p.add_argument("--skip-e2e", action="store_true")
    p.add_argument("--skip-cpu", action="store_true")
    p.add_argument("--skip-per-workload", action="store_true",
                   help="leave out the decode figures of workloads 3, 4 and 5 (workload 2 runs)")
    p.add_argument("--append", action="store_true",
                   help="the decode writes each request's new K/V rows itself "
                        "(pkv_paged_decode_attn_append; bf16 pages); slot mapping runs beside it")
    p.add_argument("--shared-prefix", action="store_true",
                   help="workload 4: decode through pkv_paged_decode_attn_shared_prefix (the "
                        "shared pages attended once for the batch)")
    p.add_argument("--hash", choices=["full", "resume"], default="full",
                   help="full: the step re-hashes every token; resume: only the blocks the "
                        "step completes (pkv_prefix_block_hash_resume)")
    p.add_argument("--seed", type=int, default=None)
    p.add_argument("--batch", type=int, default=None,
                   help="fewer requests of the same shapes (profiling captures only)")
    p.add_argument("--op", choices=["step", "copy_blocks", "prefill"], default="step",
                   help="copy_blocks: the copy-on-write block copy alone; prefill: paged "
                        "prefill attention on workload 8")
    p.add_argument("--pairs", type=int, default=4096, help="block pairs per copy_blocks launch")
    p.add_argument("--prefill-kv", choices=["bf16", "fp8", "int8", "int4"], default="bf16",
                   help="page kind of the cache the prefill reads (--op prefill)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel_src_hash, workload_name):
    """Per-launch DRAM traffic of the decode launch from the committed ncu summary, if it
    was taken on the current kernel source and on this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                line = line.strip()
                if line and not line.startswith("#") and "=" in line:
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_src_hash or kv.get("workload") != workload_name:
            return None
        return float(kv["bytes_per_launch"])
    except Exception:
        return None


def strip_c_comments(src):
    """C/C++/CUDA source without its comments, whitespace runs collapsed: the text
    that decides the compiled code (string and character literals kept intact)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """sha256 of the decode kernel's sources with comments stripped, so a comment edit
    keeps a recorded DRAM traffic figure valid and a code edit does not."""
    import hashlib
    h = hashlib.sha256()
    for name in ("pkv_decode.cu", "pkv_internal.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_289_gb300", "csrc", name),
                  encoding="utf-8") as f:
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = []
        smax = None
        reasons = set()
        for p in rows:
            try:
                sm.append(float(p[1]))
                smax = float(p[2])
            except ValueError:
                continue
            for i, n in enumerate(names):
                if p[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate_max(value, world, device=None):
    """Max of a float over ranks (identity at world size 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_sum(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def workload_config(wl):
    return {"workload": wl.name, "batch": wl.N, "num_q_heads": wl.Hq, "num_kv_heads": wl.Hkv,
            "head_dim": wl.D, "block_size": wl.BS,
            "kv_dtype": ["bf16", "fp8_e4m3", "int8", "int4"][wl.kv_kind],
            "seq_lens": "log-uniform [128, 16384]" if wl.cfg in (5, 7, 9) else
            ("uniform [1024, 8192]" if wl.cfg in (2, 6) else "see workload"),
            "query_tokens_per_request": wl.q_len,
            "mean_seq_len": round(float(wl.seq_lens.mean()), 1), "num_blocks": wl.NB,
            "kv_bytes_per_step": wl.kv_read_bytes(),
            "l2": "inputs larger than L2 (%.2f GB of pages vs 129 MB L2); no flush"
                  % (2 * wl.NB * wl.Hkv * wl.BS * wl.D * wl.elt / 1e9)}


def decode_algorithmic_bytes(wl, unique=False, append=False):
    """Bytes one decode launch must move: every cached K/V row once, plus the block
    table entries, FP8 scales, q and out.  unique: rows of shared pages counted once
    (the shared-prefix call reads them once)."""
    nblk = sum(len(wl.blocks_of(r)) for r in range(wl.N))
    b = wl.unique_kv_read_bytes() if unique else wl.kv_read_bytes()
    b += nblk * 4                                        # block table entries read
    if wl.quant:
        b += nblk * wl.Hkv * 2 * 4                       # K and V scales
    b += 2 * wl.N * wl.q_len * wl.Hq * wl.D * 2          # q in, out
    if append:
        b += 4 * wl.N * wl.Hkv * wl.D * 2                # new K/V rows read and written
    return b


# ------------------------------------------------------------------ CPU oracle timing
def oracle_sample(wl, dd, reqs):
    """Host copies of the pages of `reqs` for the oracle (compact block table)."""
    import torch
    old, seen = [], {}
    bt = np.zeros((len(reqs), wl.MB), np.int32)
    for i, r in enumerate(reqs):
        for j, b in enumerate(wl.blocks_of(r)):
            b = int(b)
            if b not in seen:
                seen[b] = len(old)
                old.append(b)
            bt[i, j] = seen[b]
    idx = torch.tensor(old, dtype=torch.int64, device=dd["q"].device)

    def bits(t):
        if t.element_size() == 2:
            return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return t.contiguous().view(torch.uint8).cpu().numpy()
    kc = bits(dd["k_cache"].index_select(0, idx))
    vc = bits(dd["v_cache"].index_select(0, idx))
    q = bits(dd["q"][torch.tensor(reqs, device=idx.device)])
    ks = vs = None
    if wl.quant:
        ks = dd["k_scale"].index_select(0, idx).cpu().numpy()
        vs = dd["v_scale"].index_select(0, idx).cpu().numpy()
    return q, kc, vc, bt, wl.seq_lens[reqs].copy(), ks, vs


def time_oracle(wl, sample, units):
    """Time the oracle on `units` = list of (local request, kv head): all G query heads of
    each unit.  Returns (seconds, algorithmic KV bytes processed)."""
    import oracle
    q, kc, vc, bt, sl, ks, vs = sample
    rows = np.array([r * wl.Hq + h * wl.G + g for (r, h) in units for g in range(wl.G)], np.int64)
    t0 = time.perf_counter()
    oracle.decode_rows(q, kc, vc, bt, sl, wl.scale, rows, ks, vs)
    dt = time.perf_counter() - t0
    nbytes = int(sum(int(sl[r]) for (r, h) in units) * wl.D * 2 * wl.elt)
    return dt, nbytes


def cpu_baseline(wl, H, budget_s=15.0, single_budget_s=4.0):
    """The oracle timed on the host cores: the whole decode step of the first 16 requests
    (all their units), repeated until about `budget_s` seconds of CPU work; then the
    same sample on one thread for about `single_budget_s` seconds."""
    import oracle
    dd = {"q": H.inputs["q"], "k_cache": H.kc, "v_cache": H.vc, "k_scale": H.ks,
          "v_scale": H.vs}
    reqs = list(range(min(wl.N, 16)))
    sample = oracle_sample(wl, dd, reqs)
    units = [(i, h) for i in range(len(reqs)) for h in range(wl.Hkv)]
    t1, _ = time_oracle(wl, sample, units)
    reps = int(max(1, min(200, budget_s / max(t1, 1e-3))))
    tot_t, tot_b = 0.0, 0
    for _ in range(reps):
        dt, nb = time_oracle(wl, sample, units)
        tot_t += dt
        tot_b += nb
    cores = oracle.num_threads()
    # one thread: whole units of request 0 until the budget is spent
    oracle.set_num_threads(1)
    try:
        st, sb, n1 = 0.0, 0, 0
        while st < single_budget_s:
            dt, nb = time_oracle(wl, sample, units[:wl.Hkv])
            st += dt
            sb += nb
            n1 += 1
        # the tiny configuration (4 requests of 17..100 tokens, one KV head), whole
        # batch per pass, on the same one thread
        from paged_kv_cache_289_gb300 import workloads as W
        tw = W.make(1)
        td = W.host_data(tw)
        tb = int(tw.seq_lens.sum()) * tw.Hkv * tw.D * 2 * 2
        tt, tn = 0.0, 0
        while tt < 1.0:
            t0 = time.perf_counter()
            oracle.decode_attn(td["q"], td["k_cache"], td["v_cache"], tw.block_table,
                               tw.seq_lens, tw.scale)
            tt += time.perf_counter() - t0
            tn += 1
    finally:
        oracle.set_num_threads(cores)
    return {"value": round(tot_b / tot_t / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} passes over all {len(units)} (request, kv head) units x {wl.G} query "
                      f"heads of requests 0..{len(reqs)-1} of {wl.name} ({tot_b/1e9:.1f} GB of K/V "
                      f"in {tot_t:.1f} s); fp64 C + OpenMP",
            "single_thread": {"value": round(sb / st / 1e9, 4), "unit": UNIT, "cores": 1,
                              "sample": f"{n1} passes over the {wl.Hkv} units of request 0 "
                                        f"({sb/1e9:.2f} GB in {st:.1f} s)"},
            "single_thread_tiny": {"value": round(tb * tn / tt / 1e9, 4), "unit": UNIT,
                                   "cores": 1,
                                   "sample": f"{tn} passes over the whole tiny batch "
                                             f"({tw.name}: {tw.N} requests, {tb} B of K/V per "
                                             f"pass, {tt:.2f} s)"}}


def l2_flush_buffer(torch, dev):
    """A buffer twice the 129 MB L2, read between launches to evict their pages.  It is
    written once here; reading it (rather than writing it every time) leaves no dirty
    lines in L2 for the timed launch to write back."""
    return torch.ones(2 * 129 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)


def gate(torch, stream):
    """A bounded GPU sleep (about 1 ms) queued just before a timed region opens: the host
    enqueues the region's first launches while it runs, so the first timed step does not
    wait on the host.  It sits before the start event and is not timed."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)


def median_of(ts):
    return statistics.median(ts) if ts else float("nan")


class StepHarness:
    """Device buffers and the launch sequence of one decode step of a workload.

    A step is slot mapping -> KV write -> decode (+ its merge kernel) on the main
    stream and the prefix block hash on a side stream.  `hash_mode` "full" re-hashes
    every request's whole token history (the chain from h_0); "resume" continues
    each chain from the hash of its last block that was full before this step
    (pkv_prefix_block_hash_resume), so only the blocks completed by the step's new
    tokens are read."""

    def __init__(self, wl, dev, hash_mode="full", shared_prefix=False, append=False):
        import torch
        import paged_kv_cache_289_gb300 as pkv
        from paged_kv_cache_289_gb300 import workloads as W
        self.wl, self.dev, self.hash_mode = wl, dev, hash_mode
        # decode through the shared-prefix call (the prefix-sharing workload only)
        self.prefix = wl.notes.get("shared_prefix_blocks", 0) * wl.BS if shared_prefix else 0
        # the decode writes the step's new rows itself (bf16 pages, one query)
        self.append = append and not wl.quant and wl.q_len == 1 and not self.prefix
        self.torch, self.pkv = torch, pkv
        dd = W.device_data(wl, dev)
        bt = torch.from_numpy(wl.block_table).to(dev)
        sl = torch.from_numpy(wl.seq_lens).to(dev)
        req_new, pos_new = wl.new_token_rows()      # the step's new tokens (q_len per request)
        if wl.quant:
            kc = torch.zeros(wl.cache_shape, dtype=torch.int8 if wl.int8 else torch.uint8,
                             device=dev)
            vc = torch.zeros_like(kc)
            req_all, pos_all = W.token_rows_order(wl)
            sm_all = pkv.compute_slot_mapping(bt, torch.from_numpy(pos_all).to(dev), wl.BS,
                                              req_idx=torch.from_numpy(req_all).to(dev))
            pkv.kv_cache_write(dd["k_rows"], dd["v_rows"], sm_all, kc, vc, dd["k_scale"],
                               dd["v_scale"])
            del dd["k_rows"], dd["v_rows"], sm_all
            self.ks, self.vs = dd["k_scale"], dd["v_scale"]
        else:
            kc, vc = dd["k_cache"], dd["v_cache"]
            self.ks = self.vs = None
        self.kc, self.vc = kc, vc
        B = wl.hash_block
        lens = np.diff(wl.token_offsets)
        tokens = torch.from_numpy(wl.tokens).to(dev)
        toffs = torch.from_numpy(wl.token_offsets).to(dev)
        full = lens // B
        if hash_mode == "full":
            per_seq = full
        else:
            # blocks that were full before this step's q_len new tokens
            self.first_np = np.maximum(lens - wl.q_len, 0) // B
            per_seq = full - self.first_np
        ho_np = np.zeros(wl.N + 1, np.int64)
        np.cumsum(per_seq, out=ho_np[1:])
        self.nh = int(ho_np[-1])
        hoffs = torch.from_numpy(ho_np).to(dev)
        self.inputs = {"q": dd["q"], "k_new": dd["k_new"], "v_new": dd["v_new"],
                       "pos": torch.from_numpy(pos_new).to(dev),
                       "req": torch.from_numpy(req_new).to(dev),
                       "qoffs": torch.from_numpy(wl.q_offsets()).to(dev), "bt": bt, "sl": sl,
                       "tokens": tokens, "toffs": toffs, "hoffs": hoffs}
        if hash_mode == "resume":
            # h_k of every sequence, carried over from the previous step in a serving
            # loop; here taken once from the full chain
            fho = np.zeros(wl.N + 1, np.int64)
            np.cumsum(full, out=fho[1:])
            chain = pkv.prefix_block_hash(tokens, toffs, B, torch.from_numpy(fho).to(dev),
                                          int(fho[-1]), seed=0).cpu().numpy().view(np.uint64)
            prev = np.array([chain[fho[s] + self.first_np[s] - 1] if self.first_np[s] > 0 else 0
                             for s in range(wl.N)], np.uint64)
            self.inputs["prev_hashes"] = torch.from_numpy(prev.view(np.int64)).to(dev)
            self.inputs["first_blocks"] = torch.from_numpy(self.first_np.astype(np.int64)).to(dev)
        self.outputs = {"out": torch.empty_like(dd["q"]),
                        "hashes": torch.empty(max(self.nh, 1), dtype=torch.int64, device=dev)}
        self.slots = torch.empty(wl.N * wl.q_len, dtype=torch.int64, device=dev)
        self.ws = torch.zeros(pkv.multiquery_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS,
                                                            wl.kv_kind, wl.q_len),
                              dtype=torch.uint8, device=dev)
        if self.prefix:
            self.ws = torch.zeros(pkv.shared_prefix_workspace_size(wl.N, wl.Hq, wl.Hkv, wl.D,
                                                                   wl.BS, self.prefix),
                                  dtype=torch.uint8, device=dev)
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(dev)
        # slot map, write, decode, wide-split merge, hash (+ the prefix pass of the
        # shared-prefix call)
        self.launches_per_step = 6 if self.prefix else (4 if self.append else 5)

    def decode(self, I, O, stream):
        wl, pkv = self.wl, self.pkv
        if self.prefix:
            pkv.paged_decode_attn_shared_prefix(I["q"], self.kc, self.vc, I["bt"], I["sl"],
                                                wl.scale, self.prefix, out=O["out"],
                                                workspace=self.ws, stream=stream)
        elif wl.q_len == 1:
            pkv.paged_decode_attn(I["q"], self.kc, self.vc, I["bt"], I["sl"], wl.scale,
                                  out=O["out"], k_scale=self.ks, v_scale=self.vs,
                                  workspace=self.ws, stream=stream)
        else:
            pkv.paged_multiquery_attn(I["q"], I["qoffs"], wl.q_len, self.kc, self.vc, I["bt"],
                                      I["sl"], wl.scale, out=O["out"], k_scale=self.ks,
                                      v_scale=self.vs, workspace=self.ws, stream=stream)

    def step(self, I, O, dec_ev=None):
        """One decode step on the per-step inputs I, writing the results O.

        The prefix hash reads only the step's tokens, so it starts first, on the side
        stream, and runs beside the main-stream chain (slot mapping -> write -> decode ->
        merge).  Started after the KV write instead, it lands on SMs that the decode grid
        already fills and stretches the decode's tail (measured: +17 us per step)."""
        wl, pkv, main, side = self.wl, self.pkv, self.main, self.side
        side.wait_stream(main)                   # the step's inputs are in place
        if self.append:
            # slot mapping feeds nothing on the main stream when the decode writes the
            # new rows itself: it runs beside the decode
            pkv.compute_slot_mapping(I["bt"], I["pos"], wl.BS, req_idx=I["req"], out=self.slots,
                                     stream=side)
        if self.hash_mode == "full":
            pkv.prefix_block_hash(I["tokens"], I["toffs"], wl.hash_block, I["hoffs"], self.nh,
                                  seed=0, out=O["hashes"], stream=side)
        else:
            pkv.prefix_block_hash_resume(I["tokens"], I["toffs"], wl.hash_block,
                                         I["prev_hashes"], I["first_blocks"], I["hoffs"],
                                         self.nh, out=O["hashes"], stream=side)
        if not self.append:
            pkv.compute_slot_mapping(I["bt"], I["pos"], wl.BS, req_idx=I["req"], out=self.slots,
                                     stream=main)
            pkv.kv_cache_write(I["k_new"], I["v_new"], self.slots, self.kc, self.vc, self.ks,
                               self.vs, stream=main)
        if dec_ev is not None:
            dec_ev[0].record(main)
        if self.append:
            pkv.paged_decode_attn_append(I["q"], I["k_new"], I["v_new"], self.kc, self.vc,
                                         I["bt"], I["sl"], wl.scale, out=O["out"],
                                         workspace=self.ws, stream=main)
        else:
            self.decode(I, O, main)
        if dec_ev is not None:
            dec_ev[1].record(main)
        main.wait_stream(side)

    def time_steps(self, K, warmup):
        """Device time of K steps (seconds), after `warmup` untimed steps."""
        torch = self.torch
        for _ in range(max(warmup, 3)):
            self.step(self.inputs, self.outputs)
        torch.cuda.synchronize(self.dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        gate(torch, self.main)
        e0.record(self.main)
        for _ in range(K):
            self.step(self.inputs, self.outputs)
        e1.record(self.main)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) / 1e3

    def time_decode_launches(self, n=50, warmup=10, flush=None):
        """Per-launch device times (seconds) of the decode call alone: `warmup` untimed
        launches, then n launches each bracketed by events; `flush` (a buffer larger
        than L2) is read through before every timed launch."""
        torch = self.torch
        for _ in range(warmup):
            self.decode(self.inputs, self.outputs, self.main)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        torch.cuda.synchronize(self.dev)
        for i in range(n):
            if flush is not None:
                flush.sum()
            ev[i][0].record(self.main)
            self.decode(self.inputs, self.outputs, self.main)
            ev[i][1].record(self.main)
        torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) / 1e3 for a, b in ev]


def per_workload_figures(dev, peak, main_harness=None):
    """Decode-launch rooflines measured in the same run: the headline workload (2), long
    contexts (3), E4M3 / INT8 / INT4 pages (5, 7, 9) and four query positions (6) with an
    L2 flush between launches; prefix sharing (4) on logical and on unique bytes, with and
    without the flush; and workload 3's whole step with the full and the resumed prefix
    hash; then the tensor-core prefill (workload 8, bf16 and INT4 pages) and the
    copy-on-write block copy.  Each decode launch figure is the median of 50 after 10
    warm-ups.  Launched alone, the
    decode kernels of workloads 6, 7 and 9 do not meet the full re-hash's CTAs, which in a
    step (hash first, on the side stream) hold SM resources those register-heavy plans
    need and delay some of their persistent CTAs."""
    import torch
    import paged_kv_cache_289_gb300 as pkv
    from paged_kv_cache_289_gb300 import workloads as W
    flush = l2_flush_buffer(torch, dev)
    res = {}
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for cfg in (2, 3, 5, 7, 9, 6, 4):
        if cfg == 2 and main_harness is None:
            continue
        wl = main_harness.wl if cfg == 2 else W.make(cfg)
        h = main_harness if cfg == 2 else StepHarness(wl, dev, "full")
        alg = decode_algorithmic_bytes(wl)
        entry = {"workload": wl.name, "batch": wl.N, "kv_dtype": ["bf16", "fp8_e4m3", "int8",
                                                                  "int4"][wl.kv_kind],
                 "algorithmic_bytes_per_launch": alg}
        ts = h.time_decode_launches(flush=flush)
        med, mean = median_of(ts), sum(ts) / len(ts)
        entry.update({"median_launch_ms": round(med * 1e3, 4), "avg_launch_ms": round(mean * 1e3, 4),
                      "achieved": round(alg / med / 1e9, 1), "frac": round(alg / med / 1e9 / peak, 4),
                      "query_tokens_per_s": round(wl.N * wl.q_len / med, 1),
                      "l2": "flushed (a 258 MB buffer read) before every timed launch"})
        assert pkv.read_device_error(h.ws) == 0, "device error word set"
        if cfg == 2:
            # the serving form of the same step: each chain resumed from its last full
            # block, the new rows written by the decode kernel (slot mapping beside it)
            K = 50
            hs = StepHarness(wl, dev, "resume", append=True)
            t_s = hs.time_steps(K, 10)
            assert pkv.read_device_error(hs.ws) == 0, "device error word set"
            entry["serving_step"] = {
                "ms_per_step": round(t_s / K * 1e3, 4),
                "kv_gbs": round(wl.kv_read_bytes() * K / t_s / 1e9, 1),
                "steps": K,
                "what": "slot mapping (beside the decode) + pkv_paged_decode_attn_append (the "
                        "new rows written by the decode kernel) + merge + "
                        "pkv_prefix_block_hash_resume (only the blocks the step completes)"}
            hs = None
        if cfg == 4:
            uniq = wl.unique_kv_read_bytes()
            logical = wl.kv_read_bytes()
            ts_nf = h.time_decode_launches(flush=None)
            med_nf = median_of(ts_nf)
            entry.update({
                "logical_kv_bytes": logical, "unique_kv_bytes": uniq,
                "flushed": {"median_launch_ms": round(med * 1e3, 4),
                            "logical_gbs": round(logical / med / 1e9, 1),
                            "unique_gbs": round(uniq / med / 1e9, 1),
                            "unique_frac": round(uniq / med / 1e9 / peak, 4)},
                "no_flush": {"median_launch_ms": round(med_nf * 1e3, 4),
                             "logical_gbs": round(logical / med_nf / 1e9, 1),
                             "unique_gbs": round(uniq / med_nf / 1e9, 1),
                             "unique_frac": round(uniq / med_nf / 1e9 / peak, 4)},
                "note": "the shared 4096-token prefix (16 MB of pages) is read by every "
                        "request; logical bytes count it per request, unique bytes once"})
            # the same batch through the shared-prefix call: the shared pages once
            hs = StepHarness(wl, dev, "full", shared_prefix=True)
            fig = {}
            for key, fl in (("flushed", flush), ("no_flush", None)):
                t = median_of(hs.time_decode_launches(flush=fl))
                fig[key] = {"median_launch_ms": round(t * 1e3, 4),
                            "logical_gbs": round(logical / t / 1e9, 1),
                            "unique_gbs": round(uniq / t / 1e9, 1),
                            "unique_frac": round(uniq / t / 1e9 / peak, 4)}
            assert pkv.read_device_error(hs.ws) == 0, "device error word set"
            fig["what"] = ("pkv_paged_decode_attn_shared_prefix: the 4096 shared tokens "
                           "attended once for all 128 requests on the tensor cores, the tails "
                           "by the decode kernel, a log-sum-exp merge")
            entry["shared_prefix_call"] = fig
            hs = None
        if cfg == 3:
            K = 50
            t_full = h.time_steps(K, 10)
            h = None                             # free its pages before the second harness
            torch.cuda.empty_cache()
            hr = StepHarness(wl, dev, "resume")
            t_res = hr.time_steps(K, 10)
            kvb = wl.kv_read_bytes()
            entry["step"] = {
                "full_hash": {"ms_per_step": round(t_full / K * 1e3, 4),
                              "kv_gbs": round(kvb * K / t_full / 1e9, 1),
                              "hashed_blocks_per_step": int(sum(np.diff(wl.token_offsets)
                                                                // wl.hash_block))},
                "resumed_hash": {"ms_per_step": round(t_res / K * 1e3, 4),
                                 "kv_gbs": round(kvb * K / t_res / 1e9, 1),
                                 "hashed_blocks_per_step": hr.nh},
                "steps": K,
                "what": "slot mapping + KV write + decode + prefix hash; full re-hashes "
                        "every token of every request, resumed hashes only the blocks the "
                        "step's new token completed (pkv_prefix_block_hash_resume)"}
            del hr
        res[str(cfg)] = entry
        del h
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    res.update(prefill_and_copy_figures(dev, peak))
    res["clocks"] = sampler.stop()
    return res


def launch_times(torch, stream, launch, n, warmup, flush=None):
    """Device times (seconds) of n launches of launch(i), each bracketed by events on
    `stream`, after `warmup` untimed ones; `flush` (a buffer larger than L2) is read
    before every timed launch when given."""
    for i in range(warmup):
        launch(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for k in range(n):
        if flush is not None:
            flush.sum()
        ev[k][0].record(stream)
        launch(warmup + k)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / 1e3 for a, b in ev]


def prefill_and_copy_figures(dev, hbm_peak):
    """The tensor-core prefill (workload 8, bf16 and INT4 pages: median of 30 launches after
    5, no flush: compute-bound) and the copy-on-write block copy (4,096 random pairs of the
    70B pool, a fresh mapping per launch: median of 50 after 10), measured in the same run
    as the decode figures."""
    import torch
    res = {}
    main = torch.cuda.current_stream(dev)
    peak, peak_kind = bf16_peak()
    for kv in ("bf16", "int4"):
        wl, dd, kc, vc, ks, vs, launch, err = prefill_case(dev, kv, None, main)
        ts = launch_times(torch, main, lambda i: launch(), 30, 5)
        assert int(err.item()) == 0, "device error word set"
        med = median_of(ts)
        flops = wl.prefill_flops()
        res["8" if kv == "bf16" else "8_int4"] = {
            "workload": wl.name, "batch": wl.N, "pages": kv,
            "kernel": "pkv_prefill_kernel" if kv == "bf16"
                      else "pkv_dequant_pages_kernel + pkv_prefill_kernel",
            "flops_per_launch": flops, "median_launch_ms": round(med * 1e3, 4),
            "achieved_tflops": round(flops / med / 1e12, 1),
            "frac": round(flops / med / 1e12 / peak, 4), "peak": peak, "peak_source": peak_kind,
            "l2": "no flush (compute-bound)"}
        del wl, dd, kc, vc, ks, vs, launch, err
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    import paged_kv_cache_289_gb300 as pkv
    NB, Hkv, BS, D, P, kc, vc, maps = copy_case(dev, 4096, 60)
    ts = launch_times(torch, main, lambda i: pkv.copy_blocks(kc, vc, maps[i % len(maps)],
                                                             stream=main), 50, 10)
    med = median_of(ts)
    alg = copy_algorithmic_bytes(P, Hkv, BS, D)
    res["copy_blocks"] = {
        "workload": "copy_blocks_llama70b_pool", "pairs_per_launch": P, "num_blocks": NB,
        "algorithmic_bytes_per_launch": alg, "median_launch_ms": round(med * 1e3, 4),
        "achieved": round(alg / med / 1e9, 1), "frac": round(alg / med / 1e9 / hbm_peak, 4),
        "l2": "fresh random mapping per launch"}
    del kc, vc, maps
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    import paged_kv_cache_289_gb300 as pkv
    from paged_kv_cache_289_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pkv.lib()

    wl = W.make(args.workload, seed=(args.seed if args.seed is not None else args.workload) + rank,
                batch=args.batch)
    H = StepHarness(wl, dev, args.hash, shared_prefix=args.shared_prefix, append=args.append)
    quant = wl.quant
    main = H.main
    inputs, outputs = H.inputs, H.outputs
    step = H.step
    for _ in range(max(args.warmup, 3)):
        step(inputs, outputs)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()

    # ---------------- device-timed region: exactly K steps
    K = args.steps
    dec_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    gate(torch, main)
    e0.record(main)
    for k in range(K):
        step(inputs, outputs, dec_events[k])
    e1.record(main)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    t_total = e0.elapsed_time(e1) / 1e3
    dec_times = [a.elapsed_time(b) / 1e3 for a, b in dec_events]
    dec_avg = sum(dec_times) / len(dec_times)
    dec_med = median_of(dec_times)
    assert pkv.read_device_error(H.ws) == 0, "device error word set during the benchmark"

    t_max = aggregate_max(t_total, world, dev)
    kv_bytes = wl.kv_read_bytes()
    total_bytes = aggregate_sum(float(kv_bytes) * K, world, dev)
    total_q = aggregate_sum(float(wl.N * wl.q_len) * K, world, dev)
    value = total_bytes / t_max / 1e9
    ms_per_step = t_max / K * 1e3

    # ---------------- roofline of the dominant launch (decode: main + merge kernels)
    peak, peak_kind = peak_hbm()
    alg = decode_algorithmic_bytes(wl, unique=bool(H.prefix), append=H.append)
    achieved = alg / dec_avg / 1e9
    traffic = recorded_traffic(kernel_source_hash(), wl.name)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} hbm_gbs (copy, read+write bytes)",
                "kernel": ("pkv_paged_decode_attn_shared_prefix (pkv_prefill_kernel over the "
                           "shared pages, pkv_decode_kernel over the tails, merge)"
                           if H.prefix else
                           ("pkv_paged_decode_attn_append (pkv_decode_kernel writing the new rows)"
                            if H.append else "pkv_paged_decode_attn (pkv_decode_kernel)")),
                "algorithmic_bytes_per_launch": alg,
                "avg_launch_ms": round(dec_avg * 1e3, 4),
                "median_launch_ms": round(dec_med * 1e3, 4),
                "note": "per-launch events inside the timed steps; an event between the KV "
                        "write and the decode stops the decode's programmatic early launch, "
                        "so the launch time includes that start-up (about 6 us)"}

    # ---------------- end to end through the public API with pinned host buffers
    e2e = None
    if not args.skip_e2e:
        # Serving-style loop: every step's inputs (q, new K/V, positions, block table,
        # lengths, tokens) go up from one packed pinned buffer and its results (out,
        # hashes) come back, one copy each way per step.  Copies run on their own
        # streams, double-buffered, so step k+1's upload overlaps step k's kernels.
        def packed(tensors):
            offs, o = {}, 0
            for name, t in tensors.items():
                offs[name] = (o, t.numel() * t.element_size())
                o += (offs[name][1] + 255) // 256 * 256
            return offs, o

        in_offs, in_bytes = packed(inputs)
        out_offs, out_bytes = packed(outputs)
        hin = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        for name, t in inputs.items():
            o, n = in_offs[name]
            hin[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        hout = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
        din = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        dout = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]

        def views(buf, offs, like):
            return {name: buf[offs[name][0]:offs[name][0] + offs[name][1]].view(t.dtype)
                    .view(t.shape) for name, t in like.items()}

        I2 = [views(din[b], in_offs, inputs) for b in range(2)]
        O2 = [views(dout[b], out_offs, outputs) for b in range(2)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(k):
            b = k & 1
            up.wait_event(ev_done[b])            # step k-2 finished reading set b
            with torch.cuda.stream(up):
                din[b].copy_(hin, non_blocking=True)
            ev_in[b].record(up)
            main.wait_event(ev_in[b])
            main.wait_event(ev_out[b])           # step k-2's results of set b are home
            step(I2[b], O2[b])
            ev_done[b].record(main)
            down.wait_event(ev_done[b])
            with torch.cuda.stream(down):
                hout[b].copy_(dout[b], non_blocking=True)
            ev_out[b].record(down)

        for k in range(4):
            e2e_step(k)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(main)
        up.wait_stream(main)                     # no upload starts before the timed region
        h0 = time.perf_counter()
        for k in range(K):
            e2e_step(k)
        main.wait_stream(down)
        f1.record(main)
        h1 = time.perf_counter()                 # host time to issue the K steps
        torch.cuda.synchronize(dev)
        te = aggregate_max(f0.elapsed_time(f1) / 1e3, world, dev)
        e2e = {"value": round(total_bytes / te / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(sum(n for _, n in in_offs.values())),
               "d2h_bytes_per_step": int(sum(n for _, n in out_offs.values())),
               "ms_per_step": round(te / K * 1e3, 4),
               "host_issue_ms_per_step": round((h1 - h0) / K * 1e3, 4),
               "copies": "one packed H2D and one D2H per step on their own streams, "
                         "double-buffered (upload of step k+1 overlaps step k)"}

    per_wl = None
    if rank == 0 and world == 1 and not args.skip_per_workload and args.workload == 2 \
            and args.batch is None:
        per_wl = per_workload_figures(dev, peak, H)

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = cpu_baseline(wl, H)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
                "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": ("bf16" if not quant else
                          ["", "fp8_e4m3", "int8", "int4"][wl.kv_kind] + " KV, bf16 q/out, fp32 accumulate"),
                "data": "synthetic (seeded N(0,1) q/K/V, uniform token ids)",
                "config": dict(workload_config(wl), hash=args.hash,
                               shared_prefix_tokens=H.prefix,
                               cache_write=("in the decode kernel (append)" if H.append
                                            else "pkv_kv_cache_write before the decode"),
                               parallelism=f"{world} independent replicas (no collective)"),
                "query_tokens_per_s": round(total_q / t_max, 1),
                "pct_of_hbm_peak": round(100 * value / peak, 2),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": H.launches_per_step * K, "clocks": clocks,
                "per_workload": per_wl}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------ block copy alone
def copy_case(dev, pairs, n_maps):
    """The 70B-layer pool (20,480 blocks of 8 KV heads x 16 tokens x 128 bf16 per cache)
    and n_maps fresh random (source, destination) mappings of `pairs` pairs each."""
    import torch
    NB, Hkv, BS, D = 20480, 8, 16, 128
    P = min(pairs, NB // 2)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    kc = torch.randn((NB, Hkv, BS, D), generator=g, device=dev, dtype=torch.bfloat16)
    vc = torch.randn((NB, Hkv, BS, D), generator=g, device=dev, dtype=torch.bfloat16)
    rng = np.random.default_rng(6)
    maps = []
    for _ in range(n_maps):
        ids = rng.permutation(NB)
        maps.append(torch.from_numpy(np.stack([ids[:P], ids[P:2 * P]], 1).astype(np.int32))
                    .to(dev))
    return NB, Hkv, BS, D, P, kc, vc, maps


def copy_algorithmic_bytes(P, Hkv, BS, D):
    """K and V blocks read and written per pair, plus the pair's two int32 ids."""
    return P * (2 * 2 * Hkv * BS * D * 2 + 2 * 4)


def run_copy_blocks(args):
    """pkv_copy_blocks on the 70B-layer pool (8 KV heads x 16 tokens x 128 bf16: 32 KB per
    block and cache, 20,480 blocks, 1.34 GB for K and V): `--pairs` (source, destination)
    pairs per launch, a fresh random mapping per launch so no launch re-reads the previous
    one's destinations from L2."""
    import torch
    import paged_kv_cache_289_gb300 as pkv
    from oracle.block_manager import copy_blocks as oracle_copy

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    K, Wm = args.steps, max(args.warmup, 3)
    NB, Hkv, BS, D, P, kc, vc, maps = copy_case(dev, args.pairs, min(K + Wm, 64))
    main = torch.cuda.current_stream(dev)
    for i in range(Wm):
        pkv.copy_blocks(kc, vc, maps[i % len(maps)], stream=main)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = ClockSampler(0)
    sampler.start()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gate(torch, main)
    e0.record(main)
    for k in range(K):
        ev[k][0].record(main)
        pkv.copy_blocks(kc, vc, maps[(Wm + k) % len(maps)], stream=main)
        ev[k][1].record(main)
    e1.record(main)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    t = e0.elapsed_time(e1) / 1e3
    avg = sum(a.elapsed_time(b) for a, b in ev) / K / 1e3
    block_bytes = Hkv * BS * D * 2
    alg = copy_algorithmic_bytes(P, Hkv, BS, D)
    peak, peak_kind = peak_hbm()
    # oracle: the same copy on host memory, a bounded sample of pairs
    kh = np.zeros((2048, Hkv, BS, D), np.uint16)
    vh = np.zeros_like(kh)
    mp = np.stack([np.arange(0, 1024), np.arange(1024, 2048)], 1)
    cpu = None
    if not args.skip_cpu:
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 10.0:
            oracle_copy(kh, vh, mp)
            reps += 1
        tc = time.perf_counter() - t0
        cpu = {"value": round(reps * 1024 * 4 * block_bytes / tc / 1e9, 3), "unit": "GB/s",
               "cores": 1, "kind": "oracle",
               "sample": f"{reps} x 1024 pairs of 32 KB blocks in host memory (numpy, {tc:.1f} s)"}
    line = {"metric": "copy-on-write block copy: HBM GB/s (read + write)",
            "value": round(alg * K / t / 1e9, 2), "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": Wm, "ms_per_step": round(t / K * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 bytes (copy)",
            "data": "synthetic", "config": {"workload": "copy_blocks_llama70b_pool",
                                            "num_blocks": NB, "pairs_per_launch": P,
                                            "block_bytes_per_cache": block_bytes,
                                            "l2": "fresh random mapping per launch; "
                                                  f"{alg / 1e6:.0f} MB moved per launch"},
            "roofline": {"bound": "hbm", "achieved": round(alg / avg / 1e9, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(alg / avg / 1e9 / peak, 4),
                         "traffic": None, "peak_source": f"{peak_kind} hbm_gbs",
                         "kernel": "pkv_copy_blocks_kernel", "algorithmic_bytes_per_launch": alg,
                         "avg_launch_ms": round(avg * 1e3, 4)},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": K, "clocks": clocks}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ prefill attention
def prefill_case(dev, kv="bf16", batch=None, stream=None):
    """Workload 8 on the device, ready to launch: (wl, device data, K/V caches, scales,
    launch(), device error word).  kv picks the page kind; quantised pages are written by
    the library's own cache write from the source rows."""
    import torch
    import paged_kv_cache_289_gb300 as pkv
    from paged_kv_cache_289_gb300 import workloads as W
    wl = W.make(8, batch=batch)
    wl.fp8, wl.int8, wl.int4 = kv == "fp8", kv == "int8", kv == "int4"
    dd = W.device_data(wl, dev)
    qo = torch.from_numpy(wl.q_offsets()).to(dev)
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(dd["q"])
    ks = vs = ws = None
    if wl.quant:
        kc = torch.zeros(wl.cache_shape, dtype=torch.int8 if wl.int8 else torch.uint8,
                         device=dev)
        vc = torch.zeros_like(kc)
        req, pos = W.token_rows_order(wl)
        slots = pkv.compute_slot_mapping(bt, torch.from_numpy(pos).to(dev), wl.BS,
                                         req_idx=torch.from_numpy(req).to(dev))
        ks, vs = dd["k_scale"], dd["v_scale"]
        pkv.kv_cache_write(dd["k_rows"], dd["v_rows"], slots, kc, vc, ks, vs)
        ws = torch.empty(pkv.prefill_workspace_size(wl.N, wl.MB, wl.Hkv, wl.D, wl.BS,
                                                    wl.kv_kind), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)
        del slots
    else:
        kc, vc = dd["k_cache"], dd["v_cache"]

    def launch():
        pkv.paged_prefill_attn(dd["q"], qo, wl.max_q_len, kc, vc, bt, sl, wl.scale, out=out,
                               k_scale=ks, v_scale=vs, workspace=ws, error_word=err,
                               stream=stream)
    return wl, dd, kc, vc, ks, vs, launch, err


def bf16_peak():
    """The bf16 tensor peak the prefill is read against: MEASURED_PEAKS.json's cuBLAS
    burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), "measured bf16_tflops (cuBLAS burst)"
    except Exception:
        return 1900.0, "fallback bf16 burst"


def run_prefill(args):
    """pkv_paged_prefill_attn on workload 8: 8 requests, each a 2048-token prompt chunk
    after a cached context of U[0, 6144] tokens, Llama-3.3-70B layer shape (64/8 heads,
    head_dim 128, bf16, 16-token blocks).  Metric: causal-effective attention TFLOP/s."""
    import torch
    import oracle

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    main = torch.cuda.current_stream(dev)
    wl, dd, kc, vc, ks, vs, launch, err = prefill_case(dev, args.prefill_kv, args.batch, main)

    K, Wm = args.steps, max(args.warmup, 3)
    for _ in range(Wm):
        launch()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = ClockSampler(0)
    sampler.start()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gate(torch, main)
    e0.record(main)
    for k in range(K):
        ev[k][0].record(main)
        launch()
        ev[k][1].record(main)
    e1.record(main)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    assert int(err.item()) == 0, "device error word set during the benchmark"
    t = e0.elapsed_time(e1) / 1e3
    avg = sum(a.elapsed_time(b) for a, b in ev) / K / 1e3
    flops = wl.prefill_flops()
    peak, peak_kind = bf16_peak()
    achieved = flops / avg / 1e12
    # oracle: sampled rows of the same workload on the host cores, about 10 s
    q = dd["q"].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    if wl.quant:
        kc_h = kc.cpu().numpy()
        vc_h = vc.cpu().numpy()
        ks_h, vs_h = ks.cpu().numpy(), vs.cpu().numpy()
    else:
        kc_h = kc.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        vc_h = vc.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        ks_h = vs_h = None
    rng = np.random.default_rng(1)
    qo_np = wl.q_offsets()
    ql = wl.query_lens
    tot_t, tot_f, n_rows = 0.0, 0, 0
    while tot_t < (0.0 if args.skip_cpu else 10.0):
        rows = rng.integers(0, wl.total_q * wl.Hq, size=64).astype(np.int64)
        t0 = time.perf_counter()
        oracle.multiquery_rows(q, qo_np, kc_h, vc_h, wl.block_table, wl.seq_lens, wl.scale, rows,
                               ks_h, vs_h)
        tot_t += time.perf_counter() - t0
        for row in rows:
            tq_ = int(row) // wl.Hq
            r = int(np.searchsorted(qo_np, tq_, side="right")) - 1
            vis = int(wl.seq_lens[r]) - int(ql[r]) + (tq_ - int(qo_np[r])) + 1
            tot_f += max(0, min(vis, int(wl.seq_lens[r]))) * 4 * wl.D
        n_rows += rows.shape[0]
    cpu = None if args.skip_cpu else {
           "value": round(tot_f / tot_t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
           "kind": "oracle", "sample": f"{n_rows} random (token, head) rows of {wl.name} "
                                       f"({tot_f/1e9:.1f} GFLOP in {tot_t:.1f} s), fp64 C + OpenMP"}
    pages = "bf16" if not wl.quant else {1: "E4M3", 2: "int8", 3: "int4"}[wl.kv_kind]
    kern = "pkv_prefill_kernel" if not wl.quant else "pkv_dequant_pages_kernel + pkv_prefill_kernel"
    line = {"metric": "paged prefill attention: causal-effective TFLOP/s (bf16 tensor cores)",
            "value": round(flops * K / t / 1e12, 2), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": K, "warmup": Wm, "ms_per_step": round(t / K * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) q/K/V)",
            "config": {"workload": wl.name, "batch": wl.N, "num_q_heads": wl.Hq,
                       "num_kv_heads": wl.Hkv, "head_dim": wl.D, "block_size": wl.BS,
                       "chunk_tokens": int(ql.max()), "context": "U[0, 6144] cached tokens",
                       "pages": pages,
                       "flops_per_launch": flops,
                       "l2": "pages %.0f MB + q/out %.0f MB; no flush (compute-bound)" % (
                           2 * wl.NB * wl.Hkv * wl.BS * wl.D * wl.elt / 1e6,
                           2 * wl.total_q * wl.Hq * wl.D * 2 / 1e6)},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_source": peak_kind, "kernel": kern,
                         "flops_per_launch": flops, "avg_launch_ms": round(avg * 1e3, 4)},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": K * (2 if wl.quant else 1),
            "clocks": clocks}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_289_gb300 import workloads as W
    wl = W.make(args.workload, seed=args.seed if args.seed is not None else args.workload)
    d = {}
    # host copies of a bounded sample (the first 4 requests) drawn on the host generator
    reqs = list(range(min(4, wl.N)))
    sub = W.custom(len(reqs), wl.Hq, wl.Hkv, wl.D, wl.BS, wl.seq_lens[reqs], fp8=wl.fp8,
                   int8=wl.int8, int4=wl.int4, seed=wl.seed, scale=wl.scale,
                   name=wl.name + "_sample")
    hd = W.host_data(sub)
    if sub.quant:
        req_all, pos_all = W.token_rows_order(sub)
        sm = oracle.slot_mapping(sub.block_table, req_all, pos_all, sub.BS)
        kc = np.zeros(sub.cache_shape, sub.cache_np_dtype)
        vc = np.zeros_like(kc)
        oracle.kv_cache_write(hd["k_rows"], hd["v_rows"], sm, kc, vc, hd["k_scale"], hd["v_scale"])
        ks, vs = hd["k_scale"], hd["v_scale"]
    else:
        kc, vc, ks, vs = hd["k_cache"], hd["v_cache"], None, None
    sample = (hd["q"], kc, vc, sub.block_table, sub.seq_lens, ks, vs)
    units = [(i, h) for i in range(len(reqs)) for h in range(wl.Hkv)]
    t1, _ = time_oracle(sub, sample, units[:1])
    K, Wm = args.steps, max(args.warmup, 3)
    per_step = min(2.0, 120.0 / (K + Wm))
    n = int(max(1, min(len(units), per_step / max(t1, 1e-4))))
    for i in range(Wm):
        time_oracle(sub, sample, units[:n])
    tot_t = 0.0
    tot_b = 0
    for i in range(K):
        dt, nb = time_oracle(sub, sample, units[:n])
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    cpu = {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"per step: {n} (request, kv head) units x {wl.G} query heads of the first "
                     f"{len(reqs)} requests of {wl.name} (same shapes and lengths), fp64 C + OpenMP"}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(tot_t / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(wl), parallelism="host cores"),
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "copy_blocks":
        run_copy_blocks(args)
    elif args.op == "prefill":
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Helpers shared by the GPU parity tests: move seeded workloads to the device,
run the library path and the oracle path on the same inputs, compare."""
from __future__ import annotations

import numpy as np

import oracle
from paged_kv_cache_289_gb300 import workloads as W

# Tolerances of the attention output against the fp64 oracle (fp32 accumulation).
BF16_MAX_ABS = 1e-2
BF16_REL_L2 = 5e-3
FP8_MAX_ABS = 5e-2


def torch_cache_dtype(wl):
    torch = torch_mod()
    return torch.int8 if wl.int8 else (torch.uint8 if (wl.fp8 or wl.int4) else torch.bfloat16)


def pkv_kind(wl):
    return wl.kv_kind


def torch_mod():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def to_dev(a, dtype=None):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits):
    torch = torch_mod()
    return to_dev(np.ascontiguousarray(bits).view(np.int16), torch.bfloat16)


def dev_bits(t):
    """Device tensor -> numpy bit patterns (uint16 for 2-byte, int8 for int8, uint8 for
    other 1-byte tensors)."""
    torch = torch_mod()
    if t.dtype == torch.int8:
        return t.contiguous().cpu().numpy()
    if t.element_size() == 2:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().view(torch.uint8).cpu().numpy()


def out_to_f64(out):
    return W.bf16_bits_to_f32(dev_bits(out)).astype(np.float64)


def compare(got, ref, fp8):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / nrm) if nrm > 0 else 0.0
    if fp8:
        assert max_abs <= FP8_MAX_ABS, f"fp8 max-abs {max_abs}"
    else:
        assert max_abs <= BF16_MAX_ABS, f"bf16 max-abs {max_abs}"
        assert rel <= BF16_REL_L2, f"bf16 rel-L2 {rel}"
    return max_abs, rel


class HostCase:
    """A workload held on the host for both sides: the oracle's own caches and
    the same inputs uploaded for the library."""

    def __init__(self, wl, seed_offset=1000):
        self.wl = wl
        self.d = W.host_data(wl, seed_offset)
        if wl.quant:
            # each side quantises the source rows with its own write
            req, pos = W.token_rows_order(wl)
            self.req_all, self.pos_all = req, pos
            slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
            self.kc = np.zeros(wl.cache_shape, wl.cache_np_dtype)
            self.vc = np.zeros_like(self.kc)
            oracle.kv_cache_write(self.d["k_rows"], self.d["v_rows"], slots, self.kc, self.vc,
                                  self.d["k_scale"], self.d["v_scale"])
        else:
            self.kc = self.d["k_cache"].copy()
            self.vc = self.d["v_cache"].copy()

    def oracle_step(self):
        """Oracle step: write each request's new tokens (its last q_len positions), then
        attend (single-query decode, or causal multi-query for q_len > 1)."""
        wl = self.wl
        req, pos = wl.new_token_rows()
        slots = oracle.slot_mapping(wl.block_table, req, pos, wl.BS)
        ks = self.d.get("k_scale")
        vs = self.d.get("v_scale")
        oracle.kv_cache_write(self.d["k_new"], self.d["v_new"], slots, self.kc, self.vc, ks, vs)
        if wl.q_len == 1:
            out = oracle.decode_attn(self.d["q"], self.kc, self.vc, wl.block_table, wl.seq_lens,
                                     wl.scale, ks, vs)
        else:
            out = oracle.multiquery_attn(self.d["q"], wl.q_offsets(), self.kc, self.vc,
                                         wl.block_table, wl.seq_lens, wl.scale, ks, vs)
        return slots, out

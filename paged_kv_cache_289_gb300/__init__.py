"""Python binding of libpagedkv (the C ABI in include/pagedkv.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (PyTorch supplies device memory and streams);
their data pointers go straight to the C entry points of the same names.
There is no CPU fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "PkvError", "lib", "library_path", "BF16", "FP8_E4M3", "INT8", "INT4", "DEVERR_WAIT_TIMEOUT",
    "DEVERR_SEQ_CLAMPED", "DEVERR_BLOCK_RANGE", "compute_slot_mapping", "kv_cache_write",
    "decode_workspace_size", "alloc_decode_workspace", "paged_decode_attn",
    "paged_decode_attn_noalloc", "prefix_block_hash", "prefix_block_hash_resume",
    "shared_prefix_workspace_size", "paged_decode_attn_shared_prefix", "paged_decode_attn_append",
    "multiquery_workspace_size",
    "paged_multiquery_attn", "DEVERR_QLEN_CLAMPED", "kv_cache_write_rescale",
    "device_num_sms", "read_device_error", "copy_blocks", "BlockManager", "ERR_NO_BLOCKS",
    "paged_prefill_attn", "prefill_workspace_size",
]

BF16 = 0
FP8_E4M3 = 1
INT8 = 2
INT4 = 3
DEVERR_WAIT_TIMEOUT = 0x1
DEVERR_SEQ_CLAMPED = 0x2
DEVERR_BLOCK_RANGE = 0x4
DEVERR_QLEN_CLAMPED = 0x8
ERR_NO_BLOCKS = -5

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "lib", "libpagedkv.so")
_lock = threading.Lock()
_lib = None


class PkvError(RuntimeError):
    def __init__(self, fn, status):
        name = lib().pkv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status


def lib():
    """Load libpagedkv.so (built by __graft_entry__.build())."""
    global _lib
    if _lib is not None:             # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(
                    f"libpagedkv.so is not built ({library_path}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(library_path)
            p, i, i64, u64, f, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                     ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t)
            L.pkv_status_string.restype = ctypes.c_char_p
            L.pkv_status_string.argtypes = [i]
            L.pkv_version.restype = i
            L.pkv_version.argtypes = []
            L.pkv_device_num_sms.restype = i
            L.pkv_device_num_sms.argtypes = [p]
            L.pkv_compute_slot_mapping.restype = i
            L.pkv_compute_slot_mapping.argtypes = [p, i, p, p, i, i, p, p]
            L.pkv_kv_cache_write.restype = i
            L.pkv_kv_cache_write.argtypes = [p, p, p, i, i, i, i, i, i, p, p, p, p, p]
            L.pkv_decode_workspace_size.restype = sz
            L.pkv_decode_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.pkv_paged_decode_attn.restype = i
            L.pkv_paged_decode_attn.argtypes = [p, p, p, p, p, p, i, p, i, i, i, i, i, i, i, f,
                                                p, p, sz, p]
            L.pkv_multiquery_workspace_size.restype = sz
            L.pkv_multiquery_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
            L.pkv_paged_multiquery_attn.restype = i
            L.pkv_paged_multiquery_attn.argtypes = [p, p, i, p, p, p, p, p, i, p, i, i, i, i, i,
                                                    i, i, f, p, p, sz, p]
            L.pkv_rescale_workspace_size.restype = sz
            L.pkv_rescale_workspace_size.argtypes = [i, i]
            L.pkv_kv_cache_write_rescale.restype = i
            L.pkv_kv_cache_write_rescale.argtypes = [p, p, p, i, i, i, i, i, i, p, p, p, p, p, sz,
                                                     p]
            L.pkv_paged_decode_attn_noalloc.restype = i
            L.pkv_paged_decode_attn_noalloc.argtypes = [p, p, p, p, p, p, i, p, i, i, i, i, i, i,
                                                        i, f, p, p]
            L.pkv_prefix_block_hash.restype = i
            L.pkv_prefix_block_hash.argtypes = [p, p, i, i, u64, p, p, p]
            L.pkv_paged_decode_attn_append.restype = i
            L.pkv_paged_decode_attn_append.argtypes = [p, p, p, p, p, p, i, p, i, i, i, i, i, i,
                                                       f, p, p, sz, p]
            L.pkv_shared_prefix_workspace_size.restype = sz
            L.pkv_shared_prefix_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.pkv_shared_prefix_plan.restype = i
            L.pkv_shared_prefix_plan.argtypes = [i, i, i, i, i, i, i, i, p, p]
            L.pkv_paged_decode_attn_shared_prefix.restype = i
            L.pkv_paged_decode_attn_shared_prefix.argtypes = [p, p, p, p, i, p, i, i, i, i, i, i,
                                                              i, f, p, p, sz, p]
            L.pkv_prefix_block_hash_resume.restype = i
            L.pkv_prefix_block_hash_resume.argtypes = [p, p, i, i, p, p, p, p, p]
            L.pkv_prefill_workspace_size.restype = sz
            L.pkv_prefill_workspace_size.argtypes = [i, i, i, i, i, i]
            L.pkv_paged_prefill_attn.restype = i
            L.pkv_paged_prefill_attn.argtypes = [p, p, i, i, p, p, p, p, p, i, p, i, i, i, i, i,
                                                 i, i, f, p, p, sz, p, p]
            L.pkv_copy_blocks.restype = i
            L.pkv_copy_blocks.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p]
            L.pkv_bm_create.restype = i
            L.pkv_bm_create.argtypes = [i, i, p]
            L.pkv_bm_destroy.restype = None
            L.pkv_bm_destroy.argtypes = [p]
            L.pkv_bm_num_available.restype = i
            L.pkv_bm_num_available.argtypes = [p]
            L.pkv_bm_add_sequence.restype = i
            L.pkv_bm_add_sequence.argtypes = [p, i64, i64, p, i, p, p]
            L.pkv_bm_grow.restype = i
            L.pkv_bm_grow.argtypes = [p, i64, i64, p]
            L.pkv_bm_commit_block_hash.restype = i
            L.pkv_bm_commit_block_hash.argtypes = [p, i64, i, u64]
            L.pkv_bm_fork.restype = i
            L.pkv_bm_fork.argtypes = [p, i64, i64]
            L.pkv_bm_prepare_write.restype = i
            L.pkv_bm_prepare_write.argtypes = [p, i64, i, p, p]
            L.pkv_bm_free_sequence.restype = i
            L.pkv_bm_free_sequence.argtypes = [p, i64]
            L.pkv_bm_block_table.restype = i
            L.pkv_bm_block_table.argtypes = [p, i64, p, i]
            L.pkv_bm_refcount.restype = i
            L.pkv_bm_refcount.argtypes = [p, i]
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != 0:
        raise PkvError(fn, status)


def _need(t, name, dtypes, contiguous=True):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtypes and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _cache_dtype(t, head_dim):
    """Page kind of a cache tensor: int8 codes, int4 (uint8 bytes holding two codes, last
    axis head_dim / 2), E4M3 bytes (uint8, last axis head_dim) or bf16."""
    import torch
    if t.dtype == torch.int8:
        return INT8
    if t.element_size() == 1:
        return INT4 if t.shape[-1] * 2 == head_dim else FP8_E4M3
    return BF16


def device_num_sms() -> int:
    n = ctypes.c_int(0)
    _check("pkv_device_num_sms", lib().pkv_device_num_sms(ctypes.byref(n)))
    return n.value


def compute_slot_mapping(block_table, positions, block_size, req_idx=None, out=None, stream=None):
    """slot[t] = block_table[r][pos/BS]*BS + pos%BS (r = req_idx[t], or t); -1 for pos < 0."""
    import torch
    _need(block_table, "block_table", (torch.int32,))
    _need(positions, "positions", (torch.int32,))
    if req_idx is not None:
        _need(req_idx, "req_idx", (torch.int32,))
    T = positions.shape[0]
    if out is None:
        out = torch.empty(T, dtype=torch.int64, device=positions.device)
    _check("pkv_compute_slot_mapping", lib().pkv_compute_slot_mapping(
        _ptr(block_table), block_table.shape[1], _ptr(req_idx), _ptr(positions), T, block_size,
        _ptr(out), _stream(stream)))
    return out


def kv_cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None, stream=None):
    """Write new K/V rows [T, Hkv, D] (bf16) into the paged caches [NB, Hkv, BS, D]."""
    import torch
    _need(k, "k", (torch.bfloat16,))
    _need(v, "v", (torch.bfloat16,))
    _need(slot_mapping, "slot_mapping", (torch.int64,))
    _need(k_cache, "k_cache", None)
    _need(v_cache, "v_cache", None)
    T, Hkv, D = k.shape
    NB, _, BS, _ = k_cache.shape
    _check("pkv_kv_cache_write", lib().pkv_kv_cache_write(
        _ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, D, BS, NB, _cache_dtype(k_cache, D),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _stream(stream)))


def kv_cache_write_rescale(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                           workspace=None, stream=None):
    """Write rows into 8-bit caches after setting each touched (block, head)'s scale to
    amax/QMAX of the rows written to it here (k_scale / v_scale are updated)."""
    import torch
    _need(k, "k", (torch.bfloat16,))
    _need(v, "v", (torch.bfloat16,))
    _need(slot_mapping, "slot_mapping", (torch.int64,))
    _need(k_scale, "k_scale", (torch.float32,))
    _need(v_scale, "v_scale", (torch.float32,))
    T, Hkv, D = k.shape
    NB, _, BS, _ = k_cache.shape
    n = int(lib().pkv_rescale_workspace_size(NB, Hkv))
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=k.device)
    _check("pkv_kv_cache_write_rescale", lib().pkv_kv_cache_write_rescale(
        _ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, D, BS, NB, _cache_dtype(k_cache, D),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size, cache_dtype,
                          num_sms=0) -> int:
    return int(lib().pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                               block_size, cache_dtype, num_sms))


def alloc_decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, block_size, cache_dtype,
                           device="cuda"):
    """A zeroed workspace of the size the decode call needs (its first word is the
    sticky device error word)."""
    import torch
    n = decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size, cache_dtype)
    if n == 0:
        raise PkvError("pkv_decode_workspace_size", -2)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def read_device_error(workspace) -> int:
    """The device error word (PKV_DEVERR_* bits) of a decode workspace (synchronises)."""
    return int(workspace[:4].view(__import__("torch").int32).item()) & 0xFFFFFFFF


def paged_decode_attn(q, k_cache, v_cache, block_table, seq_lens, scale, out=None, k_scale=None,
                      v_scale=None, workspace=None, stream=None):
    """out[r, hq] = softmax(scale * q[r, hq] K_r^T) V_r over the paged caches."""
    import torch
    _need(q, "q", (torch.bfloat16,))
    _need(k_cache, "k_cache", None)
    _need(v_cache, "v_cache", None)
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    N, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    dt = _cache_dtype(k_cache, D)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_decode_workspace(N, Hq, Hkv, D, BS, dt, device=q.device)
    _check("pkv_paged_decode_attn", lib().pkv_paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), N, Hq, Hkv, D, BS, NB, dt, float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def multiquery_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                              cache_dtype, max_q_len, num_sms=0) -> int:
    return int(lib().pkv_multiquery_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                   block_size, cache_dtype, max_q_len, num_sms))


def paged_multiquery_attn(q, q_offsets, max_q_len, k_cache, v_cache, block_table, seq_lens,
                          scale, out=None, k_scale=None, v_scale=None, workspace=None,
                          stream=None):
    """Several new query tokens per request (speculative verify): query rows
    q_offsets[r]..q_offsets[r+1]-1 of q [T, Hq, D] are request r's newest tokens and
    attend causally.  Returns out [T, Hq, D] bf16."""
    import torch
    _need(q, "q", (torch.bfloat16,))
    _need(q_offsets, "q_offsets", (torch.int32,))
    _need(k_cache, "k_cache", None)
    _need(v_cache, "v_cache", None)
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    T, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    N = seq_lens.shape[0]
    dt = _cache_dtype(k_cache, D)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = multiquery_workspace_size(N, Hq, Hkv, D, BS, dt, max_q_len)
        if n == 0:
            raise PkvError("pkv_multiquery_workspace_size", -2)
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    _check("pkv_paged_multiquery_attn", lib().pkv_paged_multiquery_attn(
        _ptr(q), _ptr(q_offsets), int(max_q_len), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), N, Hq, Hkv, D,
        BS, NB, dt, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def paged_decode_attn_append(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, scale,
                             out=None, workspace=None, stream=None):
    """paged_decode_attn with each request's newest token (k_new, v_new [N, Hkv, D] bf16,
    position seq_len - 1) written into the cache by the decode kernel itself: the same
    output and cache contents as slot mapping + kv_cache_write + paged_decode_attn."""
    import torch
    _need(q, "q", (torch.bfloat16,))
    _need(k_new, "k_new", (torch.bfloat16,))
    _need(v_new, "v_new", (torch.bfloat16,))
    _need(k_cache, "k_cache", (torch.bfloat16,))
    _need(v_cache, "v_cache", (torch.bfloat16,))
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    N, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_decode_workspace(N, Hq, Hkv, D, BS, BF16, device=q.device)
    _check("pkv_paged_decode_attn_append", lib().pkv_paged_decode_attn_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), N, Hq, Hkv, D, BS, NB, float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def shared_prefix_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                 prefix_len, num_sms=0) -> int:
    return int(lib().pkv_shared_prefix_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                      block_size, prefix_len, num_sms))


def shared_prefix_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_blocks_per_seq, prefix_len, num_sms=0):
    """(overlapped, prefix_ctas, decode_sms) that paged_decode_attn_shared_prefix takes for
    these arguments (num_sms 0: the current device's SMs); raises PkvError for a shape
    the call would refuse."""
    ctas, sms = ctypes.c_int(0), ctypes.c_int(0)
    r = lib().pkv_shared_prefix_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                     max_blocks_per_seq, prefix_len, num_sms,
                                     ctypes.byref(ctas), ctypes.byref(sms))
    if r < 0:
        _check("pkv_shared_prefix_plan", r)
    return bool(r), ctas.value, sms.value


def paged_decode_attn_shared_prefix(q, k_cache, v_cache, block_table, seq_lens, scale,
                                    prefix_len, out=None, workspace=None, stream=None):
    """paged_decode_attn for a batch whose requests all begin with the same prefix_len
    tokens in the same blocks: the shared pages are attended once for the whole batch
    (bf16 pages)."""
    import torch
    _need(q, "q", (torch.bfloat16,))
    _need(k_cache, "k_cache", (torch.bfloat16,))
    _need(v_cache, "v_cache", (torch.bfloat16,))
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    N, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = shared_prefix_workspace_size(N, Hq, Hkv, D, BS, prefix_len)
        if n == 0:
            raise PkvError("pkv_shared_prefix_workspace_size", -2)
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    _check("pkv_paged_decode_attn_shared_prefix", lib().pkv_paged_decode_attn_shared_prefix(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), N, Hq, Hkv, D, BS, NB, int(prefix_len), float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def paged_decode_attn_noalloc(q, k_cache, v_cache, block_table, seq_lens, scale, out=None,
                              k_scale=None, v_scale=None, stream=None):
    """Same as paged_decode_attn, for callers that cannot allocate: the library's static
    device scratch replaces the workspace (calls must not overlap on the GPU)."""
    import torch
    _need(q, "q", (torch.bfloat16,))
    _need(k_cache, "k_cache", None)
    _need(v_cache, "v_cache", None)
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    N, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _check("pkv_paged_decode_attn_noalloc", lib().pkv_paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), N, Hq, Hkv, D, BS, NB, _cache_dtype(k_cache, D),
        float(scale), _ptr(out), _stream(stream)))
    return out


def prefix_block_hash(tokens, offsets, block_size, hash_offsets, num_hashes, seed=0, out=None,
                      stream=None):
    """Chained block hashes of CSR token sequences; returns an int64 tensor holding the
    uint64 bit patterns, laid out by `hash_offsets`."""
    import torch
    _need(tokens, "tokens", (torch.int32,))
    _need(offsets, "offsets", (torch.int64,))
    _need(hash_offsets, "hash_offsets", (torch.int64,))
    if out is None:
        out = torch.empty(max(int(num_hashes), 1), dtype=torch.int64, device=tokens.device)
    _check("pkv_prefix_block_hash", lib().pkv_prefix_block_hash(
        _ptr(tokens), _ptr(offsets), offsets.shape[0] - 1, block_size,
        int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out), _ptr(hash_offsets), _stream(stream)))
    return out[:num_hashes]


def prefix_block_hash_resume(tokens, offsets, block_size, prev_hashes, first_blocks,
                             hash_offsets, num_hashes, out=None, stream=None):
    """The chain continued per sequence from prev_hashes[s] = h_k after
    first_blocks[s] = k full blocks (int64 tensors holding uint64 bit patterns /
    block counts); returns the new hashes laid out by `hash_offsets`."""
    import torch
    _need(tokens, "tokens", (torch.int32,))
    _need(offsets, "offsets", (torch.int64,))
    _need(prev_hashes, "prev_hashes", (torch.int64,))
    _need(first_blocks, "first_blocks", (torch.int64,))
    _need(hash_offsets, "hash_offsets", (torch.int64,))
    if out is None:
        out = torch.empty(max(int(num_hashes), 1), dtype=torch.int64, device=tokens.device)
    _check("pkv_prefix_block_hash_resume", lib().pkv_prefix_block_hash_resume(
        _ptr(tokens), _ptr(offsets), offsets.shape[0] - 1, block_size, _ptr(prev_hashes),
        _ptr(first_blocks), _ptr(out), _ptr(hash_offsets), _stream(stream)))
    return out[:num_hashes]


def copy_blocks(k_cache, v_cache, block_mapping, k_scale=None, v_scale=None, stream=None):
    """Copy block block_mapping[i, 0] to block block_mapping[i, 1] in both caches (and their
    scales for 8-bit caches); block_mapping is an int32 CUDA tensor [pairs, 2]."""
    import torch
    _need(k_cache, "k_cache", None)
    _need(v_cache, "v_cache", None)
    _need(block_mapping, "block_mapping", (torch.int32,))
    NB, Hkv, BS, D = k_cache.shape
    _check("pkv_copy_blocks", lib().pkv_copy_blocks(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_mapping),
        block_mapping.numel() // 2, Hkv, D, BS, NB, _cache_dtype(k_cache, D), _stream(stream)))


class BlockManager:
    """Host block manager of one cache pool (the pkv_bm_* calls): block tables built on
    demand, prefix reuse by chained block hash, LRU eviction, copy-on-write.  Pure host
    code; a failed call raises PkvError (status ERR_NO_BLOCKS when the pool is full)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._h = ctypes.c_void_p()
        self.block_size = block_size
        _check("pkv_bm_create", lib().pkv_bm_create(num_blocks, block_size,
                                                     ctypes.byref(self._h)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pkv_bm_destroy(h)
            self._h = None

    def num_available(self) -> int:
        n = lib().pkv_bm_num_available(self._h)
        _check("pkv_bm_num_available", min(n, 0))
        return n

    def add_sequence(self, seq_id: int, num_tokens: int, block_hashes=()):
        """Returns (block ids, number of leading blocks reused from the cache)."""
        hs = [int(h) & 0xFFFFFFFFFFFFFFFF for h in block_hashes]
        harr = (ctypes.c_uint64 * max(len(hs), 1))(*hs)
        nb = -(-num_tokens // self.block_size) if num_tokens > 0 else 0
        ids = (ctypes.c_int32 * max(nb, 1))()
        hits = ctypes.c_int(0)
        _check("pkv_bm_add_sequence", lib().pkv_bm_add_sequence(
            self._h, seq_id, num_tokens, harr, len(hs), ids, ctypes.byref(hits)))
        return list(ids[:nb]), hits.value

    def grow(self, seq_id: int, num_tokens: int) -> int:
        nb = ctypes.c_int32(-1)
        _check("pkv_bm_grow", lib().pkv_bm_grow(self._h, seq_id, num_tokens, ctypes.byref(nb)))
        return nb.value

    def commit_block_hash(self, seq_id: int, logical_block: int, block_hash: int) -> None:
        _check("pkv_bm_commit_block_hash", lib().pkv_bm_commit_block_hash(
            self._h, seq_id, logical_block, int(block_hash) & 0xFFFFFFFFFFFFFFFF))

    def fork(self, parent_id: int, child_id: int) -> None:
        _check("pkv_bm_fork", lib().pkv_bm_fork(self._h, parent_id, child_id))

    def prepare_write(self, seq_id: int, logical_block: int):
        """(source, destination) of the copy to make before writing, or (-1, -1)."""
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        _check("pkv_bm_prepare_write", lib().pkv_bm_prepare_write(
            self._h, seq_id, logical_block, ctypes.byref(src), ctypes.byref(dst)))
        return src.value, dst.value

    def free_sequence(self, seq_id: int) -> None:
        _check("pkv_bm_free_sequence", lib().pkv_bm_free_sequence(self._h, seq_id))

    def block_table(self, seq_id: int):
        n = lib().pkv_bm_block_table(self._h, seq_id, None, 0)
        _check("pkv_bm_block_table", min(n, 0))
        ids = (ctypes.c_int32 * max(n, 1))()
        n = lib().pkv_bm_block_table(self._h, seq_id, ids, n)
        _check("pkv_bm_block_table", min(n, 0))
        return list(ids[:n])

    def refcount(self, block: int) -> int:
        n = lib().pkv_bm_refcount(self._h, block)
        _check("pkv_bm_refcount", min(n, 0))
        return n


def prefill_workspace_size(batch, max_blocks_per_seq, num_kv_heads, head_dim, block_size,
                           cache_dtype) -> int:
    return int(lib().pkv_prefill_workspace_size(batch, max_blocks_per_seq, num_kv_heads,
                                                head_dim, block_size, cache_dtype))


def paged_prefill_attn(q, q_offsets, max_q_len, k_cache, v_cache, block_table, seq_lens, scale,
                       out=None, k_scale=None, v_scale=None, workspace=None, error_word=None,
                       stream=None):
    """Causal attention of prefill chunks over the paged cache on the tensor cores: request
    r's query rows q_offsets[r] .. q_offsets[r+1]-1 are its newest tokens (already written
    to the pages); query i sees positions 0 .. seq_len - q_len + i.  Quantised pages (E4M3,
    int8, int4) take their scales and a workspace (allocated here if not given).
    `error_word` (optional int32 CUDA tensor) collects the PKV_DEVERR_* bits."""
    import torch
    _need(q, "q", (torch.bfloat16,))
    _need(q_offsets, "q_offsets", (torch.int32,))
    _need(k_cache, "k_cache", None)
    _need(v_cache, "v_cache", None)
    _need(block_table, "block_table", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    if error_word is not None:
        _need(error_word, "error_word", (torch.int32,))
    T, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    dt = _cache_dtype(k_cache, D)
    N, MB = seq_lens.shape[0], block_table.shape[1]
    if dt != BF16 and workspace is None:
        n = prefill_workspace_size(N, MB, Hkv, D, BS, dt)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _check("pkv_paged_prefill_attn", lib().pkv_paged_prefill_attn(
        _ptr(q), _ptr(q_offsets), T, int(max_q_len), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale), _ptr(v_scale), _ptr(block_table), MB, _ptr(seq_lens), N, Hq, Hkv, D,
        BS, NB, dt, float(scale), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(error_word), _stream(stream)))
    return out

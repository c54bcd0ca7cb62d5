"""CPU oracle for the paged-KV decode path (fp64, plain loops in C).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg use this package; the library and its binding never import it.
It shares no code with the CUDA path.

Sources, by page title and section:
  [P1] "深入LLM推理：从KV Cache到PD分离的Serving全景解析" -- "KV Cache：Transformer的循环状态"
       (attention formula, GQA), "PagedAttention与Cache管理" (block table, 16/32-token blocks)
  [P2] "GPU推理深度拆解：KV Cache视角" -- "KV Cache 大小与分配演进", "算子优化要点"
  [P3] "ai-infra-7" -- "KV Cache 到底有多大？" (size equation), "优化一：Prefix Cache"
       (chained block hash), "优化三：KV 传输优化" (FP8), "组合拳：一次请求的完整旅程" (write-back)

Parity status per function (what pins it, see tests/test_oracle_pins.py):
  bf16_to_double, e4m3_to_double, e4m3_from_float  -- library codecs (torch CPU) + OCP spec values
  int8_from_float                                  -- torch round-half-even + clamp, brute force
  int4_code_from_float                             -- nearest-integer brute force, the nibble layout
  kv_cache_write_rescale                           -- the generator's amax/QMAX recipe, written
                                                      independently
  kv_bytes                                         -- the printed 327,680 B/token and ~10 GB at 32K
  slot_mapping, kv_cache_write                     -- worked example + write/gather round trip
  multiquery_attn                                  -- dense causal brute force, q_len = 1 case
  multiquery_rows                                  -- dense causal brute force on every row of a
                                                      ragged batch (q_len 0 and q_len > seq_len)
  decode_attn / decode_rows / decode_row_detail    -- dense brute force, permutation invariance,
                                                      GQA == replicated MHA, closed-form cases, LSE merge
  fnv1a64, fmix64                                  -- published FNV-1a and SplitMix64 test vectors
  prefix_block_hash, hash_offsets                  -- token-exact prefix equality properties
  prefix_block_hash_resume                         -- suffix of the published-vector-pinned chain
                                                      at every cut point (the chain's definition)
  block_manager.BlockManagerModel, copy_blocks     -- hand-worked call sequences and invariants
                                                      (tests/test_block_manager.py)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_d = ctypes.c_double
_u64 = ctypes.c_uint64


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/lib/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.orc_bf16_to_double.restype = _d
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_e4m3_to_double.restype = _d
            L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_from_float.restype = ctypes.c_uint8
            L.orc_e4m3_from_float.argtypes = [ctypes.c_float]
            L.orc_int8_from_float.restype = ctypes.c_int8
            L.orc_int8_from_float.argtypes = [ctypes.c_float]
            L.orc_int4_code_from_float.restype = ctypes.c_uint8
            L.orc_int4_code_from_float.argtypes = [ctypes.c_float]
            L.orc_kv_bytes.restype = _i64
            L.orc_kv_bytes.argtypes = [_i64] * 5
            L.orc_slot_mapping.restype = None
            L.orc_slot_mapping.argtypes = [_p, _i, _p, _p, _i, _i, _p]
            L.orc_kv_cache_write.restype = None
            L.orc_kv_cache_write.argtypes = [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _p, _p]
            L.orc_kv_cache_write_rescale.restype = None
            L.orc_kv_cache_write_rescale.argtypes = [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _p,
                                                     _p]
            L.orc_decode_row.restype = None
            L.orc_decode_row.argtypes = [_p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i,
                                         _d, _i, _i, _p, _p, _p]
            L.orc_paged_decode_attn.restype = None
            L.orc_paged_decode_attn.argtypes = [_p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i,
                                                _i, _i, _i, _d, _p]
            L.orc_decode_rows.restype = None
            L.orc_decode_rows.argtypes = [_p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i,
                                          _d, _p, _i64, _p]
            L.orc_multiquery_attn.restype = None
            L.orc_multiquery_attn.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i,
                                              _i, _i, _i, _d, _p]
            L.orc_prefix_block_hash_resume.restype = None
            L.orc_prefix_block_hash_resume.argtypes = [_p, _p, _i, _i, _p, _p, _p, _p]
            L.orc_multiquery_rows.restype = None
            L.orc_multiquery_rows.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i,
                                              _i, _i, _i, _d, _p, _i64, _p]
            L.orc_num_threads.restype = _i
            L.orc_num_threads.argtypes = []
            L.orc_set_num_threads.restype = None
            L.orc_set_num_threads.argtypes = [_i]
            L.orc_fnv1a64.restype = _u64
            L.orc_fnv1a64.argtypes = [_p, _i64]
            L.orc_fmix64.restype = _u64
            L.orc_fmix64.argtypes = [_u64]
            L.orc_prefix_block_hash.restype = None
            L.orc_prefix_block_hash.argtypes = [_p, _p, _i, _i, _u64, _p, _p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(int(bits))


def e4m3_to_double(byte: int) -> float:
    return lib().orc_e4m3_to_double(int(byte))


def e4m3_from_float(x: float) -> int:
    return int(lib().orc_e4m3_from_float(float(x)))


def int4_code_from_float(x: float) -> int:
    return int(lib().orc_int4_code_from_float(float(x)))


def int8_from_float(x: float) -> int:
    return int(lib().orc_int8_from_float(float(x)))


def _kind(cache, head_dim):
    """0: bf16 bit patterns (uint16), 1: E4M3 bytes (uint8), 2: int8, 3: int4 (uint8
    bytes holding two offset-binary codes each, so the last axis is head_dim / 2)."""
    if cache.dtype == np.uint16:
        return 0
    if cache.dtype == np.uint8:
        return 3 if cache.shape[-1] * 2 == head_dim else 1
    if cache.dtype == np.int8:
        return 2
    raise TypeError(f"cache dtype {cache.dtype}")


def kv_bytes(L: int, Hkv: int, d: int, S: int, b: int) -> int:
    return int(lib().orc_kv_bytes(L, Hkv, d, S, b))


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (results do not change)."""
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- steps
def slot_mapping(block_table, req_idx, positions, block_size):
    bt = _c(block_table, np.int32)
    ri = _c(req_idx, np.int32)
    pos = _c(positions, np.int32)
    out = np.empty(pos.shape[0], dtype=np.int64)
    lib().orc_slot_mapping(_ptr(bt), bt.shape[1], _ptr(ri), _ptr(pos), pos.shape[0],
                           block_size, _ptr(out))
    return out


def kv_cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None):
    """In-place write into numpy caches (uint16 bf16 bits, uint8 E4M3 bytes or int8).

    k, v: uint16 [T, Hkv, D] bf16 bit patterns.  Caches [NB, Hkv, BS, D]."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int64)
    T, Hkv, D = k.shape
    kind = _kind(k_cache, D)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    ks = _c(k_scale, np.float32) if kind else None
    vs = _c(v_scale, np.float32) if kind else None
    lib().orc_kv_cache_write(_ptr(k), _ptr(v), _ptr(sm), T, Hkv, D, k_cache.shape[2], kind,
                             _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs))


def kv_cache_write_rescale(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    """In-place: set the scale of every (block, head) written by this call to
    amax/QMAX of its rows here, then write the rows (8-bit caches only)."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int64)
    T, Hkv, D = k.shape
    kind = _kind(k_cache, D)
    assert kind in (1, 2, 3) and k_scale.dtype == np.float32 and k_scale.flags.c_contiguous
    lib().orc_kv_cache_write_rescale(_ptr(k), _ptr(v), _ptr(sm), T, Hkv, D, k_cache.shape[2], kind,
                                     _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale))


def _decode_args(q, k_cache, v_cache, block_table, seq_lens, k_scale, v_scale):
    q = _c(q, np.uint16)
    kind = _kind(k_cache, q.shape[-1])
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    ks = _c(k_scale, np.float32) if kind else None
    vs = _c(v_scale, np.float32) if kind else None
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    return q, kc, vc, ks, vs, bt, sl, kind


def decode_attn(q, k_cache, v_cache, block_table, seq_lens, scale, k_scale=None, v_scale=None):
    """fp64 output [N, Hq, D] for every (request, query head)."""
    q, kc, vc, ks, vs, bt, sl, kind = _decode_args(q, k_cache, v_cache, block_table, seq_lens,
                                                  k_scale, v_scale)
    N, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    out = np.empty((N, Hq, D), dtype=np.float64)
    lib().orc_paged_decode_attn(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
                                bt.shape[1], _ptr(sl), N, Hq, Hkv, D, BS, int(kind),
                                float(scale), _ptr(out))
    return out


def multiquery_attn(q, q_offsets, k_cache, v_cache, block_table, seq_lens, scale, k_scale=None,
                    v_scale=None):
    """fp64 output [T, Hq, D]: query rows q_offsets[r]..q_offsets[r+1]-1 of request r are
    its newest tokens and attend causally (position seq_len - q_len + i and before)."""
    q, kc, vc, ks, vs, bt, sl, kind = _decode_args(q, k_cache, v_cache, block_table, seq_lens,
                                                  k_scale, v_scale)
    qo = _c(q_offsets, np.int32)
    T, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    out = np.empty((T, Hq, D), dtype=np.float64)
    lib().orc_multiquery_attn(_ptr(q), _ptr(qo), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
                              bt.shape[1], _ptr(sl), qo.shape[0] - 1, Hq, Hkv, D, BS, int(kind),
                              float(scale), _ptr(out))
    return out


def multiquery_rows(q, q_offsets, k_cache, v_cache, block_table, seq_lens, scale, rows,
                    k_scale=None, v_scale=None):
    """fp64 rows of multiquery_attn for selected rows (row = query token * Hq + hq)."""
    q, kc, vc, ks, vs, bt, sl, kind = _decode_args(q, k_cache, v_cache, block_table, seq_lens,
                                                  k_scale, v_scale)
    qo = _c(q_offsets, np.int32)
    T, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    rows = _c(rows, np.int64)
    out = np.empty((rows.shape[0], D), dtype=np.float64)
    lib().orc_multiquery_rows(_ptr(q), _ptr(qo), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                              _ptr(bt), bt.shape[1], _ptr(sl), qo.shape[0] - 1, Hq, Hkv, D, BS,
                              int(kind), float(scale), _ptr(rows), rows.shape[0], _ptr(out))
    return out


def decode_rows(q, k_cache, v_cache, block_table, seq_lens, scale, rows, k_scale=None,
                v_scale=None):
    """fp64 output [len(rows), D] for selected rows (row = r * Hq + hq)."""
    q, kc, vc, ks, vs, bt, sl, kind = _decode_args(q, k_cache, v_cache, block_table, seq_lens,
                                                  k_scale, v_scale)
    N, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    rows = _c(rows, np.int64)
    out = np.empty((rows.shape[0], D), dtype=np.float64)
    lib().orc_decode_rows(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
                          bt.shape[1], _ptr(sl), Hq, Hkv, D, BS, int(kind), float(scale),
                          _ptr(rows), rows.shape[0], _ptr(out))
    return out


def decode_row_detail(q, k_cache, v_cache, block_table, seq_lens, scale, r, hq, k_scale=None,
                      v_scale=None):
    """(o [D], p [seq_len], lse) for one (request, query head)."""
    q, kc, vc, ks, vs, bt, sl, kind = _decode_args(q, k_cache, v_cache, block_table, seq_lens,
                                                  k_scale, v_scale)
    N, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    o = np.empty(D, dtype=np.float64)
    p = np.empty(max(int(sl[r]), 1), dtype=np.float64)
    lse = ctypes.c_double(0.0)
    lib().orc_decode_row(_ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1],
                         _ptr(sl), Hq, Hkv, D, BS, int(kind), float(scale), int(r), int(hq),
                         _ptr(o), _ptr(p), ctypes.byref(lse))
    return o, p[: max(int(sl[r]), 0)], lse.value


def fnv1a64(data: bytes) -> int:
    buf = np.frombuffer(bytes(data), dtype=np.uint8) if len(data) else np.zeros(1, np.uint8)
    return int(lib().orc_fnv1a64(_ptr(buf), len(data)))


def fmix64(x: int) -> int:
    return int(lib().orc_fmix64(int(x) & 0xFFFFFFFFFFFFFFFF))


def hash_offsets(offsets, block_size):
    lens = np.diff(np.asarray(offsets, dtype=np.int64))
    ho = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    np.cumsum(lens // block_size, out=ho[1:])
    return ho


def prefix_block_hash(tokens, offsets, block_size, seed):
    tok = _c(tokens, np.int32)
    off = _c(offsets, np.int64)
    ho = hash_offsets(off, block_size)
    out = np.zeros(int(ho[-1]), dtype=np.uint64)
    if tok.size == 0:
        tok = np.zeros(1, np.int32)
    lib().orc_prefix_block_hash(_ptr(tok), _ptr(off), off.shape[0] - 1, block_size,
                                int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out) if out.size else None,
                                _ptr(ho))
    return out, ho


def prefix_block_hash_resume(tokens, offsets, block_size, prev_hashes, first_blocks,
                             hash_offsets=None):
    """The chain continued from h_k per sequence: prev_hashes[s] = h_{k_s},
    first_blocks[s] = k_s full blocks already hashed.  Returns (hashes, hash_offsets)
    with max(0, floor(L_s / B) - k_s) hashes per sequence unless hash_offsets gives
    the room per sequence."""
    tok = _c(tokens, np.int32)
    off = _c(offsets, np.int64)
    prev = _c(np.asarray(prev_hashes, dtype=np.uint64), np.uint64)
    first = _c(first_blocks, np.int64)
    if hash_offsets is None:
        full = np.diff(off) // block_size
        n = np.maximum(full - np.maximum(first, 0), 0)
        ho = np.zeros(n.shape[0] + 1, dtype=np.int64)
        np.cumsum(n, out=ho[1:])
    else:
        ho = _c(hash_offsets, np.int64)
    out = np.zeros(max(int(ho[-1]), 1), dtype=np.uint64)
    if tok.size == 0:
        tok = np.zeros(1, np.int32)
    lib().orc_prefix_block_hash_resume(_ptr(tok), _ptr(off), off.shape[0] - 1, block_size,
                                       _ptr(prev), _ptr(first), _ptr(out), _ptr(ho))
    return out[:int(ho[-1])], ho

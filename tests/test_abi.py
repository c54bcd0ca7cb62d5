"""The C ABI library builds, loads and exports every declared entry point; host-side
argument validation rejects bad calls before any CUDA work (runs without a GPU)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import paged_kv_cache_289_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return pkv.lib()


def _declared():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]*?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("pkv_compute_slot_mapping", "pkv_kv_cache_write", "pkv_paged_decode_attn",
                 "pkv_prefix_block_hash", "pkv_decode_workspace_size", "pkv_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings_and_version(L):
    assert L.pkv_status_string(0) == b"PKV_OK"
    assert L.pkv_status_string(-2) == b"PKV_ERR_UNSUPPORTED"
    assert L.pkv_status_string(12345) == b"PKV_UNKNOWN_STATUS"
    assert L.pkv_version() >= 10000


def test_workspace_size_is_host_arithmetic(L):
    sz = L.pkv_decode_workspace_size(64, 64, 8, 128, 16, 0, 152)
    assert sz > 0 and sz % 16 == 0
    # more requests or more SMs never need less
    assert L.pkv_decode_workspace_size(128, 64, 8, 128, 16, 0, 152) > sz
    assert L.pkv_decode_workspace_size(64, 64, 8, 128, 16, 0, 300) > sz
    # unsupported shapes report 0
    assert L.pkv_decode_workspace_size(64, 64, 8, 96, 16, 0, 152) == 0     # head_dim
    assert L.pkv_decode_workspace_size(64, 64, 8, 128, 8, 0, 152) == 0     # block size
    assert L.pkv_decode_workspace_size(64, 72, 8, 128, 16, 0, 152) == 0    # G = 9
    assert L.pkv_decode_workspace_size(64, 60, 8, 128, 16, 0, 152) == 0    # Hq % Hkv
    assert L.pkv_decode_workspace_size(64, 64, 8, 64, 16, 1, 152) == 0     # fp8 d=64
    assert L.pkv_decode_workspace_size(64, 64, 8, 128, 16, 7, 152) == 0    # dtype


def _decode(L, **kw):
    a = dict(q=16, k=16, v=16, ks=None, vs=None, bt=16, MB=4, sl=16, N=2, Hq=8, Hkv=2, D=128,
             BS=16, NB=8, dt=0, scale=0.1, out=16, ws=16, wsb=1 << 20, st=None)
    a.update(kw)
    return L.pkv_paged_decode_attn(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["MB"],
                                   a["sl"], a["N"], a["Hq"], a["Hkv"], a["D"], a["BS"], a["NB"],
                                   a["dt"], a["scale"], a["out"], a["ws"], a["wsb"], a["st"])


def test_decode_rejects_bad_arguments_without_launching(L):
    # (fake, never dereferenced pointer values: every call below fails validation first)
    assert _decode(L, D=96) == -2
    assert _decode(L, BS=8) == -2
    assert _decode(L, Hq=9) == -2
    assert _decode(L, Hq=72, Hkv=8) == -2
    assert _decode(L, dt=7) == -2
    assert _decode(L, dt=1, D=64) == -2
    assert _decode(L, N=-1) == -1
    assert _decode(L, MB=0) == -1
    assert _decode(L, NB=0) == -1
    assert _decode(L, q=None) == -1
    assert _decode(L, k=None) == -1
    assert _decode(L, sl=None) == -1
    assert _decode(L, dt=1) == -1            # fp8 without scales
    assert _decode(L, q=24) == -1            # misaligned
    assert _decode(L, k=8) == -1
    assert _decode(L, N=0) == 0              # empty batch: nothing to do
    assert _decode(L, N=100000) == -2        # beyond the batch limit


def test_write_slot_hash_reject_bad_arguments(L):
    w = L.pkv_kv_cache_write
    assert w(16, 16, 16, -1, 2, 128, 16, 8, 0, 16, 16, None, None, None) == -1
    assert w(16, 16, 16, 4, 2, 12, 16, 8, 0, 16, 16, None, None, None) == -2
    assert w(16, 16, 16, 4, 2, 128, 16, 8, 5, 16, 16, None, None, None) == -2
    assert w(16, 16, 16, 4, 2, 128, 16, 8, 1, 16, 16, None, None, None) == -1   # fp8, no scales
    assert w(None, 16, 16, 4, 2, 128, 16, 8, 0, 16, 16, None, None, None) == -1
    assert w(24, 16, 16, 4, 2, 128, 16, 8, 0, 16, 16, None, None, None) == -1   # misaligned
    assert w(16, 16, 16, 0, 2, 128, 16, 8, 0, 16, 16, None, None, None) == 0    # no tokens
    s = L.pkv_compute_slot_mapping
    assert s(16, 4, None, 16, -1, 16, 16, None) == -1
    assert s(16, 0, None, 16, 4, 16, 16, None) == -1
    assert s(None, 4, None, 16, 4, 16, 16, None) == -1
    assert s(16, 4, None, 16, 0, 16, 16, None) == 0
    h = L.pkv_prefix_block_hash
    assert h(16, 16, 2, 0, 0, 16, 16, None) == -1
    assert h(16, 16, 2, 2000, 0, 16, 16, None) == -1
    assert h(None, 16, 2, 16, 0, 16, 16, None) == -1
    assert h(16, 16, 0, 16, 0, 16, 16, None) == 0
    r = L.pkv_prefix_block_hash_resume
    assert r(16, 16, 2, 0, 16, 16, 16, 16, None) == -1                  # block size
    assert r(16, 16, -1, 16, 16, 16, 16, 16, None) == -1                # num_seqs
    assert r(16, 16, 2, 16, None, 16, 16, 16, None) == -1               # no prev hashes
    assert r(16, 16, 2, 16, 16, None, 16, 16, None) == -1               # no first blocks
    assert r(16, 16, 2, 16, 16, 16, 16, None, None) == -1               # no hash offsets
    assert r(16, 16, 0, 16, 16, 16, 16, 16, None) == 0                  # nothing to do


def test_shared_prefix_rejects_bad_arguments_without_launching(L):
    f = L.pkv_paged_decode_attn_shared_prefix
    # (fake pointers; every call fails a host check before any CUDA call)
    args = [16, 16, 16, 16, 8, 16, 4, 32, 8, 128, 16, 64, 32, 0.1, 16, 16, 1 << 30, None]

    def call(**kw):
        a = list(args)
        for k, v in kw.items():
            a[{"MB": 4, "N": 6, "Hq": 7, "D": 9, "BS": 10, "prefix": 12, "scale": 13}[k]] = v
        return f(*a)
    assert call(prefix=24) == -1               # not a whole number of blocks
    assert call(prefix=16 * 9) == -1           # past the block table
    assert call(prefix=-16) == -1
    assert call(N=-1) == -1
    assert call(scale=0.0) == -1
    assert call(D=96) == -2
    assert call(Hq=24) == -2                   # G = 3: the prefix pass takes 1, 2, 4, 8
    assert call(BS=8) == -2
    assert L.pkv_shared_prefix_workspace_size(128, 32, 8, 128, 16, 4096, 152) > \
        L.pkv_decode_workspace_size(128, 32, 8, 128, 16, 0, 152)
    assert L.pkv_shared_prefix_workspace_size(128, 32, 8, 96, 16, 4096, 152) == 0


def test_shared_prefix_plan_query(L):
    """The plan query (host only) for the overlapped and the sequential shared-prefix
    plans: the overlapped one keeps the prefix pass to a third of the SMs and sizes the
    tail decode to the rest."""
    import ctypes
    f = L.pkv_shared_prefix_plan
    f.restype = ctypes.c_int
    ctas, sms = ctypes.c_int(-7), ctypes.c_int(-7)

    def plan(*a):
        r = f(*a, ctypes.byref(ctas), ctypes.byref(sms))
        return r, ctas.value, sms.value
    # 40 requests x 4 query heads per KV head = 2 tiles of 128 rows, x 8 KV heads; tails of
    # up to (128 x 16 - 256) tokens: overlapped, 16 prefix CTAs, the decode on 136 SMs
    assert plan(40, 32, 8, 128, 16, 128, 256, 152) == (1, 16, 136)
    # 128 requests over a 4096-token prefix: 4 tiles x 8 heads, split into 4 chunks of
    # 1024 tokens to fill the SMs, then the tails on every SM
    assert plan(128, 32, 8, 128, 16, 512, 4096, 152) == (0, 128, 152)
    # a third of 40 SMs is under 16 prefix CTAs: sequential
    assert plan(40, 32, 8, 128, 16, 128, 256, 40)[0] == 0
    for a in [(40, 32, 8, 128, 16, 128, 256, 152), (64, 16, 8, 128, 32, 64, 512, 152),
              (5, 64, 8, 128, 32, 15, 160, 152)]:
        r, c, s = plan(*a)
        assert r == 1 and 3 * c <= a[-1] and s == a[-1] - c
    assert f(40, 32, 8, 128, 16, 128, 24, 152, None, None) == -1   # not whole blocks
    assert f(40, 32, 8, 128, 16, 8, 256, 152, None, None) == -1    # past the block table
    assert f(40, 24, 8, 128, 16, 128, 256, 152, None, None) == -2  # G = 3
    assert f(40, 32, 8, 96, 16, 128, 256, 152, None, None) == -2   # head_dim


def test_append_rejects_bad_arguments_without_launching(L):
    f = L.pkv_paged_decode_attn_append
    # q, k_new, v_new, k_cache, v_cache, bt, MB, sl, N, Hq, Hkv, D, BS, NB, scale, out, ws,
    # ws_bytes, stream (fake pointers: each call fails a host check first)
    a = [16, 16, 16, 16, 16, 16, 4, 16, 2, 8, 2, 128, 16, 8, 0.1, 16, 16, 1 << 20, None]

    def call(i, v):
        b = list(a)
        b[i] = v
        return f(*b)
    assert call(8, -1) == -1          # batch
    assert call(6, 0) == -1           # max blocks per sequence
    assert call(11, 96) == -2         # head_dim
    assert call(9, 9) == -2           # Hq % Hkv
    assert call(1, None) == -1        # no k_new
    assert call(2, 8) == -1           # v_new misaligned
    assert call(8, 0) == 0            # empty batch


def test_binding_raises_when_library_missing(monkeypatch):
    monkeypatch.setattr(pkv, "_lib", None)
    monkeypatch.setattr(pkv, "library_path", "/nonexistent/libpagedkv.so")
    with pytest.raises(RuntimeError, match="not built"):
        pkv.lib()

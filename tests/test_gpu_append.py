"""Decode with the step's cache write folded in (pkv_paged_decode_attn_append).

For every request the newest token's K/V rows go into their slot and the query attends to
all cached tokens including it.  The call must leave the cache byte for byte as the
oracle's slot mapping + write leaves it, give the same output bits as the separate path on
the GPU (slot mapping, write, decode), and match the fp64 oracle within the attention
tolerance."""
import numpy as np
import pytest

import paged_kv_cache_289_gb300 as pkv
from paged_kv_cache_289_gb300 import workloads as W
from helpers import HostCase, bf16_dev, compare, dev_bits, out_to_f64, to_dev, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch_mod()


def _check(wl):
    torch = torch_mod()
    case = HostCase(wl)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    q = bf16_dev(case.d["q"])
    kn, vn = bf16_dev(case.d["k_new"]), bf16_dev(case.d["v_new"])
    # separate path: slot mapping, write, decode
    kc1, vc1 = bf16_dev(case.kc), bf16_dev(case.vc)
    slots = pkv.compute_slot_mapping(bt, to_dev(wl.new_token_positions()), wl.BS)
    pkv.kv_cache_write(kn, vn, slots, kc1, vc1)
    ws1 = pkv.alloc_decode_workspace(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, pkv.BF16)
    out1 = pkv.paged_decode_attn(q, kc1, vc1, bt, sl, wl.scale, workspace=ws1)
    # append: one call
    kc2, vc2 = bf16_dev(case.kc), bf16_dev(case.vc)
    ws2 = pkv.alloc_decode_workspace(wl.N, wl.Hq, wl.Hkv, wl.D, wl.BS, pkv.BF16)
    out2 = pkv.paged_decode_attn_append(q, kn, vn, kc2, vc2, bt, sl, wl.scale, workspace=ws2)
    torch.cuda.synchronize()
    _, out_o = case.oracle_step()          # the oracle's write then attention
    assert np.array_equal(dev_bits(kc2), case.kc) and np.array_equal(dev_bits(vc2), case.vc)
    assert np.array_equal(dev_bits(kc2), dev_bits(kc1))
    assert torch.equal(out2.view(torch.int16), out1.view(torch.int16))
    compare(out_to_f64(out2), out_o, False)
    assert pkv.read_device_error(ws2) == 0


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_append_equals_write_then_decode(cfg):
    _check(W.make(cfg, small=True))


@pytest.mark.parametrize("G,D,BS", [(1, 64, 16), (3, 128, 32), (8, 128, 16), (4, 64, 32)])
def test_append_at_every_position_in_a_block(G, D, BS):
    """The newest token as the first, a middle and the last row of its block, in the
    first and the second 16-token tile of a 32-token block, and a one-token request."""
    lens = [1, BS - 1, BS, BS + 1, 2 * BS, 2 * BS + 1, 17, 33, 16 * 7 + 5, 300]
    wl = W.custom(len(lens), G * 2, 2, D, BS, lens, seed=G * 10 + BS)
    _check(wl)


def test_append_skips_empty_requests():
    torch = torch_mod()
    lens = [0, 7, 0, 40]
    wl = W.custom(len(lens), 8, 2, 128, 16, lens, seed=19)
    wl.block_table[wl.seq_lens == 0] = 0
    case = HostCase(wl)
    kc, vc = bf16_dev(case.kc), bf16_dev(case.vc)
    out = pkv.paged_decode_attn_append(bf16_dev(case.d["q"]), bf16_dev(case.d["k_new"]),
                                       bf16_dev(case.d["v_new"]), kc, vc,
                                       to_dev(wl.block_table), to_dev(wl.seq_lens), wl.scale)
    torch.cuda.synchronize()
    got = out_to_f64(out)
    assert np.all(got[wl.seq_lens == 0] == 0)
    # only the two non-empty requests' newest rows changed
    changed = np.argwhere(np.any(dev_bits(kc) != case.kc, axis=-1))
    rows = {(int(b), int(t)) for b, _, t in changed}
    expect = set()
    for r in (1, 3):
        p = int(wl.seq_lens[r]) - 1
        expect.add((int(wl.block_table[r, p // wl.BS]), p % wl.BS))
    assert rows <= expect

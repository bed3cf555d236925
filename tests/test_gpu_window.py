"""Kamera's three window operations (Kamera §3), composed from the library's
calls and checked against the fp64 oracle on the GPU:

* reorder: the same canonical chunks relocated in two orders under ONE orbit
  patch kept per canonical chunk, addressed through the patch maps (no factor
  copies);
* sliding-window survival: evicting the oldest chunks shifts the survivors by
  an exact re-rotation R(δ) and no patch -- a splice of the evicted prefix,
  by block-table remapping when the chunks are whole blocks;
* recall: an evicted chunk re-hydrated from the canonical store with its
  stored patch at the window's end.
"""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, SHAPES, check_exact, check_pool, to_dev

pytestmark = pytest.mark.gpu

L = 3
B = 64


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _store(shape, n_canon, chunk_len, m, seed):
    """A canonical store: n_canon chunks of chunk_len tokens in a registry pool
    (contiguous, block-aligned), plus per-chunk patch factors."""
    cd, H, d, base = SHAPES[shape]
    reg = DevPool(shape, L, n_canon * chunk_len + B, seed)
    widths = (cd, H * d)
    u = [synth.f32_normal((L, n_canon * chunk_len, m), seed + 1 + ch, std=0.03) for ch in range(2)]
    v = [synth.f32_normal((L, n_canon, widths[ch], m), seed + 3 + ch, std=0.03) for ch in range(2)]
    return reg, u, v


def _relocate_from_store(orc, shape, reg, u, v, m, order, chunk_len, dst, bt, pos0, deltas, seed):
    """Relocate canonical chunks `order` back to back from position pos0 of
    request 0, with the stored patch addressed through the maps; the oracle
    does the same from its own mirrors.  Returns the device status."""
    C = len(order)
    tok_off = np.arange(C + 1, dtype=np.int32) * chunk_len
    src_slots = np.concatenate([np.arange(k * chunk_len, (k + 1) * chunk_len) for k in order]
                               ).astype(np.int32)
    chunk_req = np.zeros(C, np.int32)
    dst_pos = (pos0 + np.arange(C) * chunk_len).astype(np.int32)
    delta = np.asarray(deltas, np.int32)
    umap = (np.asarray(order, np.int64) * chunk_len)
    vmap = np.asarray(order, np.int32)
    dev = [to_dev(x) for x in (tok_off, src_slots, chunk_req, dst_pos, delta)]
    pd = kv.patch_desc(m, [x.cuda() for x in u], [x.cuda() for x in v], to_dev(umap),
                       to_dev(vmap))
    ws = kv.workspace(dst.desc, C * chunk_len, C)
    kv.kv_relocate(reg.desc, dst.desc, C, C * chunk_len, *dev, bt, 1, bt.shape[1], pd, ws)
    st = kv.kv_get_device_status(ws)
    assert orc.relocate(reg.orc, dst.orc, tok_off, src_slots, chunk_req, dst_pos, delta,
                        bt.cpu().numpy(), O.Patch(m, [x.numpy() for x in u],
                                                  [x.numpy() for x in v], umap, vmap)) == O.OK
    return st


@pytest.mark.parametrize("shape,m", [("mla", 8), ("gqa", 16), ("gqa", 32)])
def test_reorder_under_one_orbit_patch(orc, shape, m):
    # one stored patch per canonical chunk serves every order of the set
    chunk_len, n_canon = 192, 6
    reg, u, v = _store(shape, n_canon, chunk_len, m, 600 + m)
    for k, order in enumerate(([4, 0, 5, 2], [2, 5, 0, 4, 1])):
        ss = synth.splice_seqs(610 + k, [0], 24)
        dst = DevPool(shape, L, ss.num_slots, 620 + k)
        bt = to_dev(ss.block_tables)
        # chunk j lands at 70 + j*chunk_len: δ = target - source position
        deltas = [70 + j * chunk_len - order[j] * chunk_len for j in range(len(order))]
        assert _relocate_from_store(orc, shape, reg, u, v, m, order, chunk_len, dst, bt, 70,
                                    deltas, 630 + k) == kv.KV_OK
        check_pool(dst, f"reorder {order} ({shape}, rank {m})", copy_exact=False)


@pytest.mark.parametrize("mode", ["remap", "amortize"])
def test_window_slide_survivors_are_only_rerotated(orc, mode):
    # a window of 6 chunks of 128 tokens (whole blocks); the oldest 2 are
    # evicted: the survivors move up by 256 positions, rotated by R(-256)
    lens = [6 * 128]
    ss = synth.splice_seqs(640, lens, 16)
    dp = DevPool("gqa", L, ss.num_slots, 641)
    bt = to_dev(ss.block_tables)
    glens = torch.tensor(lens, dtype=torch.int32)
    ws = kv.workspace(dp.desc, lens[0], 1)
    mode_id = kv.KV_AMORTIZE_REMAP if mode == "remap" else kv.KV_AMORTIZE
    kv.kv_splice(dp.desc, 1, bt, 16, glens, torch.tensor([0], dtype=torch.int32),
                 torch.tensor([256], dtype=torch.int32), torch.tensor([0], dtype=torch.int32),
                 None, None, mode_id, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice(dp.orc, ss.block_tables, olens, [0], [256], [0], None, None) == O.OK
    assert glens.tolist() == olens.tolist() == [512]
    new_bt = bt.cpu().numpy()
    if mode == "remap":
        assert not np.array_equal(new_bt[0], ss.block_tables[0])
    slots = lambda row: np.array([int(row[p // B]) * B + p % B for p in range(512)])
    gc, gr = dp.gpu_bits()
    check_exact(gc[:, slots(new_bt[0])], dp.orc.copy[:, slots(ss.block_tables[0])], "V")
    check_exact(gr[:, slots(new_bt[0])], dp.orc.rot[:, slots(ss.block_tables[0])], "K")


def test_recall_evicted_chunk_with_its_stored_patch(orc):
    # after a slide, an evicted chunk comes back from the canonical store at
    # the window's end, with the patch stored for it (no re-encoding)
    chunk_len, n_canon, m = 128, 5, 16
    reg, u, v = _store("gqa", n_canon, chunk_len, m, 650)
    ss = synth.splice_seqs(651, [0], 20)
    win = DevPool("gqa", L, ss.num_slots, 652)
    bt = to_dev(ss.block_tables)
    # window holds chunks 1, 2, 3 at 0..384; chunk 0 was evicted; recall it at 384
    assert _relocate_from_store(orc, "gqa", reg, u, v, m, [1, 2, 3], chunk_len, win, bt, 0,
                                [-chunk_len, -chunk_len, -chunk_len], 653) == kv.KV_OK
    assert _relocate_from_store(orc, "gqa", reg, u, v, m, [0], chunk_len, win, bt, 384,
                                [384], 654) == kv.KV_OK
    check_pool(win, "window after recall", copy_exact=False)


def test_standalone_patch_through_the_maps(orc):
    # kv_patch reads stored factors through the same maps
    chunk_len, n_canon, m = 96, 4, 12
    _, u, v = _store("mla", n_canon, chunk_len, m, 660)
    ss = synth.splice_seqs(661, [0], 12)
    dp = DevPool("mla", L, ss.num_slots, 662)
    bt = to_dev(ss.block_tables)
    order = [3, 1, 2]
    C = len(order)
    tok_off = np.arange(C + 1, dtype=np.int32) * chunk_len
    chunk_req = np.zeros(C, np.int32)
    dst_pos = (5 + np.arange(C) * chunk_len).astype(np.int32)
    umap = np.asarray(order, np.int64) * chunk_len
    vmap = np.asarray(order, np.int32)
    pd = kv.patch_desc(m, [x.cuda() for x in u], [x.cuda() for x in v], to_dev(umap),
                       to_dev(vmap))
    ws = kv.workspace(dp.desc, C * chunk_len, C)
    kv.kv_patch(dp.desc, C, C * chunk_len, to_dev(tok_off), to_dev(chunk_req), to_dev(dst_pos),
                bt, 1, bt.shape[1], pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert orc.patch_apply(dp.orc, tok_off, chunk_req, dst_pos, ss.block_tables,
                           O.Patch(m, [x.numpy() for x in u], [x.numpy() for x in v], umap,
                                   vmap)) == O.OK
    check_pool(dp, "patch through maps", copy_exact=False)

"""Pools whose rotary pairs are interleaved, (x[2j], x[2j+1]) with the same
θ_j (pair_convention = 1): relocation (plain and patched), the standalone
patch, the splice, the composed splice and the remapped splice against the
fp64 oracle's interleaved mode, through the C ABI, for MLA and GQA rows."""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, SHAPES, check_exact, check_pool, to_dev

pytestmark = pytest.mark.gpu

L = 3
IL = 1


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _reloc_case(shape, seed):
    wl = synth.relocate_workload(seed, num_reqs=3, chunks_per_req=4, len_lo=1, len_hi=140,
                                 delta_lo=-30000, delta_hi=30000, n_pool_chunks=5, base_hi=150)
    src = DevPool(shape, L, wl.src_slots_total, seed, pair_convention=IL)
    dst = DevPool(shape, L, wl.dst_slots_total, seed + 10, pair_convention=IL)
    dev = [to_dev(getattr(wl, k)) for k in
           ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta", "block_tables")]
    return wl, src, dst, dev


@pytest.mark.parametrize("shape", ["mla", "gqa"])
@pytest.mark.parametrize("m", [0, 8])
def test_relocate(orc, shape, m):
    wl, src, dst, dev = _reloc_case(shape, 800 + m + len(shape))
    pd = patch = None
    if m:
        cd, H, d, _ = SHAPES[shape]
        widths = (cd, H * d)
        us = [synth.f32_normal((L, wl.total_tokens, m), 810 + i, std=0.02) for i in range(2)]
        vs = [synth.f32_normal((L, wl.num_chunks, widths[i], m), 812 + i, std=0.02)
              for i in range(2)]
        pd = kv.patch_desc(m, [x.cuda() for x in us], [x.cuda() for x in vs])
        patch = O.Patch(m, [x.numpy() for x in us], [x.numpy() for x in vs])
    ws = kv.workspace(dst.desc, wl.total_tokens, wl.num_chunks)
    kv.kv_relocate(src.desc, dst.desc, wl.num_chunks, wl.total_tokens, *dev,
                   wl.block_tables.shape[0], wl.block_tables.shape[1], pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert orc.relocate(src.orc, dst.orc, wl.tok_off, wl.src_slots, wl.chunk_req,
                        wl.chunk_dst_pos, wl.delta, wl.block_tables, patch) == O.OK
    stats = check_pool(dst, f"interleaved relocate {shape} rank {m}", copy_exact=m == 0)
    if m == 0:
        assert stats["exact"] >= stats["values"] - max(3, stats["values"] // 100000), stats


def test_mixed_conventions_are_rejected():
    wl, src, _, dev = _reloc_case("mla", 820)
    dst = DevPool("mla", L, wl.dst_slots_total, 821)          # rotate-half
    ws = kv.workspace(dst.desc, wl.total_tokens, wl.num_chunks)
    st = kv.kv_relocate(src.desc, dst.desc, wl.num_chunks, wl.total_tokens, *dev,
                        wl.block_tables.shape[0], wl.block_tables.shape[1], None, ws,
                        check=False)
    assert st == kv.KV_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_splices(orc, shape):
    lens = [200, 900, 1500]
    ss = synth.splice_seqs(830, lens, 40, spare_blocks=2)
    dp = DevPool(shape, L, ss.num_slots, 831, pair_convention=IL)
    bt = to_dev(ss.block_tables)
    olens = np.array(lens, np.int32)
    glens = torch.tensor(lens, dtype=torch.int32)
    # one plain directive per sequence, then a composed pair, then a remapped one
    d = synth.random_directives(832, olens, 0, 400, 0, 300)
    tot = int(d.stub_len.sum())
    sc = synth.bf16_normal((L, tot, dp.cd), 833)
    sr = synth.bf16_normal((L, tot, dp.H * dp.d), 834)
    ws = kv.workspace(dp.desc, 4000, 3)
    kv.kv_splice(dp.desc, 3, bt, 40, glens,
                 *[torch.from_numpy(x.copy()) for x in (d.s_start, d.s_end, d.stub_len)],
                 sc.cuda(), sr.cuda(), kv.KV_AMORTIZE, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert orc.splice(dp.orc, ss.block_tables, olens, d.s_start, d.s_end, d.stub_len,
                      synth.bits(sc).copy(), synth.bits(sr).copy()) == O.OK
    check_pool(dp, f"interleaved splice {shape}")
    cur = olens.copy()
    s0, s1, nr = [], [], []
    for r in range(2):
        dd = synth.random_directives(835 + r, cur, 0, 300, 0, 100)
        s0.append(dd.s_start)
        s1.append(dd.s_end)
        nr.append(dd.stub_len)
        cur = cur + dd.stub_len - (dd.s_end - dd.s_start)
    s0, s1, nr = (np.ascontiguousarray(np.stack(x)) for x in (s0, s1, nr))
    tot = int(nr.sum())
    sc = synth.bf16_normal((L, tot, dp.cd), 837)
    sr = synth.bf16_normal((L, tot, dp.H * dp.d), 838)
    ts = [torch.from_numpy(x.copy()) for x in (s0, s1, nr)]
    ws2 = torch.empty(kv.kv_splice_composed_workspace_size(dp.desc, glens, *ts),
                      dtype=torch.uint8, device="cuda")
    kv.kv_splice_composed(dp.desc, bt, 40, glens, *ts, sc.cuda(), sr.cuda(), ws2)
    assert kv.kv_get_device_status(ws2) == kv.KV_OK
    assert orc.splice_composed(dp.orc, ss.block_tables, olens, s0, s1, nr,
                               synth.bits(sc).copy(), synth.bits(sr).copy()) == O.OK
    assert glens.tolist() == olens.tolist()
    check_pool(dp, f"interleaved composed splice {shape}")


def test_remapped_splice_and_patch(orc):
    # whole-block directives by block-table remapping, then an in-place patch
    lens = [1000, 700]
    ss = synth.splice_seqs(840, lens, 24, spare_blocks=2)
    dp = DevPool("mla", L, ss.num_slots, 841, pair_convention=IL)
    bt = to_dev(ss.block_tables)
    s0, s1, nr = [64, 128], [320, 192], [128, 192]
    sc = synth.bf16_normal((L, sum(nr), 512), 842)
    sr = synth.bf16_normal((L, sum(nr), 64), 843)
    glens = torch.tensor(lens, dtype=torch.int32)
    ws = kv.workspace(dp.desc, 2000, 2)
    kv.kv_splice(dp.desc, 2, bt, 24, glens, torch.tensor(s0, dtype=torch.int32),
                 torch.tensor(s1, dtype=torch.int32), torch.tensor(nr, dtype=torch.int32),
                 sc.cuda(), sr.cuda(), kv.KV_AMORTIZE_REMAP, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice(dp.orc, ss.block_tables, olens, s0, s1, nr, synth.bits(sc).copy(),
                      synth.bits(sr).copy()) == O.OK
    new_bt = bt.cpu().numpy()
    gc, gr = dp.gpu_bits()
    for q in range(2):
        n = int(olens[q])
        old = np.array([int(ss.block_tables[q, p // 64]) * 64 + p % 64 for p in range(n)])
        new = np.array([int(new_bt[q, p // 64]) * 64 + p % 64 for p in range(n)])
        check_exact(gc[:, new], dp.orc.copy[:, old], f"sequence {q}: verbatim part")
        check_exact(gr[:, new], dp.orc.rot[:, old], f"sequence {q}: rotary part")

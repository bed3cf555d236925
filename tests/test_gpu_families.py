"""The attention families beyond MLA and 8-head GQA (Kamera §2 names MHA,
GQA and MLA as the three families of its unified operator): GQA with 4 KV
heads of 128 (RoPE base 1e6) and MHA with 32 heads of 128 (base 1e4).  Each
runs the relocation (plain, with a fused patch, and the standalone patch),
the splice, the composed splice and the remapped splice against the fp64
oracle through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, SHAPES, check_exact, check_pool, to_dev

pytestmark = pytest.mark.gpu

L = 2
FAMILIES = ["gqa4", "mha"]


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _reloc_case(shape, seed, num_reqs=3, chunks=3):
    wl = synth.relocate_workload(seed, num_reqs=num_reqs, chunks_per_req=chunks, len_lo=1,
                                 len_hi=150, delta_lo=-40000, delta_hi=40000, n_pool_chunks=5,
                                 base_hi=200)
    src = DevPool(shape, L, wl.src_slots_total, seed)
    dst = DevPool(shape, L, wl.dst_slots_total, seed + 10)
    dev = [to_dev(getattr(wl, k)) for k in
           ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta", "block_tables")]
    return wl, src, dst, dev


def _factors(shape, wl, m, seed):
    cd, H, d, _ = SHAPES[shape]
    widths = (cd, H * d)
    us = [synth.f32_normal((L, wl.total_tokens, m), seed + i, std=0.02) for i in range(2)]
    vs = [synth.f32_normal((L, wl.num_chunks, widths[i], m), seed + 2 + i, std=0.02)
          for i in range(2)]
    return us, vs


@pytest.mark.parametrize("shape", FAMILIES)
@pytest.mark.parametrize("m", [0, 16, 32])
def test_relocate(orc, shape, m):
    wl, src, dst, dev = _reloc_case(shape, 700 + m)
    pd = patch = None
    if m:
        us, vs = _factors(shape, wl, m, 710 + m)
        pd = kv.patch_desc(m, [x.cuda() for x in us], [x.cuda() for x in vs])
        patch = O.Patch(m, [x.numpy() for x in us], [x.numpy() for x in vs])
    ws = kv.workspace(dst.desc, wl.total_tokens, wl.num_chunks)
    kv.kv_relocate(src.desc, dst.desc, wl.num_chunks, wl.total_tokens, *dev,
                   wl.block_tables.shape[0], wl.block_tables.shape[1], pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert orc.relocate(src.orc, dst.orc, wl.tok_off, wl.src_slots, wl.chunk_req,
                        wl.chunk_dst_pos, wl.delta, wl.block_tables, patch) == O.OK
    stats = check_pool(dst, f"relocate {shape} rank {m}", copy_exact=m == 0)
    if m == 0:
        assert stats["exact"] >= stats["values"] - max(3, stats["values"] // 100000), stats


@pytest.mark.parametrize("shape", FAMILIES)
def test_standalone_patch(orc, shape):
    wl, src, dst, dev = _reloc_case(shape, 720)
    us, vs = _factors(shape, wl, 8, 721)
    pd = kv.patch_desc(8, [x.cuda() for x in us], [x.cuda() for x in vs])
    ws = kv.workspace(dst.desc, wl.total_tokens, wl.num_chunks)
    tok_off, _, chunk_req, dst_pos, _, bt = dev
    kv.kv_patch(dst.desc, wl.num_chunks, wl.total_tokens, tok_off, chunk_req, dst_pos, bt,
                wl.block_tables.shape[0], wl.block_tables.shape[1], pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert orc.patch_apply(dst.orc, wl.tok_off, wl.chunk_req, wl.chunk_dst_pos, wl.block_tables,
                           O.Patch(8, [x.numpy() for x in us], [x.numpy() for x in vs])) == O.OK
    check_pool(dst, f"patch {shape}", copy_exact=False)


def _splice_setup(shape, lens, max_blocks, seed):
    ss = synth.splice_seqs(seed, lens, max_blocks, spare_blocks=2)
    dp = DevPool(shape, L, ss.num_slots, seed)
    return ss, dp, to_dev(ss.block_tables)


def _stubs(dp, tot, seed):
    sc = synth.bf16_normal((L, tot, dp.cd), seed)
    sr = synth.bf16_normal((L, tot, dp.H * dp.d), seed + 1)
    return sc, sr


@pytest.mark.parametrize("shape", FAMILIES)
def test_splice(orc, shape):
    lens = [0, 70, 700, 1300]
    ss, dp, bt = _splice_setup(shape, lens, 40, 730)
    d = synth.random_directives(731, np.asarray(lens, np.int32), 0, 500, 0, 300)
    tot = int(d.stub_len.sum())
    sc, sr = _stubs(dp, tot, 732)
    glens = torch.tensor(lens, dtype=torch.int32)
    ws = kv.workspace(dp.desc, sum(lens) + tot, len(lens))
    kv.kv_splice(dp.desc, len(lens), bt, 40, glens,
                 *[torch.from_numpy(x.copy()) for x in (d.s_start, d.s_end, d.stub_len)],
                 sc.cuda() if tot else None, sr.cuda() if tot else None, kv.KV_AMORTIZE, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice(dp.orc, ss.block_tables, olens, d.s_start, d.s_end, d.stub_len,
                      synth.bits(sc).copy() if tot else None,
                      synth.bits(sr).copy() if tot else None) == O.OK
    assert glens.tolist() == olens.tolist()
    check_pool(dp, f"splice {shape}")


@pytest.mark.parametrize("shape", FAMILIES)
def test_composed_splice(orc, shape):
    lens = [300, 1100]
    ss, dp, bt = _splice_setup(shape, lens, 40, 740)
    cur = np.asarray(lens, np.int32)
    s0, s1, nr = [], [], []
    for r in range(3):
        d = synth.random_directives(741 + r, cur, 0, 300, 0, 200)
        s0.append(d.s_start)
        s1.append(d.s_end)
        nr.append(d.stub_len)
        cur = cur + d.stub_len - (d.s_end - d.s_start)
    s0, s1, nr = (np.ascontiguousarray(np.stack(x)) for x in (s0, s1, nr))
    tot = int(nr.sum())
    sc, sr = _stubs(dp, tot, 745)
    glens = torch.tensor(lens, dtype=torch.int32)
    ts = [torch.from_numpy(x.copy()) for x in (s0, s1, nr)]
    ws = torch.empty(kv.kv_splice_composed_workspace_size(dp.desc, glens, *ts),
                     dtype=torch.uint8, device="cuda")
    kv.kv_splice_composed(dp.desc, bt, 40, glens, *ts, sc.cuda() if tot else None,
                          sr.cuda() if tot else None, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice_composed(dp.orc, ss.block_tables, olens, s0, s1, nr,
                               synth.bits(sc).copy() if tot else None,
                               synth.bits(sr).copy() if tot else None) == O.OK
    assert glens.tolist() == olens.tolist()
    check_pool(dp, f"composed splice {shape}")


@pytest.mark.parametrize("shape", FAMILIES)
def test_remapped_splice(orc, shape):
    lens = [900, 1000]
    s0, s1, nr = [128, 64], [384, 128], [64, 256]            # whole blocks, shrink / grow
    ss, dp, bt = _splice_setup(shape, lens, 24, 750)
    tot = sum(nr)
    sc, sr = _stubs(dp, tot, 751)
    glens = torch.tensor(lens, dtype=torch.int32)
    ws = kv.workspace(dp.desc, sum(lens) + tot, len(lens))
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
        check_exact(gc[:, new], dp.orc.copy[:, old], f"{shape} sequence {q}: verbatim part")
        check_exact(gr[:, new], dp.orc.rot[:, old], f"{shape} sequence {q}: rotary part")

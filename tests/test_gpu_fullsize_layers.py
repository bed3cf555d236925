"""Full-size parity on whole layers: the benchmark's full workloads run once
in the launch configuration bench.py times, then the first, middle and last
layers are compared in full -- every relocated token of every request, every
live row of every sequence -- with the fp64 oracle run on that layer alone
(layers are independent units of every operation).  Copies bit-exact,
rotated and patched values within 1 bf16 ulp; the fused-patch relocations
are checked on every layer the oracle can redo in about a minute (three for
MLA, the first and last for GQA with its rank-16 patch on both channels)."""
import numpy as np
import pytest
import torch

import bench
import oracle as O
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _layers(L):
    return sorted({0, L // 2, L - 1})


def _slots(bt, req, pos):
    """Pool slots of logical positions `pos` of requests `req` (64-slot blocks)."""
    return bt[req, pos // 64].astype(np.int64) * 64 + pos % 64


def _assert_rows(got, want, what):
    copy_bad = int((got[:, :512] != want[:, :512]).any(axis=1).sum())
    r = bench.ulp_stats(got[:, 512:], want[:, 512:])
    assert copy_bad == 0, f"{what}: {copy_bad} c_KV rows differ"
    assert r["beyond"] == 0, f"{what}: {r}"
    return r


def _one_layer_pool(rows, base):
    return O.Pool(np.ascontiguousarray(rows[None, :, :512]),
                  np.ascontiguousarray(rows[None, :, 512:]), 64, 1, 64, base)


def test_relocate_mla_whole_layers():
    st = bench.build_relocate_mla(0)
    bench.relocate_call(st)
    torch.cuda.synchronize()
    wl, base, orc = st["wl"], st["cfg"]["base"], O.get()
    tok = np.arange(wl.total_tokens)
    chunk = np.searchsorted(wl.tok_off, tok, side="right") - 1
    pos = wl.chunk_dst_pos[chunk] + (tok - wl.tok_off[chunk])
    dslot = _slots(wl.block_tables, wl.chunk_req[chunk], pos)
    assert len(np.unique(dslot)) == wl.total_tokens
    for l in _layers(st["L"]):
        src = _one_layer_pool(synth.bits(st["src"][l].cpu()), base)
        dst = _one_layer_pool(np.zeros((wl.dst_slots_total, 576), np.uint16), base)
        assert orc.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos,
                            wl.delta, wl.block_tables) == O.OK
        want = np.concatenate([dst.copy[0][dslot], dst.rot[0][dslot]], axis=1)
        got = synth.bits(st["dst"][l].cpu())[dslot]
        _assert_rows(got, want, f"relocate layer {l}")


def _oracle_splice_layer(st, l, orc, composed):
    base = st["cfg"]["base"]
    pool = _one_layer_pool(synth.bits(st["pristine"][l].cpu()), base)
    lens = st["ss"].seq_lens.astype(np.int32).copy()
    bt = st["ss"].block_tables
    if composed:
        rd = st["rounds"]
        s0 = np.stack([r["d"].s_start for r in rd]).astype(np.int32)
        s1 = np.stack([r["d"].s_end for r in rd]).astype(np.int32)
        nr = np.stack([r["d"].stub_len for r in rd]).astype(np.int32)
        sc = np.ascontiguousarray(np.concatenate(
            [synth.bits(r["stub_c"][l].cpu()) for r in rd])[None])
        sr = np.ascontiguousarray(np.concatenate(
            [synth.bits(r["stub_r"][l].cpu()) for r in rd])[None])
        assert orc.splice_composed(pool, bt, lens, s0, s1, nr, sc, sr) == O.OK
    else:
        for r in st["rounds"]:
            d = r["d"]
            sc = np.ascontiguousarray(synth.bits(r["stub_c"][l].cpu())[None])
            sr = np.ascontiguousarray(synth.bits(r["stub_r"][l].cpu())[None])
            assert orc.splice(pool, bt, lens, d.s_start, d.s_end, d.stub_len, sc, sr,
                              O.AMORTIZE) == O.OK
    assert np.array_equal(lens, st["final_lens"])
    return pool


def _check_splice(st, composed=False, final_bt=None):
    orc = O.get()
    lens = st["final_lens"]
    req = np.repeat(np.arange(st["S"]), lens)
    pos = np.concatenate([np.arange(n) for n in lens])
    want_slot = _slots(st["ss"].block_tables, req, pos)
    got_slot = _slots(st["ss"].block_tables if final_bt is None else final_bt, req, pos)
    stats = []
    for l in _layers(st["L"]):
        pool = _oracle_splice_layer(st, l, orc, composed)
        want = np.concatenate([pool.copy[0][want_slot], pool.rot[0][want_slot]], axis=1)
        got = synth.bits(st["pool"][l].cpu())[got_slot]
        stats.append(_assert_rows(got, want, f"splice layer {l}"))
    return stats


def test_splice_128k_whole_layers():
    st = bench.build_splice(0, bench.SPLICE_128K)
    _, lens = bench.splice_step(st)
    torch.cuda.synchronize()
    assert np.array_equal(lens.numpy(), st["final_lens"])
    _check_splice(st)


def test_splice_128k_composed_whole_layers():
    import position_independent_mla_gb300 as kv

    st = bench.build_splice(0, bench.SPLICE_128K)
    s0, s1, nr = (torch.stack([rd["args"][j] for rd in st["rounds"]]).contiguous()
                  for j in range(3))
    stub_c = torch.cat([rd["stub_c"] for rd in st["rounds"]], dim=1).contiguous()
    stub_r = torch.cat([rd["stub_r"] for rd in st["rounds"]], dim=1).contiguous()
    lens = torch.from_numpy(st["ss"].seq_lens.copy())
    ws = torch.empty(kv.kv_splice_composed_workspace_size(st["desc"], lens, s0, s1, nr),
                     dtype=torch.uint8, device="cuda")
    kv.kv_splice_composed(st["desc"], st["bt"], st["max_blocks"], lens, s0, s1, nr, stub_c,
                          stub_r, ws)
    torch.cuda.synchronize()
    assert np.array_equal(lens.numpy(), st["final_lens"])
    _check_splice(st, composed=True)


def test_splice_128k_remap_whole_layers():
    import position_independent_mla_gb300 as kv

    st = bench.build_splice(0, bench.SPLICE_128K, aligned=True)
    _, lens = bench.splice_step(st, mode=kv.KV_AMORTIZE_REMAP)
    torch.cuda.synchronize()
    assert np.array_equal(lens.numpy(), st["final_lens"])
    _check_splice(st, final_bt=st["bt"].cpu().numpy())


def _patch_for_layer(m, us, vs, l):
    """The oracle's patch for one layer: factors of layer l as a 1-layer set."""
    return O.Patch(m, [np.ascontiguousarray(u[l:l + 1].cpu().numpy()) for u in us],
                   [np.ascontiguousarray(v[l:l + 1].cpu().numpy()) for v in vs])


def _dest_slots(wl):
    tok = np.arange(wl.total_tokens)
    chunk = np.searchsorted(wl.tok_off, tok, side="right") - 1
    pos = wl.chunk_dst_pos[chunk] + (tok - wl.tok_off[chunk])
    return _slots(wl.block_tables, wl.chunk_req[chunk], pos)


def test_relocate_mla_fused_patch_whole_layers():
    import position_independent_mla_gb300 as kv

    st = bench.build_relocate_mla(0)
    wl, L, m, base, orc = st["wl"], st["L"], 8, st["cfg"]["base"], O.get()
    g = torch.Generator(device="cuda")
    g.manual_seed(6006)
    u = torch.randn((L, wl.total_tokens, m), generator=g, device="cuda").mul_(0.02)
    v = torch.randn((L, wl.num_chunks, 576, m), generator=g, device="cuda").mul_(0.02)
    patch = kv.patch_desc(m, [u, u], [v[:, :, :512], v[:, :, 512:]])
    d = st["dev"]
    kv.kv_relocate(st["sd"], st["dd"], wl.num_chunks, wl.total_tokens, d["tok_off"],
                   d["src_slots"], d["chunk_req"], d["chunk_dst_pos"], d["delta"],
                   d["block_tables"], wl.block_tables.shape[0], wl.block_tables.shape[1],
                   patch, st["ws"])
    assert kv.kv_get_device_status(st["ws"]) == kv.KV_OK
    dslot = _dest_slots(wl)
    for l in _layers(L):
        src = _one_layer_pool(synth.bits(st["src"][l].cpu()), base)
        dst = _one_layer_pool(np.zeros((wl.dst_slots_total, 576), np.uint16), base)
        vv = [v[:, :, :512], v[:, :, 512:]]
        assert orc.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos,
                            wl.delta, wl.block_tables, _patch_for_layer(m, [u, u], vv, l)) == O.OK
        want = np.concatenate([dst.copy[0][dslot], dst.rot[0][dslot]], axis=1)
        got = synth.bits(st["dst"][l].cpu())[dslot]
        r = bench.ulp_stats(got, want)   # patched copy part too: within 1 ulp
        assert r["beyond"] == 0, f"fused MLA patch layer {l}: {r}"


def test_relocate_gqa_fused_patch_first_and_last_layer():
    st = bench.build_relocate_gqa(0, bench.RELOC_GQA)
    bench.relocate_gqa_call(st, patch=True)
    torch.cuda.synchronize()
    wl, L, base, orc = st["wl"], st["L"], st["cfg"]["base"], O.get()
    m, fac = st["cfg"]["rank"], st["fac"]
    dslot = _dest_slots(wl)
    for l in (0, L - 1):
        src = O.Pool(synth.bits(st["src_v"][l].cpu())[None].copy(),
                     synth.bits(st["src_k"][l].cpu())[None].copy(), 64, 8, 128, base)
        dst = O.Pool(np.zeros((1, wl.dst_slots_total, 1024), np.uint16),
                     np.zeros((1, wl.dst_slots_total, 1024), np.uint16), 64, 8, 128, base)
        pt = _patch_for_layer(m, [fac["u_v"], fac["u_k"]], [fac["v_v"], fac["v_k"]], l)
        assert orc.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos,
                            wl.delta, wl.block_tables, pt) == O.OK
        for name, dev_t, want in (("V", st["dst_v"], dst.copy[0]), ("K", st["dst_k"], dst.rot[0])):
            got = synth.bits(dev_t[l].cpu())[dslot]
            r = bench.ulp_stats(got, want[dslot])
            assert r["beyond"] == 0, f"fused GQA patch layer {l} {name}: {r}"

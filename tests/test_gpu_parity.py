"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle,
element by element, on seeded inputs that span several tiles with ragged
tails, for both row shapes (MLA c_KV 512 + k_pe 64, RoPE base 10000; GQA
V and K of 8 x 128, base 500000).

Pages: Irminsul §2.1-§2.2 and Kamera §2 (relocation, patch), Leyline
§2.1-§2.3 (splice).  Tolerance: see tests/_gpu.py.
"""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, check_exact, check_pool, check_ulp, i32, resync, to_dev

pytestmark = pytest.mark.gpu

L = 3


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _reloc_case(shape, seed, num_reqs=5, chunks=4, lo=1, hi=150, deltas=None, layers=L):
    wl = synth.relocate_workload(seed, num_reqs=num_reqs, chunks_per_req=chunks, len_lo=lo,
                                 len_hi=hi, delta_lo=-32768, delta_hi=32768, n_pool_chunks=6,
                                 base_hi=300)
    if deltas is not None:
        wl.delta[:len(deltas)] = deltas
    src = DevPool(shape, layers, wl.src_slots_total, seed)
    dst = DevPool(shape, layers, wl.dst_slots_total, seed + 10)
    dev = {k: to_dev(getattr(wl, k)) for k in
           ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta", "block_tables")}
    return wl, src, dst, dev


def _run_relocate(wl, src, dst, dev, patch=None, ws=None):
    ws = ws if ws is not None else kv.workspace(dst.desc, wl.total_tokens, wl.num_chunks)
    kv.kv_relocate(src.desc, dst.desc, wl.num_chunks, wl.total_tokens, dev["tok_off"],
                   dev["src_slots"], dev["chunk_req"], dev["chunk_dst_pos"], dev["delta"],
                   dev["block_tables"], wl.block_tables.shape[0], wl.block_tables.shape[1],
                   patch, ws)
    return kv.kv_get_device_status(ws)


def _oracle_relocate(orc, wl, src, dst, patch=None):
    assert orc.relocate(src.orc, dst.orc, wl.tok_off, wl.src_slots, wl.chunk_req,
                        wl.chunk_dst_pos, wl.delta, wl.block_tables, patch) == O.OK


# ---------------------------------------------------------------------------
# Relocation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_relocate_matches_oracle(orc, shape):
    deltas = [0, 1, -1, 1000, -1000, 100000, -100000, 65536, 32768, -32768]
    wl, src, dst, dev = _reloc_case(shape, 200, deltas=deltas)
    src_before = src.gpu_bits()
    assert _run_relocate(wl, src, dst, dev) == kv.KV_OK
    assert kv.kv_last_launch_count() == 2
    _oracle_relocate(orc, wl, src, dst)
    stats = check_pool(dst, f"relocate {shape}")
    # the rotation is compensated: the oracle's bits almost everywhere (a rare
    # 1-ulp flip can only come from fp64 pow/sincos differing in the last bit)
    assert stats["exact"] >= stats["values"] - max(3, stats["values"] // 100000), stats
    sc, sr = src_before
    gc, gr = src.gpu_bits()
    check_exact(gc, sc, "source verbatim part unchanged")
    check_exact(gr, sr, "source rotary part unchanged")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_relocate_chunk_and_tile_edges(orc, shape):
    # single-token chunks, empty chunks and chunks much longer than a tile
    wl, src, dst, dev = _reloc_case(shape, 210, num_reqs=3, chunks=6, lo=0, hi=70)
    assert _run_relocate(wl, src, dst, dev) == kv.KV_OK
    _oracle_relocate(orc, wl, src, dst)
    check_pool(dst, f"relocate edges {shape}")


def test_relocate_zero_tokens_is_a_no_op(orc):
    wl, src, dst, dev = _reloc_case("mla", 220, num_reqs=1, chunks=1)
    before = dst.gpu_bits()
    ws = kv.workspace(dst.desc, 1, 1)
    kv.kv_relocate(src.desc, dst.desc, 0, 0, None, None, None, None, None, None, 0, 0, None, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert kv.kv_last_launch_count() == 0
    after = dst.gpu_bits()
    check_exact(after[0], before[0], "copy")
    check_exact(after[1], before[1], "rot")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_relocate_with_fused_patch(orc, shape):
    wl, src, dst, dev = _reloc_case(shape, 230, deltas=[0, 7, -40000])
    Ln, T, Cn = L, wl.total_tokens, wl.num_chunks
    if shape == "mla":
        m = 8  # one factor pair over the whole 576-wide row (Kamera §2, both channels)
        u = synth.f32_normal((Ln, T, m), 231, std=0.02)
        v = synth.f32_normal((Ln, Cn, 576, m), 232, std=0.02)
        us, vs = [u, u], [v[:, :, :512], v[:, :, 512:]]
    else:
        m = 16  # independent factors for V (channel 0) and K (channel 1)
        us = [synth.f32_normal((Ln, T, m), 233 + i, std=0.02) for i in range(2)]
        vs = [synth.f32_normal((Ln, Cn, 1024, m), 235 + i, std=0.02) for i in range(2)]
    ud = [x.cuda() for x in us]
    if shape == "mla":
        vd = v.cuda()
        vds = [vd[:, :, :512], vd[:, :, 512:]]
    else:
        vds = [x.cuda() for x in vs]
    pd = kv.patch_desc(m, ud, vds)
    assert _run_relocate(wl, src, dst, dev, patch=pd) == kv.KV_OK
    _oracle_relocate(orc, wl, src, dst,
                     O.Patch(m, [x.numpy() for x in us], [x.numpy() for x in vs]))
    check_pool(dst, f"relocate+patch {shape}", copy_exact=False)


@pytest.mark.parametrize("m", [32, 64])
def test_relocate_with_fused_patch_large_rank(orc, m):
    # ranks above 16 take the general per-item path
    wl, src, dst, dev = _reloc_case("gqa", 235, num_reqs=2, chunks=3, deltas=[0, 99])
    us = [synth.f32_normal((L, wl.total_tokens, m), 236 + i, std=0.01) for i in range(2)]
    vs = [synth.f32_normal((L, wl.num_chunks, 1024, m), 238 + i, std=0.01) for i in range(2)]
    pd = kv.patch_desc(m, [x.cuda() for x in us], [x.cuda() for x in vs])
    assert _run_relocate(wl, src, dst, dev, patch=pd) == kv.KV_OK
    _oracle_relocate(orc, wl, src, dst,
                     O.Patch(m, [x.numpy() for x in us], [x.numpy() for x in vs]))
    check_pool(dst, f"relocate+patch rank {m}", copy_exact=False)


# chunks of 1-150 tokens (mostly under one 128-row tile) and of 200-600
# tokens (several tiles per block); in place, MLA's c_KV and k_pe slices are
# launched separately
@pytest.mark.parametrize("shape", ["mla", "gqa"])
@pytest.mark.parametrize("lens", [(1, 150), (200, 600)])
def test_standalone_patch(orc, shape, lens):
    wl, src, dst, dev = _reloc_case(shape, 240, lo=lens[0], hi=lens[1])
    m = 4 if shape == "mla" else 12
    us = [synth.f32_normal((L, wl.total_tokens, m), 241 + i, std=0.05) for i in range(2)]
    widths = (512, 64) if shape == "mla" else (1024, 1024)
    vs = [synth.f32_normal((L, wl.num_chunks, widths[i], m), 243 + i, std=0.05)
          for i in range(2)]
    ws = kv.workspace(dst.desc, wl.total_tokens, wl.num_chunks)
    pd = kv.patch_desc(m, [x.cuda() for x in us], [x.cuda() for x in vs])
    kv.kv_patch(dst.desc, wl.num_chunks, wl.total_tokens, dev["tok_off"], dev["chunk_req"],
                dev["chunk_dst_pos"], dev["block_tables"], wl.block_tables.shape[0],
                wl.block_tables.shape[1], pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    assert kv.kv_last_launch_count() == (2 if shape == "mla" else 1)
    assert orc.patch_apply(dst.orc, wl.tok_off, wl.chunk_req, wl.chunk_dst_pos, wl.block_tables,
                           O.Patch(m, [x.numpy() for x in us],
                                   [x.numpy() for x in vs])) == O.OK
    check_pool(dst, f"patch {shape}", copy_exact=False)


@pytest.mark.parametrize("shape", ["mla", "gqa"])
@pytest.mark.parametrize("patched_ch", [0, 1])
def test_patch_on_one_channel_only(orc, shape, patched_ch):
    # the other channel is copied verbatim / rotated exactly, as without a patch
    wl, src, dst, dev = _reloc_case(shape, 245 + patched_ch, num_reqs=2, chunks=3,
                                    deltas=[0, 3, -20000])
    m = 4  # ranks are multiples of 4
    widths = (src.cd, src.H * src.d)
    us, vs = [None, None], [None, None]
    us[patched_ch] = synth.f32_normal((L, wl.total_tokens, m), 247, std=0.03)
    vs[patched_ch] = synth.f32_normal((L, wl.num_chunks, widths[patched_ch], m), 248,
                                      std=0.03)
    pd = kv.patch_desc(m, [None if x is None else x.cuda() for x in us],
                       [None if x is None else x.cuda() for x in vs])
    assert _run_relocate(wl, src, dst, dev, patch=pd) == kv.KV_OK
    _oracle_relocate(orc, wl, src, dst, O.Patch(m, [None if x is None else x.numpy() for x in us],
                                                [None if x is None else x.numpy() for x in vs]))
    stats = check_pool(dst, f"one-channel patch {shape} ch{patched_ch}",
                       copy_exact=patched_ch == 1)
    if patched_ch == 0:  # the unpatched rotation keeps the oracle's bits, as without a patch
        assert stats["exact"] >= stats["values"] - max(3, stats["values"] // 100000), stats


def test_relocate_reports_a_bad_index_and_skips_its_row(orc):
    wl, src, dst, dev = _reloc_case("mla", 250, num_reqs=2, chunks=2)
    before = dst.gpu_bits()
    bad_t = wl.total_tokens - 1
    slots = wl.src_slots.copy()
    slots[bad_t] = wl.src_slots_total          # one past the source pool
    dev["src_slots"] = to_dev(slots)
    assert _run_relocate(wl, src, dst, dev) == kv.KV_ERR_OUT_OF_RANGE
    # every other row matches the oracle; the bad token's target row is untouched
    _oracle_relocate(orc, wl, src, dst)
    c = int(np.searchsorted(wl.tok_off, bad_t, side="right") - 1)
    p = int(wl.chunk_dst_pos[c]) + bad_t - int(wl.tok_off[c])
    s = int(wl.block_tables[wl.chunk_req[c], p // 64]) * 64 + p % 64
    dst.orc.copy[:, s] = before[0][:, s]
    dst.orc.rot[:, s] = before[1][:, s]
    check_pool(dst, "relocate with one bad index")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_relocate_nonfinite_inputs(orc, shape):
    wl, src, dst, dev = _reloc_case(shape, 260, num_reqs=1, chunks=2, lo=40, hi=60,
                                    deltas=[321, -77])

    def plant(s, cols, b):
        src.orc.rot[0, s, cols] = b
        src.rot_view[0, s, cols] = torch.tensor(int(np.array(b, np.uint16).view(np.int16)),
                                                dtype=torch.int16).view(torch.bfloat16)

    # Inf / NaN in a few source rotary values (and their bf16 mirrors)
    specials = [0x7F80, 0xFF80, 0x7FC0, 0x7F81]
    for k, b in enumerate(specials):
        plant(int(wl.src_slots[k]), 3 + 17 * k, b)
    # a whole half-head at +Inf, and the largest finite bf16 (0x7F7F) in both
    # halves of a head, with equal and opposite signs: the rotated value
    # overflows fp32 for some frequencies, the rounding gives +-Inf
    h = src.d // 2
    plant(int(wl.src_slots[4]), slice(0, h), 0x7F80)
    plant(int(wl.src_slots[5]), slice(0, src.d), 0x7F7F)
    plant(int(wl.src_slots[6]), slice(0, h), 0x7F7F)
    plant(int(wl.src_slots[6]), slice(h, src.d), 0xFF7F)
    assert _run_relocate(wl, src, dst, dev) == kv.KV_OK
    _oracle_relocate(orc, wl, src, dst)
    check_pool(dst, "relocate with Inf/NaN and overflow")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_fused_patch_nonfinite_inputs(orc, shape):
    wl, src, dst, dev = _reloc_case(shape, 265, num_reqs=1, chunks=2, lo=40, hi=60,
                                    deltas=[-555, 4321])
    def plant(which, s, cols, b):
        arr, view = (src.orc.rot, src.rot_view) if which == "rot" else (src.orc.copy,
                                                                        src.copy_view)
        arr[1, s, cols] = b
        view[1, s, cols] = torch.tensor(int(np.array(b, np.uint16).view(np.int16)),
                                        dtype=torch.int16).view(torch.bfloat16)

    specials = [0x7F80, 0xFF80, 0x7FC0, 0x7F81, 0x7F80]
    for k, b in enumerate(specials):
        plant("rot", int(wl.src_slots[k]), (3 + 17 * k) % (src.H * src.d), b)
    # whole rotary half-heads at +-Inf: every frequency of the head, so the
    # rotation meets both signs of the split cos / sin parts
    h = src.d // 2
    plant("rot", int(wl.src_slots[5]), slice(0, h), 0x7F80)
    plant("rot", int(wl.src_slots[6]), slice(src.d + h, 2 * src.d) if src.H > 1
          else slice(h, src.d), 0xFF80)
    plant("copy", int(wl.src_slots[7]), slice(0, 8), 0x7F80)
    # the largest finite bf16 in both halves of a head: the rotated value
    # overflows for some frequencies
    plant("rot", int(wl.src_slots[8]), slice(0, src.d), 0x7F7F)
    plant("copy", int(wl.src_slots[7]), slice(8, 16), 0x7FC0)
    m = 8
    widths = (src.cd, src.H * src.d)
    us = [synth.f32_normal((L, wl.total_tokens, m), 266 + i, std=0.02) for i in range(2)]
    vs = [synth.f32_normal((L, wl.num_chunks, widths[i], m), 268 + i, std=0.02)
          for i in range(2)]
    ud, vd = [x.cuda() for x in us], [x.cuda() for x in vs]
    assert _run_relocate(wl, src, dst, dev, patch=kv.patch_desc(m, ud, vd)) == kv.KV_OK
    _oracle_relocate(orc, wl, src, dst,
                     O.Patch(m, [x.numpy() for x in us], [x.numpy() for x in vs]))
    check_pool(dst, f"fused patch with Inf/NaN ({shape})", copy_exact=False)


# ---------------------------------------------------------------------------
# Splice
# ---------------------------------------------------------------------------

def _splice_pool(shape, lens, max_blocks, seed, layers=L, spare=3):
    ss = synth.splice_seqs(seed, lens, max_blocks, spare_blocks=spare)
    dp = DevPool(shape, layers, ss.num_slots, seed)
    return ss, dp, to_dev(ss.block_tables)


def _splice_both(orc, ss, dp, bt, glens, olens, s0, s1, nr, seed, layers=L, ws=None):
    tot = int(np.sum(nr))
    sc = synth.bf16_normal((layers, tot, dp.cd), seed)
    sr = synth.bf16_normal((layers, tot, dp.H * dp.d), seed + 1)
    if ws is None:
        rows = int(np.sum(np.asarray(glens) - np.asarray(s1))) + tot
        ws = kv.workspace(dp.desc, rows, len(s0))
    kv.kv_splice(dp.desc, len(s0), bt, ss.block_tables.shape[1], glens,
                 torch.tensor(s0, dtype=torch.int32), torch.tensor(s1, dtype=torch.int32),
                 torch.tensor(nr, dtype=torch.int32), sc.cuda() if tot else None,
                 sr.cuda() if tot else None, kv.KV_AMORTIZE, ws)
    st = kv.kv_get_device_status(ws)
    assert orc.splice(dp.orc, ss.block_tables, olens, s0, s1, nr,
                      synth.bits(sc).copy() if tot else None,
                      synth.bits(sr).copy() if tot else None) == O.OK
    assert glens.tolist() == olens.tolist()
    return st


def test_splice_single_layer_4096_tokens(orc):
    # one MLA layer, 4096 cached tokens, [1024, 2048) replaced by a 16-row stub: Δ = -1008
    ss, dp, bt = _splice_pool("mla", [4096], 64, 300, layers=1)
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    assert _splice_both(orc, ss, dp, bt, glens, olens, [1024], [2048], [16], 301,
                        layers=1) == kv.KV_OK
    assert glens.tolist() == [3088]
    stats = check_pool(dp, "splice 4096")
    assert stats["exact"] >= stats["values"] - 3, stats


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_splice_successive_random_directives(orc, shape):
    lens = [0, 1, 63, 64, 65, 700, 1500, 2900]
    ss, dp, bt = _splice_pool(shape, lens, 80, 310 + len(shape))
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    for rnd in range(3):
        d = synth.random_directives(320 + rnd, olens, 0, 800, 0, 900)
        assert _splice_both(orc, ss, dp, bt, glens, olens, d.s_start.tolist(),
                            d.s_end.tolist(), d.stub_len.tolist(), 330 + rnd) == kv.KV_OK
        stats = check_pool(dp, f"splice {shape}, directive round {rnd}")
        assert stats["exact"] >= stats["values"] - max(3, stats["values"] // 100000), stats
        # each round is compared on identical inputs
        resync(dp)


@pytest.mark.parametrize("delta", [-1, 1, -63, 64, 65, -129])
def test_splice_small_shifts_over_long_sequences(orc, delta):
    # |Δ| below a tile: every tile waits on its predecessor's reads
    n = 9000
    ss, dp, bt = _splice_pool("mla", [n], 150, 400 + delta, layers=2)
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    s0 = 1234
    nr = max(5, delta + 5)
    s1 = s0 + nr - delta
    assert _splice_both(orc, ss, dp, bt, glens, olens, [s0], [s1], [nr], 401,
                        layers=2) == kv.KV_OK
    check_pool(dp, f"splice Δ={delta}")


def test_splice_large_insertion_and_removal(orc):
    ss, dp, bt = _splice_pool("mla", [2000, 6000], 120, 410, layers=2)
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    # seq 0: a 5000-row stub inserted at 300 (Δ = +4990); seq 1: 5000 rows removed
    assert _splice_both(orc, ss, dp, bt, glens, olens, [300, 100], [310, 5100], [5000, 0], 411,
                        layers=2) == kv.KV_OK
    check_pool(dp, "splice large Δ")


def test_splice_degenerate_directives(orc):
    lens = [50, 50, 50, 50, 50, 0, 50]
    ss, dp, bt = _splice_pool("gqa", lens, 3, 420, layers=2)
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    s0 = [50, 10, 10, 10, 0, 0, 0]    # tail append, insertion, deletion, same-length, all, empty
    s1 = [50, 10, 30, 20, 50, 0, 50]
    nr = [7, 9, 0, 10, 0, 20, 60]
    assert _splice_both(orc, ss, dp, bt, glens, olens, s0, s1, nr, 421, layers=2) == kv.KV_OK
    check_pool(dp, "degenerate splices")


def test_splice_more_sequences_than_one_launch(orc):
    lens = [int(x) for x in np.random.default_rng(5).integers(0, 300, 70)]
    ss, dp, bt = _splice_pool("mla", lens, 8, 430, layers=2)
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    d = synth.random_directives(431, lens, 0, 100, 0, 120)
    assert _splice_both(orc, ss, dp, bt, glens, olens, d.s_start.tolist(), d.s_end.tolist(),
                        d.stub_len.tolist(), 432, layers=2) == kv.KV_OK
    # two launches (64 + 6 sequences); both are short enough to form their
    # cos/sin rows inside the splice kernel, so no δ-table kernel runs
    assert kv.kv_last_launch_count() == 2
    check_pool(dp, "splice 70 sequences")


def test_splice_forget_moves_nothing(orc):
    ss, dp, bt = _splice_pool("mla", [500], 10, 440, layers=1)
    before = dp.gpu_bits()
    lens = torch.from_numpy(ss.seq_lens.copy())
    kv.kv_splice(dp.desc, 1, bt, 10, lens, i32(100), i32(200), i32(5), None, None, kv.KV_FORGET,
                 None)
    assert lens.tolist() == [100] and kv.kv_last_launch_count() == 0
    after = dp.gpu_bits()
    check_exact(after[0], before[0], "copy")
    check_exact(after[1], before[1], "rot")


# ---------------------------------------------------------------------------
# Bounded waits: the failure path without a fault
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_context_survives(orc):
    ss, dp, bt = _splice_pool("mla", [300], 8, 450, layers=1)
    ws = kv.workspace(dp.desc, 400, 1)
    assert kv.kv_check_wait_timeout(ws, 50_000_000) == kv.KV_OK
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_TIMEOUT
    # the context is still usable: a splice right after succeeds and matches
    glens = torch.from_numpy(ss.seq_lens.copy())
    olens = ss.seq_lens.copy()
    assert _splice_both(orc, ss, dp, bt, glens, olens, [10], [40], [3], 451, layers=1,
                        ws=ws) == kv.KV_OK
    check_pool(dp, "splice after timeout")

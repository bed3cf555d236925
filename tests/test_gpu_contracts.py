"""GPU tests of the caller contracts and failure paths of the in-place kernels.

* Debug checks (kv_set_debug_checks): a relocation inside one pool whose
  destination slots meet its source slots (Irminsul §2.2: stored rows are
  gathered into new slots), and a splice whose block-table entries name a
  block twice (Leyline §2.1-§2.3: the in-place shift assumes distinct slots),
  are reported as KV_ERR_OVERLAP and leave the pools and block tables bit for
  bit unchanged; calls that keep the contracts still match the oracle.
* Factor extents: a patch whose mapped U row or V slot falls outside the
  factor arrays is reported as KV_ERR_OUT_OF_RANGE instead of being read.
* The splice kernels' own timeout branch: one tile is made to skip its read
  publications (kv_set_splice_skip_publish), so the tiles that overwrite its
  rows wait until a short limit, report KV_ERR_TIMEOUT and skip their stores;
  the launch still ends, and the next call on the same workspace matches the
  oracle bit for bit.  No GPU is faulted or hung: every wait is bounded.
"""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, check_exact, check_pool, i32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return O.get()


@pytest.fixture
def debug_checks():
    kv.kv_set_debug_checks(True)
    yield
    kv.kv_set_debug_checks(False)


@pytest.fixture
def skip_publish():
    kv.kv_set_wait_limit_ns(20_000_000)   # 20 ms: the starved waits end quickly
    yield kv.kv_set_splice_skip_publish
    kv.kv_set_splice_skip_publish(-1)
    kv.kv_set_wait_limit_ns(0)            # back to the default


def _snapshot(dp: DevPool):
    c, r = dp.gpu_bits()
    return c.copy(), r.copy()


def _unchanged(dp: DevPool, snap, what):
    c, r = dp.gpu_bits()
    check_exact(c, snap[0], what + " (verbatim part)")
    check_exact(r, snap[1], what + " (rotary part)")


# ---------------------------------------------------------------------------
# Relocation inside one pool
# ---------------------------------------------------------------------------

def _one_pool_relocation(shape, src_slots, dst_pos, delta, blocks, seed):
    """One request, one chunk: rows from `src_slots` of a pool of `blocks`
    blocks to logical positions dst_pos.. of a request whose block table is
    the identity (logical block b = physical block b) -- in the same pool."""
    dp = DevPool(shape, 2, blocks * 64, seed)
    n = len(src_slots)
    host = dict(tok_off=np.array([0, n], np.int32), src_slots=np.array(src_slots, np.int32),
                chunk_req=np.array([0], np.int32), chunk_dst_pos=np.array([dst_pos], np.int32),
                delta=np.array([delta], np.int32),
                block_tables=np.arange(blocks, dtype=np.int32).reshape(1, blocks))
    dev = {k: to_dev(v) for k, v in host.items()}
    return dp, host, dev


def _relocate_same_pool(dp, host, dev, ws):
    n = int(host["tok_off"][-1])
    kv.kv_relocate(dp.desc, dp.desc, 1, n, dev["tok_off"], dev["src_slots"], dev["chunk_req"],
                   dev["chunk_dst_pos"], dev["delta"], dev["block_tables"], 1,
                   host["block_tables"].shape[1], None, ws)
    return kv.kv_get_device_status(ws)


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_relocation_overlap_is_reported_and_nothing_is_stored(shape, debug_checks):
    # rows of slots 0..39 moved to positions 20..59 of the same pool: slots 20..39 meet
    dp, host, dev = _one_pool_relocation(shape, list(range(40)), 20, 777, 4, 900)
    ws = kv.workspace(dp.desc, 40, 1)
    snap = _snapshot(dp)
    assert _relocate_same_pool(dp, host, dev, ws) == kv.KV_ERR_OVERLAP
    _unchanged(dp, snap, f"{shape} overlapping relocation")
    # a single shared slot is enough
    dp, host, dev = _one_pool_relocation(shape, [3, 70, 71], 130, -5, 4, 901)
    host["src_slots"][1] = 131   # source slot 131 is also the destination of token 1
    dev["src_slots"] = to_dev(host["src_slots"])
    snap = _snapshot(dp)
    assert _relocate_same_pool(dp, host, dev, ws) == kv.KV_ERR_OVERLAP
    _unchanged(dp, snap, f"{shape} one shared slot")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_relocation_in_one_pool_without_overlap_matches_oracle(orc, shape, debug_checks):
    # rows of block 0 to positions 100.. (blocks 1-2): no slot is read and written
    dp, host, dev = _one_pool_relocation(shape, list(range(5, 65)), 100, 12345, 4, 910)
    ws = kv.workspace(dp.desc, 60, 1)
    assert _relocate_same_pool(dp, host, dev, ws) == kv.KV_OK
    assert kv.kv_last_launch_count() == 4   # 2 checks + table + relocation
    assert orc.relocate(dp.orc, dp.orc, host["tok_off"], host["src_slots"], host["chunk_req"],
                        host["chunk_dst_pos"], host["delta"], host["block_tables"]) == O.OK
    check_pool(dp, f"{shape} relocation inside one pool", rot_exact=True)


def test_debug_checks_off_launch_nothing_more():
    dp, host, dev = _one_pool_relocation("mla", list(range(5, 65)), 100, 1, 4, 920)
    ws = kv.workspace(dp.desc, 60, 1)
    assert _relocate_same_pool(dp, host, dev, ws) == kv.KV_OK
    assert kv.kv_last_launch_count() == 2   # table + relocation


# ---------------------------------------------------------------------------
# Splices with a duplicated block
# ---------------------------------------------------------------------------

def _splice_case(shape, lens, max_blocks, seed, layers=2):
    ss = synth.splice_seqs(seed, lens, max_blocks, spare_blocks=2)
    dp = DevPool(shape, layers, ss.num_slots, seed)
    return ss, dp


def _stubs(dp, nr, seed, layers=2):
    tot = int(np.sum(nr))
    sc = synth.bf16_normal((layers, tot, dp.cd), seed)
    sr = synth.bf16_normal((layers, tot, dp.H * dp.d), seed + 1)
    return sc, sr


@pytest.mark.parametrize("mode", ["amortize", "remap"])
def test_splice_duplicate_block_is_reported_and_nothing_is_stored(mode, debug_checks):
    lens = [640, 320]
    ss, dp = _splice_case("mla", lens, 12, 930)
    bt_h = ss.block_tables.copy()
    bt_h[1, 2] = bt_h[0, 7]          # both entries are in use
    bt = to_dev(bt_h)
    if mode == "remap":               # block-aligned directives that shift
        s0, s1, nr = [64, 0], [192, 64], [64, 128]
        m = kv.KV_AMORTIZE_REMAP
    else:
        s0, s1, nr = [100, 10], [130, 20], [3, 40]
        m = kv.KV_AMORTIZE
    sc, sr = _stubs(dp, nr, 931)
    ws = kv.workspace(dp.desc, sum(lens) + sum(nr), 2)
    snap = _snapshot(dp)
    glens = torch.tensor(lens, dtype=torch.int32)
    kv.kv_splice(dp.desc, 2, bt, 12, glens, i32(*s0), i32(*s1), i32(*nr), sc.cuda(), sr.cuda(),
                 m, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_OVERLAP
    _unchanged(dp, snap, f"splice with a duplicated block ({mode})")
    assert np.array_equal(bt.cpu().numpy(), bt_h), "block tables were rewritten"


def test_splice_duplicate_in_unused_entry_is_not_a_finding(orc, debug_checks):
    lens = [640, 320]
    ss, dp = _splice_case("mla", lens, 12, 940)
    bt_h = ss.block_tables.copy()
    bt_h[1, 11] = bt_h[0, 3]   # sequence 1 uses entries 0..5 only
    s0, s1, nr = [100, 10], [130, 20], [3, 40]
    sc, sr = _stubs(dp, nr, 941)
    ws = kv.workspace(dp.desc, sum(lens) + sum(nr), 2)
    glens = torch.tensor(lens, dtype=torch.int32)
    kv.kv_splice(dp.desc, 2, to_dev(bt_h), 12, glens, i32(*s0), i32(*s1), i32(*nr), sc.cuda(),
                 sr.cuda(), kv.KV_AMORTIZE, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice(dp.orc, bt_h, olens, s0, s1, nr, synth.bits(sc).copy(),
                      synth.bits(sr).copy()) == O.OK
    assert glens.tolist() == olens.tolist()
    check_pool(dp, "splice with debug checks on", rot_exact=True)


def test_composed_splice_duplicate_block_is_reported(debug_checks):
    lens = [900, 700]
    ss, dp = _splice_case("gqa", lens, 16, 950)
    bt_h = ss.block_tables.copy()
    bt_h[0, 1] = bt_h[1, 10]     # entry 10 of sequence 1 holds its rows 640..703
    bt = to_dev(bt_h)
    s0 = np.array([[100, 50], [10, 5]], np.int32)
    s1 = np.array([[130, 90], [20, 8]], np.int32)
    nr = np.array([[3, 7], [9, 0]], np.int32)
    sc, sr = _stubs(dp, nr, 951)
    glens = torch.tensor(lens, dtype=torch.int32)
    ts0, ts1, tnr = (torch.from_numpy(x.copy()) for x in (s0, s1, nr))
    ws = torch.empty(kv.kv_splice_composed_workspace_size(dp.desc, glens, ts0, ts1, tnr),
                     dtype=torch.uint8, device="cuda")
    snap = _snapshot(dp)
    kv.kv_splice_composed(dp.desc, bt, 16, glens, ts0, ts1, tnr, sc.cuda(), sr.cuda(), ws)
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_OVERLAP
    _unchanged(dp, snap, "composed splice with a duplicated block")


# ---------------------------------------------------------------------------
# Patch factors addressed outside their arrays
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rank", [8, 32])   # tensor-core kernel, token-tiled kernel
def test_patch_map_outside_the_factors_is_reported(rank):
    wl = synth.relocate_workload(960, num_reqs=2, chunks_per_req=3, len_lo=20, len_hi=60,
                                 delta_lo=-500, delta_hi=500, n_pool_chunks=3, base_hi=100)
    src = DevPool("mla", 2, wl.src_slots_total, 961)
    dst = DevPool("mla", 2, wl.dst_slots_total, 962)
    dev = {k: to_dev(getattr(wl, k)) for k in
           ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta", "block_tables")}
    T, C = wl.total_tokens, wl.num_chunks
    u = torch.zeros((2, T, rank), device="cuda")
    v = torch.zeros((2, C, 576, rank), device="cuda")
    ws = kv.workspace(dst.desc, T, C)
    args = (wl.num_chunks, T, dev["tok_off"], dev["src_slots"], dev["chunk_req"],
            dev["chunk_dst_pos"], dev["delta"], dev["block_tables"], wl.block_tables.shape[0],
            wl.block_tables.shape[1])
    # U rows of chunk 1 mapped so that its last tokens fall past the U array
    u_map = torch.tensor(wl.tok_off[:-1], dtype=torch.int64, device="cuda")
    u_map[1] = T - 2
    pd = kv.patch_desc(rank, [u, u], [v[:, :, :512], v[:, :, 512:]], u_chunk_tok=u_map)
    kv.kv_relocate(src.desc, dst.desc, *args, pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_OUT_OF_RANGE
    # a V slot past the V array
    v_map = torch.arange(C, dtype=torch.int32, device="cuda")
    v_map[2] = C
    pd = kv.patch_desc(rank, [u, u], [v[:, :, :512], v[:, :, 512:]], v_chunk=v_map)
    kv.kv_relocate(src.desc, dst.desc, *args, pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_OUT_OF_RANGE
    # in range: no finding
    pd = kv.patch_desc(rank, [u, u], [v[:, :, :512], v[:, :, 512:]])
    kv.kv_relocate(src.desc, dst.desc, *args, pd, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK


# ---------------------------------------------------------------------------
# The splice kernels' timeout branch
# ---------------------------------------------------------------------------

def test_splice_kernel_timeout_branch_then_a_clean_call_matches(orc, skip_publish):
    n, s0, nr, delta = 9000, 1234, 5, -1
    s1 = s0 + nr - delta
    ss, dp = _splice_case("mla", [n], 150, 970)
    bt = to_dev(ss.block_tables)
    sc, sr = _stubs(dp, [nr], 971)
    ws = kv.workspace(dp.desc, n + nr, 1)
    pristine = dp.fused.clone()
    # ticket 0 is the first downstream tile (Δ < 0: ascending); tile 1 writes
    # one of its rows and so waits for it
    skip_publish(0)
    glens = torch.tensor([n], dtype=torch.int32)
    kv.kv_splice(dp.desc, 1, bt, 150, glens, i32(s0), i32(s1), i32(nr), sc.cuda(), sr.cuda(),
                 kv.KV_AMORTIZE, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_TIMEOUT
    # no injection: the same workspace, the pool restored, bit-exact with the oracle
    skip_publish(-1)
    dp.fused.copy_(pristine)
    glens = torch.tensor([n], dtype=torch.int32)
    kv.kv_splice(dp.desc, 1, bt, 150, glens, i32(s0), i32(s1), i32(nr), sc.cuda(), sr.cuda(),
                 kv.KV_AMORTIZE, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array([n], np.int32)
    assert orc.splice(dp.orc, ss.block_tables, olens, [s0], [s1], [nr], synth.bits(sc).copy(),
                      synth.bits(sr).copy()) == O.OK
    check_pool(dp, "splice after the injected timeout", rot_exact=True)


def test_composed_kernel_timeout_branch_then_a_clean_call_matches(orc, skip_publish):
    lens = [6000]
    ss, dp = _splice_case("mla", lens, 100, 980)
    bt = to_dev(ss.block_tables)
    s0 = np.array([[1000], [3000]], np.int32)
    s1 = np.array([[1003], [3004]], np.int32)
    nr = np.array([[2], [1]], np.int32)
    sc, sr = _stubs(dp, nr, 981)
    glens = torch.tensor(lens, dtype=torch.int32)
    ts0, ts1, tnr = (torch.from_numpy(x.copy()) for x in (s0, s1, nr))
    st, tiles, _ = kv.kv_splice_composed_plan(dp.desc, glens, ts0, ts1, tnr)
    assert st == kv.KV_OK
    # a tile that other tiles wait for
    waited = sorted({j for t in tiles for a, b in ((t["dep"][0], t["dep"][1]),
                                                   (t["dep"][2], t["dep"][3])) if a >= 0
                     for j in range(a, b + 1)})
    assert waited, "the plan has no dependency to starve"
    ws = torch.empty(kv.kv_splice_composed_workspace_size(dp.desc, glens, ts0, ts1, tnr),
                     dtype=torch.uint8, device="cuda")
    pristine = dp.fused.clone()
    skip_publish(waited[0])
    kv.kv_splice_composed(dp.desc, bt, 100, glens, ts0, ts1, tnr, sc.cuda(), sr.cuda(), ws)
    assert kv.kv_get_device_status(ws) == kv.KV_ERR_TIMEOUT
    skip_publish(-1)
    dp.fused.copy_(pristine)
    glens = torch.tensor(lens, dtype=torch.int32)
    kv.kv_splice_composed(dp.desc, bt, 100, glens, ts0, ts1, tnr, sc.cuda(), sr.cuda(), ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice_composed(dp.orc, ss.block_tables, olens, s0, s1, nr, synth.bits(sc).copy(),
                               synth.bits(sr).copy()) == O.OK
    assert glens.tolist() == olens.tolist()
    check_pool(dp, "composed splice after the injected timeout", rot_exact=True)

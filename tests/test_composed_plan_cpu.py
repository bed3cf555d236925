"""Host-side plan of the composed splice (several directives per sequence as
one in-place edit, Leyline §2.1-§2.3 with R(a)R(b) = R(a+b)), checked on the
CPU: the tiles cover exactly the rows that move or come from a stub, each
row's origin and total shift agree with a symbolic composition of the
directives, every tile waits on every earlier tile whose source rows it
overwrites (and on no later one), and running the tiles one at a time in
ticket order on a small cache reproduces the oracle's composed splice."""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth

kv.load(build_if_missing=True)


def _desc(kind, slots=1 << 20):
    d = kv.kv_pool_desc()
    d.num_layers, d.block_size, d.num_slots = 2, 64, slots
    if kind == "mla":
        d.copy_dim, d.rot_heads, d.rot_head_dim = 512, 1, 64
        d.copy_slot_stride = d.rot_slot_stride = 576
    else:
        d.copy_dim, d.rot_heads, d.rot_head_dim = 1024, 8, 128
        d.copy_slot_stride = d.rot_slot_stride = 1024
    d.copy_layer_stride = d.rot_layer_stride = slots * d.copy_slot_stride
    d.copy_base, d.rot_base = 1 << 20, 1 << 21      # never dereferenced by the planner
    d.rope_base = 10000.0
    return d


def _random_dirs(rng, lens, k, max_span, max_stub):
    cur = list(lens)
    out = []
    for _ in range(k):
        a_s, b_s, n_s = [], [], []
        for q, n in enumerate(cur):
            a = int(rng.integers(0, n + 1))
            b = int(rng.integers(a, min(n, a + max_span) + 1))
            nr = int(rng.integers(0, max_stub + 1))
            a_s.append(a)
            b_s.append(b)
            n_s.append(nr)
            cur[q] = n + nr - (b - a)
        out.append((a_s, b_s, n_s))
    return out


def _tensors(lens, dirs):
    return (torch.tensor(lens, dtype=torch.int32),
            *[torch.tensor([d[j] for d in dirs], dtype=torch.int32) for j in range(3)])


def _origins(lens, dirs):
    """Per sequence: the final rows as (kind, index, written position)."""
    first, off = {}, 0
    for i, (_, _, nrs) in enumerate(dirs):
        for q, nr in enumerate(nrs):
            first[(i, q)] = off
            off += nr
    seqs = []
    for q, n in enumerate(lens):
        seq = [("old", p, p) for p in range(n)]
        for i, (a_s, b_s, nrs) in enumerate(dirs):
            a, b, nr = a_s[q], b_s[q], nrs[q]
            seq = seq[:a] + [("stub", first[(i, q)] + k, a + k) for k in range(nr)] + seq[b:]
        seqs.append(seq)
    return seqs


def _check_plan(kind, lens, dirs):
    tl, s0, s1, nr = _tensors(lens, dirs)
    st, tiles, deltas = kv.kv_splice_composed_plan(_desc(kind), tl, s0, s1, nr)
    assert st == kv.KV_OK
    T = 32 if kind == "mla" else 8
    seqs = _origins(lens, dirs)
    covered = {}
    for t, tile in enumerate(tiles):
        assert 1 <= tile["n"] <= T
        shift = deltas[tile["unit"]] if tile["unit"] >= 0 else 0
        assert tile["unit"] < 0 or shift != 0
        for i in range(tile["n"]):
            p = tile["dst_lo"] + i
            kind_, idx, written = seqs[tile["seq"]][p]
            assert (kind_ == "stub") == bool(tile["stub"])
            assert idx == tile["src_lo"] + i
            assert p - written == shift
            key = (tile["seq"], p)
            assert key not in covered
            covered[key] = t
    for q, seq in enumerate(seqs):
        for p, (kind_, idx, written) in enumerate(seq):
            moves = kind_ == "stub" or p != written
            assert ((q, p) in covered) == moves
    # hazards: a tile waits on every other tile whose source rows it overwrites
    for t, tile in enumerate(tiles):
        deps = set()
        for r in range(2):
            lo, hi = tile["dep"][2 * r], tile["dep"][2 * r + 1]
            if lo >= 0:
                assert lo <= hi < t
                deps.update(range(lo, hi + 1))
        d0, d1 = tile["dst_lo"], tile["dst_lo"] + tile["n"]
        for u, other in enumerate(tiles):
            if u == t or other["stub"] or other["seq"] != tile["seq"]:
                continue
            if other["src_lo"] < d1 and d0 < other["src_lo"] + other["n"]:
                assert u < t, (t, u)
                assert u in deps, (t, u)
    return tiles, deltas


@pytest.mark.parametrize("kind", ["mla", "gqa"])
def test_plan_covers_moves_and_orders_hazards(kind):
    rng = np.random.default_rng(71 if kind == "mla" else 72)
    for _ in range(60):
        S = int(rng.integers(1, 4))
        lens = [int(x) for x in rng.integers(0, 400, size=S)]
        dirs = _random_dirs(rng, lens, int(rng.integers(1, 6)), 150, 90)
        _check_plan(kind, lens, dirs)


def test_plan_of_small_shifts_and_long_sequences():
    # shifts of one row in both directions inside one sequence, and a long tail
    lens = [5000]
    dirs = [([100], [101], [0]), ([2000], [2000], [3]), ([4000], [4001], [0])]
    tiles, deltas = _check_plan("mla", lens, dirs)
    assert sorted(deltas) == [-1, 1, 2]
    assert any(t["dep"][0] >= 0 for t in tiles)


def test_plan_of_a_single_directive_matches_the_splice_shape():
    tiles, deltas = _check_plan("mla", [300], [([40], [140], [7])])
    assert deltas == [-93]
    moving = [t for t in tiles if not t["stub"]]
    assert sum(t["n"] for t in moving) == 300 - 140
    assert all(a["src_lo"] < b["src_lo"] for a, b in zip(moving, moving[1:]))  # ascending


def test_plan_rejects_bad_directives_and_sizes_its_workspace():
    d = _desc("mla")
    tl, s0, s1, nr = _tensors([10], [([2], [5], [1]), ([3], [9], [0])])  # 2nd ends past 8
    st, _, _ = kv.kv_splice_composed_plan(d, tl, s0, s1, nr)
    assert st == kv.KV_ERR_INVALID_ARG
    assert kv.kv_splice_composed_workspace_size(d, tl, s0, s1, nr) == 0
    tl, s0, s1, nr = _tensors([10], [([2], [5], [1])])
    assert kv.kv_splice_composed_workspace_size(d, tl, s0, s1, nr) > 0
    # argument errors come back before any device work, on a CPU-only box too:
    # 100 rows do not fit one 64-row block
    lens = torch.tensor([100], dtype=torch.int32)
    assert kv.kv_splice_composed(d, 0x1000, 1, lens, s0, s1, nr, None, None, None,
                                 check=False) == kv.KV_ERR_CAPACITY
    assert lens.tolist() == [100]


def test_running_the_plan_tile_by_tile_matches_the_oracle():
    # execute the tiles in ticket order on a small MLA-shaped cache (c_KV cut
    # to 8 values, k_pe 64 rotated with the oracle's own R): the in-place
    # result must equal the oracle's composed splice
    orc = O.get()
    rng = np.random.default_rng(81)
    for trial in range(6):
        lens = [int(x) for x in rng.integers(60, 300, size=2)]
        dirs = _random_dirs(rng, lens, int(rng.integers(2, 5)), 70, 50)
        final = []
        for q, n in enumerate(lens):
            for a_s, b_s, nrs in dirs:
                n = n + nrs[q] - (b_s[q] - a_s[q])
            final.append(n)
        maxb = (max(max(lens), max(final)) + 63) // 64 + 1
        ss = synth.splice_seqs(82 + trial, [0] * len(lens), maxb)
        L, cd, rd = 2, 8, 64
        cp = synth.bits(synth.bf16_normal((L, ss.num_slots, cd), 83 + trial)).copy()
        rt = synth.bits(synth.bf16_normal((L, ss.num_slots, rd), 84 + trial)).copy()
        tot = sum(sum(nrs) for _, _, nrs in dirs)
        sc = synth.bits(synth.bf16_normal((L, max(tot, 1), cd), 85 + trial)).copy()[:, :tot]
        sr = synth.bits(synth.bf16_normal((L, max(tot, 1), rd), 86 + trial)).copy()[:, :tot]
        sc, sr = np.ascontiguousarray(sc), np.ascontiguousarray(sr)
        # the oracle
        pool = O.Pool(cp.copy(), rt.copy(), 64, 1, rd, 10000.0)
        seq = np.array(lens, np.int32)
        s0 = np.array([d[0] for d in dirs], np.int32)
        s1 = np.array([d[1] for d in dirs], np.int32)
        nr = np.array([d[2] for d in dirs], np.int32)
        assert orc.splice_composed(pool, ss.block_tables, seq, s0, s1, nr, sc, sr) == O.OK
        # the plan, run tile by tile
        tl, t0, t1, tn = _tensors(lens, dirs)
        st, tiles, deltas = kv.kv_splice_composed_plan(_desc("mla"), tl, t0, t1, tn)
        assert st == kv.KV_OK
        c2, r2 = cp.copy(), rt.copy()
        slot = lambda q, p: int(ss.block_tables[q, p // 64]) * 64 + p % 64
        for tile in tiles:
            q, n = tile["seq"], tile["n"]
            shift = deltas[tile["unit"]] if tile["unit"] >= 0 else 0
            if tile["stub"]:
                rows = [(sc[:, tile["src_lo"] + i].copy(), sr[:, tile["src_lo"] + i].copy())
                        for i in range(n)]
            else:
                rows = [(c2[:, slot(q, tile["src_lo"] + i)].copy(),
                         r2[:, slot(q, tile["src_lo"] + i)].copy()) for i in range(n)]
            for i, (rc, rr) in enumerate(rows):
                s = slot(q, tile["dst_lo"] + i)
                c2[:, s] = rc
                for l in range(L):
                    r2[l, s] = orc.rotate_bf16(rr[l], shift, 10000.0) if shift else rr[l]
        assert seq.tolist() == final
        assert np.array_equal(c2, pool.copy) and np.array_equal(r2, pool.rot)

"""GPU parity of the composed splice (several directives per sequence applied
as one in-place edit: every row moved once, turned by its total shift,
rounded once; Leyline §2.1-§2.3 with R(a)R(b) = R(a+b)) against the fp64
oracle's composed mode, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, check_exact, check_pool, to_dev

pytestmark = pytest.mark.gpu

L = 3


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _pool(shape, lens, max_blocks, seed, layers=L):
    ss = synth.splice_seqs(seed, lens, max_blocks, spare_blocks=3)
    dp = DevPool(shape, layers, ss.num_slots, seed)
    return ss, dp, to_dev(ss.block_tables)


def _random_rounds(seed, lens, rounds, span_hi, stub_hi):
    cur = np.asarray(lens, np.int32)
    s0, s1, nr = [], [], []
    for r in range(rounds):
        d = synth.random_directives(seed + r, cur, 0, span_hi, 0, stub_hi)
        s0.append(d.s_start)
        s1.append(d.s_end)
        nr.append(d.stub_len)
        cur = cur + d.stub_len - (d.s_end - d.s_start)
    return np.stack(s0), np.stack(s1), np.stack(nr)


def _composed_both(orc, ss, dp, bt, lens, s0, s1, nr, seed, layers=L):
    s0, s1, nr = (np.ascontiguousarray(x, dtype=np.int32) for x in (s0, s1, nr))
    tot = int(nr.sum())
    sc = synth.bf16_normal((layers, tot, dp.cd), seed)
    sr = synth.bf16_normal((layers, tot, dp.H * dp.d), seed + 1)
    glens = torch.tensor(lens, dtype=torch.int32)
    ts0, ts1, tnr = (torch.from_numpy(x.copy()) for x in (s0, s1, nr))
    n = kv.kv_splice_composed_workspace_size(dp.desc, glens, ts0, ts1, tnr)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    kv.kv_splice_composed(dp.desc, bt, ss.block_tables.shape[1], glens, ts0, ts1, tnr,
                          sc.cuda() if tot else None, sr.cuda() if tot else None, ws)
    st = kv.kv_get_device_status(ws)
    olens = np.array(lens, np.int32)
    assert orc.splice_composed(dp.orc, ss.block_tables, olens, s0, s1, nr,
                               synth.bits(sc).copy() if tot else None,
                               synth.bits(sr).copy() if tot else None) == O.OK
    assert glens.tolist() == olens.tolist()
    return st


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_composed_random_directives_match_oracle(orc, shape):
    lens = [0, 1, 63, 64, 65, 700, 1500, 2900]
    s0, s1, nr = _random_rounds(400 + len(shape), lens, 4, 700, 600)
    ss, dp, bt = _pool(shape, lens, 96, 410 + len(shape))
    assert _composed_both(orc, ss, dp, bt, lens, s0, s1, nr, 420) == kv.KV_OK
    stats = check_pool(dp, f"composed splice {shape}")
    assert stats["exact"] >= stats["values"] - max(3, stats["values"] // 100000), stats


def test_composed_small_shifts_both_ways_over_a_long_sequence(orc):
    # shifts of -1, +1 and +2 in one edit: neighbouring tiles wait on each other
    lens = [6000]
    s0 = np.array([[100], [3000], [5000]])
    s1 = np.array([[101], [3000], [5000]])
    nr = np.array([[0], [2], [1]])
    ss, dp, bt = _pool("mla", lens, 96, 430)
    assert _composed_both(orc, ss, dp, bt, lens, s0, s1, nr, 431) == kv.KV_OK
    check_pool(dp, "composed small shifts")


def test_composed_single_directive_equals_kv_splice(orc):
    lens = [900, 2500, 40]
    d = synth.random_directives(440, np.asarray(lens, np.int32), 0, 800, 0, 500)
    ss, a, bt = _pool("mla", lens, 64, 441)
    _, b, _ = _pool("mla", lens, 64, 441)
    tot = int(d.stub_len.sum())
    sc = synth.bf16_normal((L, tot, 512), 442).cuda()
    sr = synth.bf16_normal((L, tot, 64), 443).cuda()
    la, lb = torch.tensor(lens, dtype=torch.int32), torch.tensor(lens, dtype=torch.int32)
    args = [torch.from_numpy(x.copy()) for x in (d.s_start, d.s_end, d.stub_len)]
    ws = kv.workspace(a.desc, sum(lens) + tot, len(lens))
    kv.kv_splice(a.desc, len(lens), bt, 64, la, *args, sc, sr, kv.KV_AMORTIZE, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    args2 = [x.reshape(1, -1).contiguous() for x in args]
    ws2 = torch.empty(kv.kv_splice_composed_workspace_size(b.desc, lb, *args2),
                      dtype=torch.uint8, device="cuda")
    kv.kv_splice_composed(b.desc, bt, 64, lb, *args2, sc, sr, ws2)
    assert kv.kv_get_device_status(ws2) == kv.KV_OK
    assert la.tolist() == lb.tolist()
    ga, gb = a.gpu_bits(), b.gpu_bits()
    check_exact(gb[0], ga[0], "verbatim part")
    check_exact(gb[1], ga[1], "rotary part")


def test_composed_insert_then_remove_moves_nothing(orc):
    lens = [500]
    ss, dp, bt = _pool("mla", lens, 16, 450)
    before = dp.gpu_bits()
    assert _composed_both(orc, ss, dp, bt, lens, [[200], [200]], [[200], [230]], [[30], [0]],
                          451) == kv.KV_OK
    assert kv.kv_last_launch_count() == 0
    after = dp.gpu_bits()
    check_exact(after[0], before[0], "verbatim part")
    check_exact(after[1], before[1], "rotary part")


def test_composed_many_sequences_in_one_call(orc):
    rng = np.random.default_rng(460)
    lens = [int(x) for x in rng.integers(0, 400, size=70)]
    s0, s1, nr = _random_rounds(461, lens, 3, 200, 120)
    ss, dp, bt = _pool("gqa", lens, 16, 462)
    assert _composed_both(orc, ss, dp, bt, lens, s0, s1, nr, 463) == kv.KV_OK
    check_pool(dp, "composed splice, 70 sequences")

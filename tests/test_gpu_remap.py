"""GPU parity of the block-aligned splice by block-table remapping
(KV_AMORTIZE_REMAP): a directive whose span and stub are whole blocks moves
the downstream rows by permuting the sequence's block-table row and turning
their rotary part in place.  The logical sequence read through the new row
must equal the oracle's AMORTIZE splice read through the old one, bit for bit
(Leyline §2.1-§2.3)."""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, check_exact, to_dev

pytestmark = pytest.mark.gpu

L = 3
B = 64


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _logical(bits_c, bits_r, bt_row, n):
    slots = np.array([int(bt_row[p // B]) * B + p % B for p in range(n)], np.int64)
    return bits_c[:, slots], bits_r[:, slots]


def _run(orc, shape, lens, s0, s1, nr, max_blocks, seed):
    ss = synth.splice_seqs(seed, lens, max_blocks, spare_blocks=3)
    dp = DevPool(shape, L, ss.num_slots, seed)
    bt = to_dev(ss.block_tables)
    tot = int(np.sum(nr))
    sc = synth.bf16_normal((L, tot, dp.cd), seed + 1)
    sr = synth.bf16_normal((L, tot, dp.H * dp.d), seed + 2)
    glens = torch.tensor(lens, dtype=torch.int32)
    ws = kv.workspace(dp.desc, sum(lens) + tot, len(lens))
    kv.kv_splice(dp.desc, len(lens), bt, max_blocks, glens,
                 torch.tensor(s0, dtype=torch.int32), torch.tensor(s1, dtype=torch.int32),
                 torch.tensor(nr, dtype=torch.int32), sc.cuda() if tot else None,
                 sr.cuda() if tot else None, kv.KV_AMORTIZE_REMAP, ws)
    assert kv.kv_get_device_status(ws) == kv.KV_OK
    olens = np.array(lens, np.int32)
    assert orc.splice(dp.orc, ss.block_tables, olens, s0, s1, nr,
                      synth.bits(sc).copy() if tot else None,
                      synth.bits(sr).copy() if tot else None) == O.OK
    assert glens.tolist() == olens.tolist()
    new_bt = bt.cpu().numpy()
    gc, gr = dp.gpu_bits()
    for q in range(len(lens)):
        assert sorted(new_bt[q].tolist()) == sorted(ss.block_tables[q].tolist())
        aligned = s0[q] % B == 0 and s1[q] % B == 0 and nr[q] % B == 0
        if not (aligned and nr[q] != s1[q] - s0[q]):
            assert np.array_equal(new_bt[q], ss.block_tables[q])   # data-moving path
        n = int(olens[q])
        wc, wr = _logical(dp.orc.copy, dp.orc.rot, ss.block_tables[q], n)
        hc, hr = _logical(gc, gr, new_bt[q], n)
        check_exact(hc, wc, f"sequence {q}: verbatim part")
        check_exact(hr, wr, f"sequence {q}: rotary part")
    return ss, new_bt


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_remap_equals_amortize_logically(orc, shape):
    # aligned shrinking, aligned growing, aligned with a ragged tail, an
    # unaligned directive (data-moving path) and a Δ = 0 one
    lens = [1000, 2000, 777, 900, 640]
    s0 = [128, 64, 256, 100, 64]
    s1 = [512, 192, 320, 300, 192]
    nr = [64, 448, 0, 30, 128]
    ss, new_bt = _run(orc, shape, lens, s0, s1, nr, 48, 500 + len(shape))
    assert not np.array_equal(new_bt[0], ss.block_tables[0])
    assert not np.array_equal(new_bt[1], ss.block_tables[1])


def test_remap_successive_directives(orc):
    # the device block table evolves from call to call; the logical contents
    # must follow the oracle's successive AMORTIZE splices
    lens = [3000, 1500]
    ss = synth.splice_seqs(510, lens, 80, spare_blocks=2)
    dp = DevPool("mla", L, ss.num_slots, 510)
    bt = to_dev(ss.block_tables)
    glens = torch.tensor(lens, dtype=torch.int32)
    olens = np.array(lens, np.int32)
    rounds = [([640, 0], [1280, 128], [64, 256]),       # aligned: shrink / grow
              ([64, 1024], [64, 1280], [192, 0]),      # pure insertion / removal
              ([100, 64], [200, 192], [3, 64])]        # unaligned / aligned
    ws = kv.workspace(dp.desc, 4000, 2)
    for r, (s0, s1, nr) in enumerate(rounds):
        tot = sum(nr)
        sc = synth.bf16_normal((L, tot, 512), 520 + r)
        sr = synth.bf16_normal((L, tot, 64), 530 + r)
        kv.kv_splice(dp.desc, 2, bt, 80, glens, torch.tensor(s0, dtype=torch.int32),
                     torch.tensor(s1, dtype=torch.int32), torch.tensor(nr, dtype=torch.int32),
                     sc.cuda(), sr.cuda(), kv.KV_AMORTIZE_REMAP, ws)
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        assert orc.splice(dp.orc, ss.block_tables, olens, s0, s1, nr, synth.bits(sc).copy(),
                          synth.bits(sr).copy()) == O.OK
        assert glens.tolist() == olens.tolist()
        new_bt = bt.cpu().numpy()
        gc, gr = dp.gpu_bits()
        for q in range(2):
            n = int(olens[q])
            wc, wr = _logical(dp.orc.copy, dp.orc.rot, ss.block_tables[q], n)
            hc, hr = _logical(gc, gr, new_bt[q], n)
            check_exact(hc, wc, f"round {r}, sequence {q}: verbatim part")
            check_exact(hr, wr, f"round {r}, sequence {q}: rotary part")

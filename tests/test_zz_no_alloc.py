"""kv_relocate_noalloc: relocation for callers that cannot allocate device
memory (their device memory is owned by a host runtime's allocator, or an
allocation and its synchronisation would stall a latency-critical path).
It takes no workspace; its scratch is a fixed device array inside the
library.

Its output is compared element by element with the fp64 oracle, and with
kv_relocate's (the same kernels on a caller's workspace: equal bit for bit),
on two calls in a row -- every call reuses the same scratch -- with and
without a patch, and at the largest chunk counts the built-in table holds.

Kept in a file that pytest collects last, so a run that stops at the first
failure has run every other test before this one; it also passes alone in a
fresh process.
"""
import numpy as np
import pytest
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, check_exact, check_pool, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return O.get()


def _case(shape, seed, layers=3, num_reqs=4, chunks=5, lo=1, hi=130):
    wl = synth.relocate_workload(seed, num_reqs=num_reqs, chunks_per_req=chunks, len_lo=lo,
                                 len_hi=hi, delta_lo=-32768, delta_hi=32768, n_pool_chunks=7,
                                 base_hi=200)
    src = DevPool(shape, layers, wl.src_slots_total, seed)
    dev = {k: to_dev(getattr(wl, k)) for k in
           ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta", "block_tables")}
    return wl, src, dev


def _args(wl, dev):
    return (wl.num_chunks, wl.total_tokens, dev["tok_off"], dev["src_slots"], dev["chunk_req"],
            dev["chunk_dst_pos"], dev["delta"], dev["block_tables"], wl.block_tables.shape[0],
            wl.block_tables.shape[1])


def _oracle(orc, wl, src, dst, patch=None):
    assert orc.relocate(src.orc, dst.orc, wl.tok_off, wl.src_slots, wl.chunk_req,
                        wl.chunk_dst_pos, wl.delta, wl.block_tables, patch) == O.OK


def _same_bits(a: DevPool, b: DevPool, what: str):
    ac, ar = a.gpu_bits()
    bc, br = b.gpu_bits()
    check_exact(ac, bc, what + " (verbatim part)")
    check_exact(ar, br, what + " (rotary part)")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_noalloc_matches_oracle_and_workspace_relocate_on_two_calls(orc, shape):
    for call, seed in enumerate((700, 701)):
        layers = 3
        wl, src, dev = _case(shape, seed + (10 if shape == "gqa" else 0), layers=layers)
        got = DevPool(shape, layers, wl.dst_slots_total, seed + 50)
        want = DevPool(shape, layers, wl.dst_slots_total, seed + 50)
        st, dev_status = kv.kv_relocate_noalloc(src.desc, got.desc, *_args(wl, dev), None)
        assert st == kv.KV_OK and dev_status == kv.KV_OK
        _oracle(orc, wl, src, got)
        check_pool(got, f"{shape} call {call} vs oracle", rot_exact=True)
        ws = kv.workspace(want.desc, wl.total_tokens, wl.num_chunks)
        kv.kv_relocate(src.desc, want.desc, *_args(wl, dev), None, ws)
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        _same_bits(got, want, f"{shape} call {call} vs kv_relocate")


def test_noalloc_patched_gqa_rank16_on_the_tensor_cores(orc):
    layers, m = 2, 16
    for call, seed in enumerate((730, 731)):
        wl, src, dev = _case("gqa", seed, layers=layers, lo=50, hi=300)
        got = DevPool("gqa", layers, wl.dst_slots_total, seed + 5)
        want = DevPool("gqa", layers, wl.dst_slots_total, seed + 5)
        us = [synth.f32_normal((layers, wl.total_tokens, m), seed + 10 + i, std=0.02)
              for i in range(2)]
        vs = [synth.f32_normal((layers, wl.num_chunks, 1024, m), seed + 20 + i, std=0.02)
              for i in range(2)]
        pd = kv.patch_desc(m, [x.cuda() for x in us], [x.cuda() for x in vs])
        st, dev_status = kv.kv_relocate_noalloc(src.desc, got.desc, *_args(wl, dev), pd)
        assert st == kv.KV_OK and dev_status == kv.KV_OK
        _oracle(orc, wl, src, got, O.Patch(m, [x.numpy() for x in us], [x.numpy() for x in vs]))
        check_pool(got, f"patched gqa call {call} vs oracle", copy_exact=False)
        ws = kv.workspace(want.desc, wl.total_tokens, wl.num_chunks)
        kv.kv_relocate(src.desc, want.desc, *_args(wl, dev), pd, ws)
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        _same_bits(got, want, f"patched gqa call {call} vs kv_relocate")


@pytest.mark.parametrize("shape,limit,reqs", [("mla", 4095, 5), ("gqa", 2047, 23)])
def test_noalloc_accepts_the_largest_call_and_rejects_one_more(orc, shape, limit, reqs):
    # one-token chunks: as many cos/sin rows as the built-in table holds
    wl, src, dev = _case(shape, 740, layers=2, num_reqs=reqs, chunks=limit // reqs, lo=1, hi=1)
    assert wl.num_chunks == limit
    dst = DevPool(shape, 2, wl.dst_slots_total, 741)
    st, dev_status = kv.kv_relocate_noalloc(src.desc, dst.desc, *_args(wl, dev), None)
    assert st == kv.KV_OK and dev_status == kv.KV_OK
    _oracle(orc, wl, src, dst)
    check_pool(dst, f"{shape} at {limit} chunks", rot_exact=True)
    # one chunk more than the table holds: rejected before anything is enqueued
    n = limit + 1
    tok_off = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    zeros = torch.zeros(n, dtype=torch.int32, device="cuda")
    st, _ = kv.kv_relocate_noalloc(src.desc, dst.desc, n, n, tok_off, zeros, zeros, zeros, zeros,
                                   dev["block_tables"], wl.block_tables.shape[0],
                                   wl.block_tables.shape[1], None, check=False)
    assert st == kv.KV_ERR_WORKSPACE


def test_noalloc_status_is_per_call(orc):
    wl, src, dev = _case("mla", 720)
    dst = DevPool("mla", 3, wl.dst_slots_total, 721)
    bad = wl.src_slots.copy()
    bad[0] = wl.src_slots_total
    bad_dev = dict(dev, src_slots=to_dev(bad))
    st, dev_status = kv.kv_relocate_noalloc(src.desc, dst.desc, *_args(wl, bad_dev), None)
    assert st == kv.KV_OK and dev_status == kv.KV_ERR_OUT_OF_RANGE
    # the next call starts from a cleared status word and is correct
    st, dev_status = kv.kv_relocate_noalloc(src.desc, dst.desc, *_args(wl, dev), None)
    assert st == kv.KV_OK and dev_status == kv.KV_OK
    _oracle(orc, wl, src, dst)
    check_pool(dst, "after a failed call", rot_exact=True)

"""kv_relocate_noalloc: relocation for callers that cannot allocate device
memory (their device memory is owned by a host runtime's allocator, or an
allocation and its synchronisation would stall a latency-critical path).
It takes no workspace; its scratch is a fixed device array inside the
library.  Its output must match kv_relocate's, call after call, even though
every call reuses the same scratch.

Kept in a file that pytest collects last, so a run that stops at the first
failure has run every other test before this one; it also passes alone in a
fresh process.
"""
import numpy as np
import pytest
import torch

import position_independent_mla_gb300 as kv
import synth
from _gpu import DevPool, check_exact, check_ulp, to_dev

pytestmark = pytest.mark.gpu


def _case(shape, seed, layers=3, num_reqs=4, chunks=5):
    wl = synth.relocate_workload(seed, num_reqs=num_reqs, chunks_per_req=chunks, len_lo=1,
                                 len_hi=130, delta_lo=-32768, delta_hi=32768, n_pool_chunks=7,
                                 base_hi=200)
    src = DevPool(shape, layers, wl.src_slots_total, seed)
    dev = {k: to_dev(getattr(wl, k)) for k in
           ("tok_off", "src_slots", "chunk_req", "chunk_dst_pos", "delta", "block_tables")}
    return wl, src, dev


def _args(wl, dev):
    return (wl.num_chunks, wl.total_tokens, dev["tok_off"], dev["src_slots"], dev["chunk_req"],
            dev["chunk_dst_pos"], dev["delta"], dev["block_tables"], wl.block_tables.shape[0],
            wl.block_tables.shape[1])


def _compare(a: DevPool, b: DevPool, what: str):
    ac, ar = a.gpu_bits()
    bc, br = b.gpu_bits()
    check_exact(ac, bc, what + " (verbatim part)")
    check_ulp(ar, br, what + " (rotary part)")


@pytest.mark.parametrize("shape", ["mla", "gqa"])
def test_noalloc_matches_workspace_relocate_on_two_calls(shape):
    for call, seed in enumerate((700, 701)):
        wl, src, dev = _case(shape, seed + (10 if shape == "gqa" else 0))
        want = DevPool(shape, 3, wl.dst_slots_total, seed + 50)
        got = DevPool(shape, 3, wl.dst_slots_total, seed + 50)
        ws = kv.workspace(want.desc, wl.total_tokens, wl.num_chunks)
        kv.kv_relocate(src.desc, want.desc, *_args(wl, dev), None, ws)
        assert kv.kv_get_device_status(ws) == kv.KV_OK
        st, dev_status = kv.kv_relocate_noalloc(src.desc, got.desc, *_args(wl, dev), None)
        assert st == kv.KV_OK and dev_status == kv.KV_OK
        _compare(got, want, f"{shape} call {call}")


def test_noalloc_status_is_per_call_and_limit_is_enforced():
    wl, src, dev = _case("mla", 720)
    dst = DevPool("mla", 3, wl.dst_slots_total, 721)
    bad = wl.src_slots.copy()
    bad[0] = wl.src_slots_total
    bad_dev = dict(dev, src_slots=to_dev(bad))
    st, dev_status = kv.kv_relocate_noalloc(src.desc, dst.desc, *_args(wl, bad_dev), None)
    assert st == kv.KV_OK and dev_status == kv.KV_ERR_OUT_OF_RANGE
    # the next call starts from a cleared status word
    st, dev_status = kv.kv_relocate_noalloc(src.desc, dst.desc, *_args(wl, dev), None)
    assert st == kv.KV_OK and dev_status == kv.KV_OK
    # more chunks than the built-in table holds (4095 for MLA rows): rejected up front
    n = 4096
    tok_off = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    zeros = torch.zeros(n, dtype=torch.int32, device="cuda")
    st, _ = kv.kv_relocate_noalloc(src.desc, dst.desc, n, n, tok_off, zeros, zeros, zeros, zeros,
                                   dev["block_tables"], wl.block_tables.shape[0],
                                   wl.block_tables.shape[1], None, check=False)
    assert st == kv.KV_ERR_WORKSPACE

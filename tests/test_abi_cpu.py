"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes as C
import os
import re
import subprocess

import pytest
import torch

import position_independent_mla_gb300 as kv
from position_independent_mla_gb300 import build as kbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvreloc.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kv.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ("kv_relocate", "kv_splice", "kv_patch", "kv_workspace_size",
              "kv_get_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kv_[a-z_0-9]+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib, n)


def test_status_strings_and_version(lib):
    assert kv.status_string(kv.KV_OK) == "ok"
    assert kv.status_string(kv.KV_ERR_TIMEOUT) == "bounded wait ran out"
    assert kv.kv_version() >= 100


def _fake_pool(copy_dim=512, heads=1, hd=64, slots=128, block=64, base=10000.0, addr=1 << 20,
               layers=2):
    # device addresses are never dereferenced by the host-side checks
    return kv.kv_pool_desc(layers, block, slots, addr, slots * 576, 576, copy_dim, addr + 1024,
                           slots * 576, 576, heads, hd, base)


def test_workspace_size_rules(lib):
    p = _fake_pool()
    n = kv.kv_workspace_size(p, 1000, 4)
    assert n > 256 and n % 256 == 0
    assert kv.kv_workspace_size(p, 100000, 4) > n
    assert kv.kv_workspace_size(_fake_pool(slots=100), 10, 1) == 0      # not whole blocks
    assert kv.kv_workspace_size(_fake_pool(hd=40), 10, 1) == 0          # head dim % 16
    assert kv.kv_workspace_size(_fake_pool(addr=(1 << 20) + 8), 10, 1) == 0  # misaligned


def test_host_checks_reject_before_any_launch(lib):
    p = _fake_pool()
    ws = C.c_void_p(1 << 24)
    # NULL pool
    assert lib.kv_relocate(None, C.byref(p), 1, 10, None, None, None, None, None, None, 1, 1,
                           None, ws, 1 << 20, None) == kv.KV_ERR_INVALID_ARG
    # shape mismatch between source and destination
    q = _fake_pool(base=500000.0)
    assert lib.kv_relocate(C.byref(p), C.byref(q), 1, 10, None, None, None, None, None, None, 1,
                           1, None, ws, 1 << 20, None) == kv.KV_ERR_INVALID_ARG
    # a row shape without a compiled kernel
    r = _fake_pool(copy_dim=256, heads=2)
    assert lib.kv_relocate(C.byref(r), C.byref(r), 1, 10, None, None, None, None, None, None, 1,
                           1, None, ws, 1 << 20, None) == kv.KV_ERR_UNSUPPORTED
    # missing index arrays
    assert lib.kv_relocate(C.byref(p), C.byref(p), 1, 10, None, None, None, None, None, None, 1,
                           1, None, ws, 1 << 20, None) == kv.KV_ERR_INVALID_ARG
    # bad patch rank
    d = kv.kv_patch_desc()
    d.rank = 6
    assert lib.kv_patch(C.byref(p), 1, 10, C.c_void_p(256), C.c_void_p(256), C.c_void_p(256),
                        C.c_void_p(256), 1, 1, C.byref(d), ws, 1 << 20,
                        None) == kv.KV_ERR_INVALID_ARG


def test_splice_host_checks_and_forget(lib):
    p = _fake_pool()
    i32 = lambda *v: torch.tensor(v, dtype=torch.int32)
    lens = i32(100, 50)
    # s_end beyond seq_len
    assert kv.kv_splice(p, 2, None, 4, lens, i32(0, 0), i32(101, 5), i32(0, 0), None, None,
                        kv.KV_AMORTIZE, None, check=False) == kv.KV_ERR_INVALID_ARG
    # capacity: 100 + 200 - 10 tokens need 5 blocks of 64, only 4 given
    assert kv.kv_splice(p, 2, C.c_void_p(256), 4, lens, i32(0, 0), i32(10, 5), i32(200, 0),
                        C.c_void_p(256), C.c_void_p(256), kv.KV_AMORTIZE, None,
                        check=False) == kv.KV_ERR_CAPACITY
    assert lens.tolist() == [100, 50]
    # FORGET moves nothing and needs no device: it truncates to s_start
    assert kv.kv_splice(p, 2, None, 4, lens, i32(30, 7), i32(40, 9), i32(3, 1), None, None,
                        kv.KV_FORGET, None) == kv.KV_OK
    assert lens.tolist() == [30, 7]
    assert kv.kv_last_launch_count() == 0


def test_workspace_checks(lib):
    p = _fake_pool()
    # misaligned workspace
    assert lib.kv_check_wait_timeout(C.c_void_p((1 << 24) + 16), 1 << 20, 1000,
                                     None) == kv.KV_ERR_WORKSPACE
    # too small
    assert lib.kv_check_wait_timeout(C.c_void_p(1 << 24), 64, 1000, None) == kv.KV_ERR_WORKSPACE


def test_cdc_host_checks(lib):
    ws = torch.empty(1 << 12, dtype=torch.uint8)
    assert kv.kv_cdc_workspace_size(-1) == 0
    assert kv.kv_cdc_workspace_size(0) == 256
    assert kv.kv_cdc_workspace_size(1 << 20) > kv.kv_cdc_workspace_size(1 << 10) > 256
    # negative stream count, missing offsets, tokens without streams
    assert kv.kv_cdc(-1, None, 0, None, 0, 0, 0, 0, None, None, None, ws,
                     check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_cdc(1, None, 10, C.c_void_p(256), 0, 0, 0, 10, C.c_void_p(256),
                     C.c_void_p(256), C.c_void_p(256), ws, check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_cdc(0, C.c_void_p(256), 10, C.c_void_p(256), 0, 0, 0, 10, C.c_void_p(256),
                     C.c_void_p(256), C.c_void_p(256), ws, check=False) == kv.KV_ERR_INVALID_ARG
    # workspace too small for the token count
    small = C.c_void_p(1 << 24)
    assert lib.kv_cdc(1, C.c_void_p(256), 1 << 20, C.c_void_p(256), 0, 0, 0, 10,
                      C.c_void_p(256), C.c_void_p(256), C.c_void_p(256), small, 256,
                      None) == kv.KV_ERR_WORKSPACE
    assert kv.kv_fingerprint(3, None, None, 10, None, 0, None, ws,
                             check=False) == kv.KV_ERR_INVALID_ARG


def test_misaligned_index_arrays_are_rejected(lib):
    p = _fake_pool()
    ws = C.c_void_p(1 << 24)
    ok4, bad4 = C.c_void_p(1 << 20), C.c_void_p((1 << 20) + 2)
    # an int32 index array not on a 4-byte boundary
    for i in range(6):
        args = [ok4] * 6
        args[i] = bad4
        tok_off, src_slots, chunk_req, chunk_dst_pos, delta, bt = args
        assert lib.kv_relocate(C.byref(p), C.byref(p), 1, 10, tok_off, src_slots, chunk_req,
                               chunk_dst_pos, delta, bt, 1, 1, None, ws, 1 << 20,
                               None) == kv.KV_ERR_INVALID_ARG
    # kv_cdc: int64 offsets, int32 tokens
    ws_t = torch.empty(1 << 12, dtype=torch.uint8)
    assert kv.kv_cdc(1, C.c_void_p((1 << 20) + 4), 10, ok4, 0, 0, 0, 10, ok4, ok4, ok4, ws_t,
                     check=False) == kv.KV_ERR_INVALID_ARG
    assert kv.kv_fingerprint(2, ok4, ok4, 10, bad4, 0, ok4, ws_t,
                             check=False) == kv.KV_ERR_INVALID_ARG


def test_debug_checks_need_their_bitmap(lib):
    """With the debug checks on, a relocation inside one pool and a splice need
    the bitmap part of the workspace (one bit per slot); kv_workspace_size
    always includes it.  Only rejections are exercised here: nothing reaches
    the device."""
    slots = 1 << 20
    p = _fake_pool(slots=slots)
    assert kv.kv_workspace_size(p, 1000, 4) >= slots // 8
    assert kv.status_string(kv.KV_ERR_OVERLAP).startswith("overlapping")
    ws = C.c_void_p(1 << 24)
    a = C.c_void_p(256)
    exact = 256 + 512            # header + cos/sin table of one 64-dim chunk
    kv.kv_set_debug_checks(True)
    try:
        assert lib.kv_relocate(C.byref(p), C.byref(p), 1, 10, a, a, a, a, a, a, 1, 1, None, ws,
                               exact, None) == kv.KV_ERR_WORKSPACE
        i32 = lambda *v: torch.tensor(v, dtype=torch.int32)
        lens = i32(100)
        # header + table + three tiles' counters: enough without the checks
        assert kv.kv_splice(p, 1, a, 4, lens, i32(10), i32(20), i32(0), None, None,
                            kv.KV_AMORTIZE, torch.empty(0, dtype=torch.uint8), check=False) \
            == kv.KV_ERR_WORKSPACE
        assert lib.kv_splice(C.byref(p), 1, a, 4, lens.data_ptr(), i32(10).data_ptr(),
                             i32(20).data_ptr(), i32(0).data_ptr(), None, None, kv.KV_AMORTIZE,
                             ws, 256 + 512 + 256, None) == kv.KV_ERR_WORKSPACE
        assert lens.tolist() == [100]
    finally:
        kv.kv_set_debug_checks(False)


def test_patch_extents_are_validated_on_the_host(lib):
    p = _fake_pool()
    d = kv.kv_patch_desc()
    d.rank = 8
    d.u[0] = d.u[1] = 1 << 20
    d.v[0] = d.v[1] = 1 << 21
    d.u_rows[0] = -1
    assert lib.kv_patch(C.byref(p), 1, 10, C.c_void_p(256), C.c_void_p(256), C.c_void_p(256),
                        C.c_void_p(256), 1, 1, C.byref(d), C.c_void_p(1 << 24), 1 << 20,
                        None) == kv.KV_ERR_INVALID_ARG

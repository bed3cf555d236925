"""Python binding of ``libkvreloc.so`` -- GB300 KV relocation / splice / patch.

Argument marshalling only: every step of the data path runs in the CUDA
kernels behind the C ABI (``include/kvreloc.h``).  PyTorch provides device
memory and streams.  There is no CPU fallback: if the compiled library is
missing, importing the binding's entry points raises.

    kv_relocate(src, dst, ...)   gather + R(δ) rotation (+ fused rank-m patch)
    kv_splice(pool, ...)         in-place Leyline AMORTIZE / FORGET directive
    kv_splice_composed(pool, ...) several directives per sequence as one edit
    kv_patch(pool, ...)          in-place rank-m patch U_m V_mᵀ
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_OUT_OF_RANGE, KV_ERR_CAPACITY = 0, 1, 2, 3
KV_ERR_WORKSPACE, KV_ERR_TIMEOUT, KV_ERR_CUDA, KV_ERR_UNSUPPORTED = 4, 5, 6, 7
KV_ERR_OVERLAP = 8
KV_AMORTIZE, KV_FORGET, KV_AMORTIZE_REMAP = 0, 1, 2

LIB_PATH = _build.LIB


class KVError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class kv_pool_desc(C.Structure):
    _fields_ = [
        ("num_layers", C.c_int32),
        ("block_size", C.c_int32),
        ("num_slots", C.c_int64),
        ("copy_base", C.c_void_p),
        ("copy_layer_stride", C.c_int64),
        ("copy_slot_stride", C.c_int64),
        ("copy_dim", C.c_int32),
        ("rot_base", C.c_void_p),
        ("rot_layer_stride", C.c_int64),
        ("rot_slot_stride", C.c_int64),
        ("rot_heads", C.c_int32),
        ("rot_head_dim", C.c_int32),
        ("rope_base", C.c_double),
        ("pair_convention", C.c_int32),
    ]


class kv_patch_desc(C.Structure):
    _fields_ = [
        ("rank", C.c_int32),
        ("u", C.c_void_p * 2),
        ("u_layer_stride", C.c_int64 * 2),
        ("u_tok_stride", C.c_int64 * 2),
        ("v", C.c_void_p * 2),
        ("v_layer_stride", C.c_int64 * 2),
        ("v_chunk_stride", C.c_int64 * 2),
        ("v_col_stride", C.c_int64 * 2),
        ("d_u_chunk_tok", C.c_void_p),
        ("d_v_chunk", C.c_void_p),
        ("u_rows", C.c_int64 * 2),
        ("v_slots", C.c_int64 * 2),
    ]


class kv_splice_tile(C.Structure):
    _fields_ = [
        ("src_lo", C.c_int64),
        ("dst_lo", C.c_int64),
        ("n", C.c_int32),
        ("seq", C.c_int32),
        ("unit", C.c_int32),
        ("stub", C.c_int32),
        ("dep", C.c_int32 * 4),
    ]


_lib: Optional[C.CDLL] = None


def load(build_if_missing: bool = False) -> C.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        if not build_if_missing:
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        _build.build()
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    P, PP = C.POINTER(kv_pool_desc), C.POINTER(kv_patch_desc)
    sig = {
        "kv_workspace_size": (sz, [P, i64, i32]),
        "kv_relocate": (i32, [P, P, i32, i64, vp, vp, vp, vp, vp, vp, i32, i32, PP, vp, sz, vp]),
        "kv_splice": (i32, [P, i32, vp, i32, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]),
        "kv_patch": (i32, [P, i32, i64, vp, vp, vp, vp, i32, i32, PP, vp, sz, vp]),
        "kv_splice_composed_workspace_size": (sz, [P, i32, i32, vp, vp, vp, vp]),
        "kv_splice_composed": (i32, [P, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "kv_splice_composed_plan": (i32, [P, i32, i32, vp, vp, vp, vp, vp, i64, vp, i32,
                                          C.POINTER(i64), C.POINTER(i32)]),
        "kv_get_device_status": (i32, [vp, vp]),
        "kv_set_wait_limit_ns": (None, [i64]),
        "kv_set_debug_checks": (None, [i32]),
        "kv_set_splice_skip_publish": (None, [i64]),
        "kv_check_wait_timeout": (i32, [vp, sz, i64, vp]),
        "kv_last_launch_count": (i32, []),
        "kv_set_kernel_events": (None, [vp, vp]),
        "kv_relocate_noalloc": (i32, [P, P, i32, i64, vp, vp, vp, vp, vp, vp, i32, i32, PP,
                                      C.POINTER(C.c_int32), vp]),
        "kv_cdc_workspace_size": (sz, [i64]),
        "kv_cdc": (i32, [i32, vp, i64, vp, C.c_uint64, C.c_uint64, C.c_uint64, i64, vp, vp, vp,
                         vp, sz, vp]),
        "kv_fingerprint": (i32, [i64, vp, vp, i64, vp, C.c_uint64, vp, vp, sz, vp]),
        "kv_status_string": (C.c_char_p, [i32]),
        "kv_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().kv_status_string(int(status)).decode()


def _ptr(t):
    """Device address of a tensor; raw addresses (int / c_void_p) pass through."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return t.value if isinstance(t, C.c_void_p) else int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        if not torch.cuda.is_available():
            return None  # host-side argument checks need no stream
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != KV_OK:
        raise KVError(status, where)


# ---------------------------------------------------------------------------
# Descriptors
# ---------------------------------------------------------------------------

def pool_desc(copy: torch.Tensor, rot: torch.Tensor, block_size: int, rot_heads: int,
              rope_base: float, pair_convention: int = 0) -> kv_pool_desc:
    """Describe a pool from two bf16 views: ``copy`` [L][slots][copy_dim] and
    ``rot`` [L][slots][rot_heads*head_dim] (any strides with a unit last stride;
    e.g. the two column ranges of one fused [L][slots][576] MLA tensor).
    ``pair_convention`` 1: rotary pairs stored interleaved (x[2j], x[2j+1])."""
    assert copy.dtype == torch.bfloat16 and rot.dtype == torch.bfloat16
    assert copy.dim() == 3 and rot.dim() == 3 and copy.stride(2) == 1 and rot.stride(2) == 1
    assert copy.shape[:2] == rot.shape[:2]
    L, S, cd = copy.shape
    d = kv_pool_desc(L, block_size, S, copy.data_ptr(), copy.stride(0), copy.stride(1), cd,
                     rot.data_ptr(), rot.stride(0), rot.stride(1), rot_heads,
                     rot.shape[2] // rot_heads, float(rope_base), int(pair_convention))
    d._tensors = (copy, rot)  # the descriptor keeps the memory it points at alive
    return d


def patch_desc(rank: int, u: Sequence[Optional[torch.Tensor]],
               v: Sequence[Optional[torch.Tensor]], u_chunk_tok: Optional[torch.Tensor] = None,
               v_chunk: Optional[torch.Tensor] = None,
               check_extents: bool = True) -> kv_patch_desc:
    """Factors per channel (0 = verbatim part, 1 = rotated part): ``u[ch]``
    fp32 (L, tokens, rank), ``v[ch]`` fp32 (L, chunks, columns, rank), any
    strides with a unit last stride; None = channel not patched.  Optional
    device maps into factors kept per canonical chunk: ``u_chunk_tok`` int64
    (chunks,) U row of each chunk's first token, ``v_chunk`` int32 (chunks,)
    V slot of each chunk.  ``check_extents``: pass the factor arrays' row and
    slot counts, so a token or chunk addressing outside them is skipped and
    reported (KV_ERR_OUT_OF_RANGE) instead of read out of bounds."""
    d = kv_patch_desc()
    d.rank = rank
    # keep the factors and maps alive as long as the descriptor
    d._tensors = (list(u), list(v), u_chunk_tok, v_chunk)
    if u_chunk_tok is not None:
        assert u_chunk_tok.dtype == torch.int64 and u_chunk_tok.is_contiguous()
        d.d_u_chunk_tok = u_chunk_tok.data_ptr()
    if v_chunk is not None:
        assert v_chunk.dtype == torch.int32 and v_chunk.is_contiguous()
        d.d_v_chunk = v_chunk.data_ptr()
    for ch in range(2):
        if u[ch] is None or v[ch] is None:
            continue
        uu, vv = u[ch], v[ch]
        assert uu.dtype == torch.float32 and vv.dtype == torch.float32
        assert uu.stride(2) == 1 and vv.stride(3) == 1
        d.u[ch] = uu.data_ptr()
        d.u_layer_stride[ch] = uu.stride(0)
        d.u_tok_stride[ch] = uu.stride(1)
        d.v[ch] = vv.data_ptr()
        d.v_layer_stride[ch] = vv.stride(0)
        d.v_chunk_stride[ch] = vv.stride(1)
        d.v_col_stride[ch] = vv.stride(2)
        if check_extents:
            d.u_rows[ch] = uu.shape[1]
            d.v_slots[ch] = vv.shape[1]
    return d


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def kv_workspace_size(pool: kv_pool_desc, max_rows: int, max_units: int) -> int:
    return int(load().kv_workspace_size(C.byref(pool), int(max_rows), int(max_units)))


def workspace(pool: kv_pool_desc, max_rows: int, max_units: int, device="cuda") -> torch.Tensor:
    """A device workspace (uint8, 256-byte aligned) for calls on ``pool``."""
    n = kv_workspace_size(pool, max_rows, max_units)
    if n == 0:
        raise KVError(KV_ERR_INVALID_ARG, "kv_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def kv_relocate(src: kv_pool_desc, dst: kv_pool_desc, num_chunks: int, total_tokens: int,
                tok_off, src_slots, chunk_req, chunk_dst_pos, delta, block_tables,
                num_reqs: int, max_blocks: int, patch: Optional[kv_patch_desc],
                ws: torch.Tensor, stream=None, check: bool = True) -> int:
    st = load().kv_relocate(
        C.byref(src), C.byref(dst), int(num_chunks), int(total_tokens), _ptr(tok_off),
        _ptr(src_slots), _ptr(chunk_req), _ptr(chunk_dst_pos), _ptr(delta), _ptr(block_tables),
        int(num_reqs), int(max_blocks), C.byref(patch) if patch is not None else None,
        ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "kv_relocate")
    return st


def kv_splice(pool: kv_pool_desc, num_seqs: int, block_tables, max_blocks: int,
              seq_lens, s_start, s_end, stub_len, stub_copy, stub_rot, mode: int,
              ws: Optional[torch.Tensor], stream=None, check: bool = True) -> int:
    """``seq_lens`` is a host int32 tensor updated in place; ``s_start``,
    ``s_end``, ``stub_len`` host int32 tensors; stubs device bf16 tensors."""
    for t in (seq_lens, s_start, s_end, stub_len):
        assert t.device.type == "cpu" and t.dtype == torch.int32 and t.is_contiguous()
    st = load().kv_splice(
        C.byref(pool), int(num_seqs), _ptr(block_tables), int(max_blocks), seq_lens.data_ptr(),
        s_start.data_ptr(), s_end.data_ptr(), stub_len.data_ptr(), _ptr(stub_copy),
        _ptr(stub_rot), int(mode), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
        _stream(stream))
    if check:
        _check(st, "kv_splice")
    return st


def _dirs(seq_lens, s_start, s_end, stub_len):
    for t in (seq_lens, s_start, s_end, stub_len):
        assert t.device.type == "cpu" and t.dtype == torch.int32 and t.is_contiguous()
    assert s_start.dim() == 2 and s_start.shape[1] == seq_lens.numel()
    assert s_end.shape == s_start.shape and stub_len.shape == s_start.shape
    return int(seq_lens.numel()), int(s_start.shape[0])


def kv_splice_composed_workspace_size(pool: kv_pool_desc, seq_lens, s_start, s_end,
                                      stub_len) -> int:
    """Bytes of workspace the composed splice of these directives needs (0:
    invalid directives).  ``s_start``, ``s_end``, ``stub_len``: host int32
    (num_dirs, num_seqs)."""
    S, D = _dirs(seq_lens, s_start, s_end, stub_len)
    return int(load().kv_splice_composed_workspace_size(
        C.byref(pool), S, D, seq_lens.data_ptr(), s_start.data_ptr(), s_end.data_ptr(),
        stub_len.data_ptr()))


def kv_splice_composed(pool: kv_pool_desc, block_tables, max_blocks: int, seq_lens, s_start,
                       s_end, stub_len, stub_copy, stub_rot, ws: Optional[torch.Tensor],
                       stream=None, check: bool = True) -> int:
    """Several directives per sequence as one in-place edit; ``seq_lens`` (host
    int32) becomes the final lengths; directives host int32 (num_dirs,
    num_seqs), directive i in the indexing the previous ones left; stubs
    device bf16, directive-major then sequence."""
    S, D = _dirs(seq_lens, s_start, s_end, stub_len)
    st = load().kv_splice_composed(
        C.byref(pool), S, D, _ptr(block_tables), int(max_blocks), seq_lens.data_ptr(),
        s_start.data_ptr(), s_end.data_ptr(), stub_len.data_ptr(), _ptr(stub_copy),
        _ptr(stub_rot), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
        _stream(stream))
    if check:
        _check(st, "kv_splice_composed")
    return st


def kv_splice_composed_plan(pool: kv_pool_desc, seq_lens, s_start, s_end, stub_len):
    """(status, tiles, deltas) of the composed splice's plan (host only):
    tiles as a list of dicts with src_lo, dst_lo, n, seq, unit, stub, dep."""
    S, D = _dirs(seq_lens, s_start, s_end, stub_len)
    lib = load()
    nt, nu = C.c_int64(0), C.c_int32(0)
    args = (C.byref(pool), S, D, seq_lens.data_ptr(), s_start.data_ptr(), s_end.data_ptr(),
            stub_len.data_ptr())
    st = lib.kv_splice_composed_plan(*args, None, 0, None, 0, C.byref(nt), C.byref(nu))
    if st != KV_OK:
        return st, [], []
    tiles = (kv_splice_tile * max(nt.value, 1))()
    deltas = (C.c_int32 * max(nu.value, 1))()
    st = lib.kv_splice_composed_plan(*args, tiles, nt.value, deltas, nu.value, C.byref(nt),
                                     C.byref(nu))
    out = [dict(src_lo=t.src_lo, dst_lo=t.dst_lo, n=t.n, seq=t.seq, unit=t.unit, stub=t.stub,
                dep=list(t.dep)) for t in tiles[:nt.value]]
    return st, out, list(deltas[:nu.value])


def kv_patch(pool: kv_pool_desc, num_chunks: int, total_tokens: int, tok_off, chunk_req,
             chunk_dst_pos, block_tables, num_reqs: int, max_blocks: int,
             patch: kv_patch_desc, ws: torch.Tensor, stream=None, check: bool = True) -> int:
    st = load().kv_patch(
        C.byref(pool), int(num_chunks), int(total_tokens), _ptr(tok_off), _ptr(chunk_req),
        _ptr(chunk_dst_pos), _ptr(block_tables), int(num_reqs), int(max_blocks),
        C.byref(patch), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "kv_patch")
    return st


def kv_cdc_workspace_size(total_tokens: int) -> int:
    return int(load().kv_cdc_workspace_size(int(total_tokens)))


def kv_cdc(num_streams: int, stream_off, total_tokens: int, tokens, gear_seed: int,
           threshold: int, fp_seed: int, max_chunks: int, chunk_end, fingerprint, num_chunks,
           ws: torch.Tensor, stream=None, check: bool = True) -> int:
    """Content-defined chunking (Irminsul §2.2); device tensors: stream_off
    int64 [S+1], tokens int32, chunk_end int64 and fingerprint (uint64 bits in
    an int64 tensor) [max_chunks], num_chunks int64 [1]."""
    m = 2**64 - 1
    st = load().kv_cdc(int(num_streams), _ptr(stream_off), int(total_tokens), _ptr(tokens),
                       int(gear_seed) & m, int(threshold) & m, int(fp_seed) & m, int(max_chunks),
                       _ptr(chunk_end), _ptr(fingerprint), _ptr(num_chunks), ws.data_ptr(),
                       ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "kv_cdc")
    return st


def kv_fingerprint(num_ranges: int, start, end, total_tokens: int, tokens, fp_seed: int,
                   fingerprint, ws: torch.Tensor, stream=None, check: bool = True) -> int:
    st = load().kv_fingerprint(int(num_ranges), _ptr(start), _ptr(end), int(total_tokens),
                               _ptr(tokens), int(fp_seed) & (2**64 - 1), _ptr(fingerprint),
                               ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "kv_fingerprint")
    return st


def kv_get_device_status(ws: torch.Tensor, stream=None) -> int:
    return int(load().kv_get_device_status(ws.data_ptr(), _stream(stream)))


def kv_set_wait_limit_ns(limit_ns: int) -> None:
    load().kv_set_wait_limit_ns(int(limit_ns))


def kv_set_debug_checks(on: bool) -> None:
    """Process-wide: check the overlap / distinct-block contracts on the device
    before every relocation and splice (KV_ERR_OVERLAP, nothing stored)."""
    load().kv_set_debug_checks(1 if on else 0)


def kv_set_splice_skip_publish(ticket: int) -> None:
    """Test hook: the splice tile drawing ``ticket`` does not publish its reads
    (its dependants time out); -1 turns it off."""
    load().kv_set_splice_skip_publish(int(ticket))


def kv_check_wait_timeout(ws: torch.Tensor, limit_ns: int, stream=None) -> int:
    return int(load().kv_check_wait_timeout(ws.data_ptr(), ws.numel() * ws.element_size(),
                                            int(limit_ns), _stream(stream)))


def kv_set_kernel_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event ``start``/``stop`` around the row-moving kernel
    of every later call on this thread (None, None = off).  The events must
    have been recorded once through torch first (torch creates them lazily)."""
    if start is not None and (start.cuda_event == 0 or stop.cuda_event == 0):
        raise ValueError("record the events once through torch before passing them")
    load().kv_set_kernel_events(None if start is None else start.cuda_event,
                                None if stop is None else stop.cuda_event)


def kv_last_launch_count() -> int:
    return int(load().kv_last_launch_count())


def kv_version() -> int:
    return int(load().kv_version())


def kv_relocate_noalloc(src: kv_pool_desc, dst: kv_pool_desc, num_chunks: int,
                        total_tokens: int, tok_off, src_slots, chunk_req, chunk_dst_pos, delta,
                        block_tables, num_reqs: int, max_blocks: int,
                        patch: Optional[kv_patch_desc], stream=None, wait: bool = True,
                        check: bool = True):
    """kv_relocate for callers that cannot allocate device memory: no workspace
    argument; the library's built-in device scratch is used instead.  With
    ``wait`` the call synchronises and returns (status, device_status)."""
    dev_status = C.c_int32(-1)
    st = load().kv_relocate_noalloc(
        C.byref(src), C.byref(dst), int(num_chunks), int(total_tokens), _ptr(tok_off),
        _ptr(src_slots), _ptr(chunk_req), _ptr(chunk_dst_pos), _ptr(delta), _ptr(block_tables),
        int(num_reqs), int(max_blocks), C.byref(patch) if patch is not None else None,
        C.byref(dev_status) if wait else None, _stream(stream))
    if check:
        _check(st, "kv_relocate_noalloc")
    return st, (int(dev_status.value) if wait else None)

"""ctypes front end of the fp64 CPU oracle (``kvoracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg load it; the CUDA library never does.  Arrays are numpy:
bf16 values travel as their uint16 bit patterns, indices as int32, patch
factors as float32.  Nothing here does arithmetic of the method; every step
of it is in the C file.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

from . import build as _build

OK, ERR_INVALID, ERR_RANGE, ERR_CAPACITY = 0, 1, 2, 3
AMORTIZE, FORGET = 0, 1


class _Pool(C.Structure):
    _fields_ = [
        ("num_layers", C.c_int),
        ("num_slots", C.c_int64),
        ("block_size", C.c_int),
        ("copy_dim", C.c_int),
        ("rot_heads", C.c_int),
        ("rot_d", C.c_int),
        ("rope_base", C.c_double),
        ("copy", C.c_void_p),
        ("rot", C.c_void_p),
        ("pair_convention", C.c_int),
    ]


class _Patch(C.Structure):
    _fields_ = [
        ("m", C.c_int),
        ("u", C.c_void_p * 2),
        ("u_layer_stride", C.c_int64 * 2),
        ("u_tok_stride", C.c_int64 * 2),
        ("v", C.c_void_p * 2),
        ("v_layer_stride", C.c_int64 * 2),
        ("v_chunk_stride", C.c_int64 * 2),
        ("v_col_stride", C.c_int64 * 2),
        ("u_chunk_tok", C.c_void_p),
        ("v_chunk", C.c_void_p),
    ]


@dataclass
class Pool:
    """A paged KV pool in the oracle's layout.

    ``copy`` is [L][slots][copy_dim] and ``rot`` is [L][slots][rot_heads*rot_d],
    both uint16 (bf16 bits), C-contiguous.  Logical position p of request q
    lives in slot ``block_tables[q][p // block_size] * block_size + p % block_size``.
    """
    copy: np.ndarray
    rot: np.ndarray
    block_size: int
    rot_heads: int
    rot_d: int
    rope_base: float
    pair_convention: int = 0   # 0: rotate-half pairs (x[j], x[j+d/2]); 1: interleaved

    def __post_init__(self):
        assert self.copy.dtype == np.uint16 and self.rot.dtype == np.uint16
        assert self.copy.flags.c_contiguous and self.rot.flags.c_contiguous
        assert self.copy.shape[:2] == self.rot.shape[:2]
        assert self.rot.shape[2] == self.rot_heads * self.rot_d

    def _c(self) -> _Pool:
        L, S, cd = self.copy.shape
        return _Pool(L, S, self.block_size, cd, self.rot_heads, self.rot_d,
                     float(self.rope_base), self.copy.ctypes.data, self.rot.ctypes.data,
                     int(self.pair_convention))


@dataclass
class Patch:
    """Rank-m factors per channel (0 = verbatim part, 1 = rotated part).

    ``u[ch]`` is a float32 array indexed (layer, token, r) and ``v[ch]`` a
    float32 array indexed (layer, chunk, column, r); any strides (views are
    fine, e.g. two column ranges of one 576-wide factor).  ``None`` = no patch
    on that channel.
    """
    m: int
    u: Sequence[Optional[np.ndarray]] = field(default_factory=lambda: [None, None])
    v: Sequence[Optional[np.ndarray]] = field(default_factory=lambda: [None, None])
    # optional per-chunk maps into factors kept per canonical chunk: U row of
    # the chunk's first token (int64) and V slot of the chunk (int32)
    u_chunk_tok: Optional[np.ndarray] = None
    v_chunk: Optional[np.ndarray] = None

    def _c(self) -> _Patch:
        p = _Patch()
        p.m = self.m
        for ch in range(2):
            u, v = self.u[ch], self.v[ch]
            if u is None or v is None:
                p.u[ch] = None
                p.v[ch] = None
                continue
            assert u.dtype == np.float32 and v.dtype == np.float32
            assert u.ndim == 3 and v.ndim == 4 and u.shape[2] == self.m and v.shape[3] == self.m
            assert u.strides[2] == 4 and v.strides[3] == 4
            p.u[ch] = u.ctypes.data
            p.u_layer_stride[ch] = u.strides[0] // 4
            p.u_tok_stride[ch] = u.strides[1] // 4
            p.v[ch] = v.ctypes.data
            p.v_layer_stride[ch] = v.strides[0] // 4
            p.v_chunk_stride[ch] = v.strides[1] // 4
            p.v_col_stride[ch] = v.strides[2] // 4
        if self.u_chunk_tok is not None:
            self.u_chunk_tok = np.ascontiguousarray(self.u_chunk_tok, dtype=np.int64)
            p.u_chunk_tok = self.u_chunk_tok.ctypes.data
        if self.v_chunk is not None:
            self.v_chunk = np.ascontiguousarray(self.v_chunk, dtype=np.int32)
            p.v_chunk = self.v_chunk.ctypes.data
        return p


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


class Oracle:
    """Handle on one compiled copy of the oracle library."""

    def __init__(self, path: Optional[str] = None):
        if path is None:
            if _build.needs_build():
                _build.build()
            path = _build.LIB
        self.path = path
        lib = C.CDLL(path)
        self._lib = lib
        vp, i64, i32, dbl = C.c_void_p, C.c_int64, C.c_int, C.c_double
        lib.kvo_bf16_to_f64.restype = dbl
        lib.kvo_bf16_to_f64.argtypes = [C.c_uint16]
        lib.kvo_round_bf16.restype = C.c_uint16
        lib.kvo_round_bf16.argtypes = [dbl]
        lib.kvo_round_bf16_n.argtypes = [vp, vp, i64]
        lib.kvo_bf16_to_f64_n.argtypes = [vp, vp, i64]
        lib.kvo_theta.restype = dbl
        lib.kvo_theta.argtypes = [dbl, i32, i32]
        lib.kvo_rotate_f64.argtypes = [vp, vp, i32, i64, dbl]
        lib.kvo_rotate_bf16.argtypes = [vp, vp, i32, i64, dbl]
        lib.kvo_rotate_bf16_il.argtypes = [vp, vp, i32, i64, dbl]
        lib.kvo_rotate_f64_il.argtypes = [vp, vp, i32, i64, dbl]
        lib.kvo_relocate.restype = i32
        lib.kvo_relocate.argtypes = [C.POINTER(_Pool), C.POINTER(_Pool), i32, vp, vp, vp, vp, vp,
                                     vp, i32, i32, C.POINTER(_Patch)]
        lib.kvo_patch_apply.restype = i32
        lib.kvo_patch_apply.argtypes = [C.POINTER(_Pool), i32, vp, vp, vp, vp, i32, i32,
                                        C.POINTER(_Patch)]
        lib.kvo_splice.restype = i32
        lib.kvo_splice.argtypes = [C.POINTER(_Pool), i32, vp, i32, vp, vp, vp, vp, vp, vp, i32]
        lib.kvo_splice_composed.restype = i32
        lib.kvo_splice_composed.argtypes = [C.POINTER(_Pool), i32, i32, vp, i32, vp, vp, vp, vp,
                                            vp, vp]
        u64 = C.c_uint64
        lib.kvo_splitmix64_at.restype = u64
        lib.kvo_splitmix64_at.argtypes = [u64, u64]
        lib.kvo_xxh64.restype = u64
        lib.kvo_xxh64.argtypes = [vp, i64, u64]
        lib.kvo_gear_hashes.argtypes = [vp, i64, u64, vp]
        lib.kvo_cdc.restype = i64
        lib.kvo_cdc.argtypes = [i32, vp, vp, u64, u64, u64, i64, vp, vp]
        lib.kvo_fingerprint.restype = i32
        lib.kvo_fingerprint.argtypes = [i64, vp, vp, vp, u64, vp]

    # -- scalar / vector helpers ------------------------------------------
    def round_bf16(self, v: float) -> int:
        return int(self._lib.kvo_round_bf16(float(v)))

    def round_bf16_array(self, v) -> np.ndarray:
        v = np.asarray(v, dtype=np.float64)
        flat = np.ascontiguousarray(v.reshape(-1))
        out = np.empty(flat.shape, dtype=np.uint16)
        self._lib.kvo_round_bf16_n(flat.ctypes.data, out.ctypes.data, flat.size)
        return out.reshape(v.shape)

    def bf16_to_f64(self, b) -> np.ndarray:
        b = np.asarray(b, dtype=np.uint16)
        flat = np.ascontiguousarray(b.reshape(-1))
        out = np.empty(flat.shape, dtype=np.float64)
        self._lib.kvo_bf16_to_f64_n(flat.ctypes.data, out.ctypes.data, flat.size)
        return out.reshape(b.shape)

    def theta(self, base: float, j: int, d: int) -> float:
        return float(self._lib.kvo_theta(base, j, d))

    def rotate_f64(self, x, delta: int, base: float) -> np.ndarray:
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        y = np.empty_like(x)
        self._lib.kvo_rotate_f64(x.ctypes.data, y.ctypes.data, x.shape[-1], int(delta), base)
        return y

    def rotate_bf16(self, x, delta: int, base: float, interleaved: bool = False) -> np.ndarray:
        x = np.ascontiguousarray(np.asarray(x, dtype=np.uint16))
        y = np.empty_like(x)
        fn = self._lib.kvo_rotate_bf16_il if interleaved else self._lib.kvo_rotate_bf16
        fn(x.ctypes.data, y.ctypes.data, x.shape[-1], int(delta), base)
        return y

    # -- the three operations ------------------------------------------------
    def relocate(self, src: Pool, dst: Pool, tok_off, src_slots, chunk_req, chunk_dst_pos,
                 delta, block_tables, patch: Optional[Patch] = None) -> int:
        """Out-of-place gather + rotation (+ patch); ``dst`` is written in place."""
        tok_off, src_slots = _i32(tok_off), _i32(src_slots)
        chunk_req, chunk_dst_pos, delta = _i32(chunk_req), _i32(chunk_dst_pos), _i32(delta)
        bt = _i32(block_tables)
        nreq, maxb = (bt.shape if bt.ndim == 2 else (0, 0))
        ps, pd = src._c(), dst._c()
        pp = patch._c() if patch is not None else None
        return int(self._lib.kvo_relocate(
            C.byref(ps), C.byref(pd), len(chunk_req), _ptr(tok_off), _ptr(src_slots),
            _ptr(chunk_req), _ptr(chunk_dst_pos), _ptr(delta), _ptr(bt), nreq, maxb,
            C.byref(pp) if pp is not None else None))

    def patch_apply(self, pool: Pool, tok_off, chunk_req, chunk_dst_pos, block_tables,
                    patch: Patch) -> int:
        tok_off, chunk_req, chunk_dst_pos = _i32(tok_off), _i32(chunk_req), _i32(chunk_dst_pos)
        bt = _i32(block_tables)
        nreq, maxb = bt.shape
        pp = pool._c()
        pt = patch._c()
        return int(self._lib.kvo_patch_apply(
            C.byref(pp), len(chunk_req), _ptr(tok_off), _ptr(chunk_req), _ptr(chunk_dst_pos),
            _ptr(bt), nreq, maxb, C.byref(pt)))

    def splice(self, pool: Pool, block_tables, seq_lens: np.ndarray, s_start, s_end, stub_len,
               stub_copy: Optional[np.ndarray], stub_rot: Optional[np.ndarray],
               mode: int = AMORTIZE) -> int:
        """In-place splice; ``seq_lens`` (int32 array) is updated in place."""
        assert seq_lens.dtype == np.int32 and seq_lens.flags.c_contiguous
        bt = _i32(block_tables)
        s_start, s_end, stub_len = _i32(s_start), _i32(s_end), _i32(stub_len)
        if stub_copy is not None:
            assert stub_copy.dtype == np.uint16 and stub_copy.flags.c_contiguous
            assert stub_rot.dtype == np.uint16 and stub_rot.flags.c_contiguous
        pp = pool._c()
        return int(self._lib.kvo_splice(
            C.byref(pp), len(seq_lens), _ptr(bt), bt.shape[1], _ptr(seq_lens), _ptr(s_start),
            _ptr(s_end), _ptr(stub_len), _ptr(stub_copy), _ptr(stub_rot), int(mode)))


    def splice_composed(self, pool: Pool, block_tables, seq_lens: np.ndarray, s_start, s_end,
                        stub_len, stub_copy: Optional[np.ndarray],
                        stub_rot: Optional[np.ndarray]) -> int:
        """Several directives per sequence applied as one composed edit (one
        bf16 rounding per row).  ``s_start``, ``s_end``, ``stub_len`` are
        (num_dirs, num_seqs) int32 arrays, directive i in the indexing left by
        directives before it; stub rows directive-major, then sequence."""
        assert seq_lens.dtype == np.int32 and seq_lens.flags.c_contiguous
        bt = _i32(block_tables)
        s_start, s_end, stub_len = _i32(s_start), _i32(s_end), _i32(stub_len)
        assert s_start.ndim == 2 and s_start.shape[1] == len(seq_lens)
        assert s_end.shape == s_start.shape and stub_len.shape == s_start.shape
        if stub_copy is not None:
            assert stub_copy.dtype == np.uint16 and stub_copy.flags.c_contiguous
            assert stub_rot.dtype == np.uint16 and stub_rot.flags.c_contiguous
        pp = pool._c()
        return int(self._lib.kvo_splice_composed(
            C.byref(pp), len(seq_lens), s_start.shape[0], _ptr(bt), bt.shape[1], _ptr(seq_lens),
            _ptr(s_start), _ptr(s_end), _ptr(stub_len), _ptr(stub_copy), _ptr(stub_rot)))


    # -- content-defined chunking (Irminsul §2.2) ---------------------------
    def splitmix64_at(self, seed: int, n: int) -> int:
        return int(self._lib.kvo_splitmix64_at(seed & (2**64 - 1), n & (2**64 - 1)))

    def xxh64(self, data: bytes, seed: int = 0) -> int:
        buf = C.create_string_buffer(bytes(data), max(1, len(data)))
        return int(self._lib.kvo_xxh64(C.cast(buf, C.c_void_p), len(data), seed & (2**64 - 1)))

    def gear_hashes(self, tokens, gear_seed: int) -> np.ndarray:
        t = _i32(tokens)
        h = np.empty(len(t), dtype=np.uint64)
        self._lib.kvo_gear_hashes(_ptr(t), len(t), gear_seed & (2**64 - 1), _ptr(h))
        return h

    def cdc(self, stream_off, tokens, gear_seed: int, threshold: int, fp_seed: int = 0,
            max_chunks: Optional[int] = None):
        """(chunk_end int64, fingerprint uint64, count): every stream's chunks in order."""
        off = np.ascontiguousarray(np.asarray(stream_off, dtype=np.int64))
        t = _i32(tokens)
        cap = len(t) if max_chunks is None else int(max_chunks)
        ends = np.zeros(max(cap, 1), dtype=np.int64)
        fps = np.zeros(max(cap, 1), dtype=np.uint64)
        n = int(self._lib.kvo_cdc(len(off) - 1, _ptr(off), _ptr(t), gear_seed & (2**64 - 1),
                                  threshold & (2**64 - 1), fp_seed & (2**64 - 1), cap,
                                  _ptr(ends), _ptr(fps)))
        if n < 0:
            raise ValueError("malformed stream offsets")
        k = min(n, cap)
        return ends[:k], fps[:k], n

    def fingerprint(self, starts, ends, tokens, fp_seed: int = 0) -> np.ndarray:
        a = np.ascontiguousarray(np.asarray(starts, dtype=np.int64))
        b = np.ascontiguousarray(np.asarray(ends, dtype=np.int64))
        t = _i32(tokens)
        out = np.zeros(max(len(a), 1), dtype=np.uint64)
        if self._lib.kvo_fingerprint(len(a), _ptr(a), _ptr(b), _ptr(t), fp_seed & (2**64 - 1),
                                     _ptr(out)) != 0:
            raise ValueError("bad token range")
        return out[:len(a)]


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from ``kvoracle.c`` next to this file (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default

"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays out index structure; it holds
none of the method's arithmetic (no rotation, no rounding rule of its own, no
patch product).  KV values are bf16 obtained from fp32 ``torch.randn`` draws of
a seeded ``torch.Generator`` (torch's own fp32 -> bf16 cast); index structure
comes from ``numpy.random.default_rng(seed)``.

Workload shapes follow the three pages:
  * MLA rows (Irminsul §2.1, Leyline §2.2): c_KV 512 + k_pe 64, bf16.
  * GQA rows (Kamera §2): K and V of H_kv x D each, bf16.
  * paged storage in blocks of 64 tokens (Irminsul §1 names PagedAttention).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

BLOCK = 64


def bf16_normal(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws (fp32 randn, scaled, cast to bf16)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def f32_normal(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a CPU bf16 tensor (a view, no copy when contiguous)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# Relocation workloads (Irminsul §2.2, Kamera §2)
# ---------------------------------------------------------------------------

@dataclass
class RelocateWorkload:
    """Chunks gathered from a source (registry) pool into per-request block tables.

    Token t of the call is token ``t - tok_off[c]`` of chunk c; it is read from
    source slot ``src_slots[t]`` and lands at logical position
    ``chunk_dst_pos[c] + (t - tok_off[c])`` of request ``chunk_req[c]``.
    """
    src_slots_total: int          # slots in the source pool
    dst_slots_total: int          # slots in the destination pool
    tok_off: np.ndarray           # int32 [C+1]
    src_slots: np.ndarray         # int32 [T]
    chunk_req: np.ndarray         # int32 [C]
    chunk_dst_pos: np.ndarray     # int32 [C]
    delta: np.ndarray             # int32 [C]
    block_tables: np.ndarray      # int32 [R][max_blocks], -1 where never written
    chunk_len: np.ndarray         # int32 [C]

    @property
    def num_chunks(self) -> int:
        return len(self.chunk_req)

    @property
    def total_tokens(self) -> int:
        return int(self.tok_off[-1])


def _registry(rng, n_pool_chunks, len_lo, len_hi, block):
    """Canonical chunks stored as contiguous runs inside randomly placed blocks."""
    lens = rng.integers(len_lo, len_hi + 1, size=n_pool_chunks)
    nblk = [(int(n) + block - 1) // block for n in lens]
    perm = rng.permutation(sum(nblk))
    slots, k = [], 0
    for n, nb in zip(lens, nblk):
        blks = perm[k:k + nb]
        k += nb
        i = np.arange(int(n))
        slots.append((blks[i // block] * block + i % block).astype(np.int32))
    return lens.astype(np.int32), slots, int(sum(nblk)) * block


def relocate_workload(seed: int, num_reqs: int, chunks_per_req: int, len_lo: int, len_hi: int,
                      delta_lo: int, delta_hi: int, n_pool_chunks: int, base_hi: int = 32768,
                      block: int = BLOCK, fixed_len: Optional[int] = None) -> RelocateWorkload:
    """Irminsul-style assembly: each request takes ``chunks_per_req`` chunks
    from a registry of ``n_pool_chunks`` canonical chunks (with replacement) and
    lays them back to back from a random, generally unaligned, base position.
    δ per chunk is uniform in [delta_lo, delta_hi]."""
    rng = np.random.default_rng(seed)
    if fixed_len is not None:
        len_lo = len_hi = fixed_len
    pool_lens, pool_slots, src_total = _registry(rng, n_pool_chunks, len_lo, len_hi, block)
    picks = rng.integers(0, n_pool_chunks, size=(num_reqs, chunks_per_req))
    bases = rng.integers(0, base_hi + 1, size=num_reqs)
    chunk_req, chunk_dst_pos, chunk_len, src = [], [], [], []
    req_extent = []
    for r in range(num_reqs):
        pos = int(bases[r])
        for k in picks[r]:
            chunk_req.append(r)
            chunk_dst_pos.append(pos)
            chunk_len.append(int(pool_lens[k]))
            src.append(pool_slots[k])
            pos += int(pool_lens[k])
        req_extent.append((int(bases[r]), pos))
    # destination block tables: only the blocks a request writes are real
    max_blocks = max((hi + block - 1) // block for _, hi in req_extent) if req_extent else 1
    bt = np.full((max(num_reqs, 1), max(max_blocks, 1)), -1, dtype=np.int32)
    need = [((lo // block), (hi + block - 1) // block) for lo, hi in req_extent]
    nblocks = sum(b - a for a, b in need)
    perm = rng.permutation(nblocks).astype(np.int32)
    k = 0
    for r, (a, b) in enumerate(need):
        bt[r, a:b] = perm[k:k + b - a]
        k += b - a
    C = len(chunk_req)
    tok_off = np.zeros(C + 1, dtype=np.int32)
    tok_off[1:] = np.cumsum(chunk_len)
    delta = rng.integers(delta_lo, delta_hi + 1, size=C).astype(np.int32)
    return RelocateWorkload(
        src_slots_total=src_total, dst_slots_total=max(nblocks, 1) * block,
        tok_off=tok_off,
        src_slots=np.concatenate(src).astype(np.int32) if src else np.zeros(0, np.int32),
        chunk_req=np.asarray(chunk_req, np.int32), chunk_dst_pos=np.asarray(chunk_dst_pos, np.int32),
        delta=delta, block_tables=bt, chunk_len=np.asarray(chunk_len, np.int32))


def fixed_chunk_workload(seed: int, chunk_len: int, delta: int, num_reqs: int, req_tokens: int,
                         block: int = BLOCK) -> RelocateWorkload:
    """Relocation of ``num_reqs`` x ``req_tokens`` tokens in chunks of exactly
    ``chunk_len`` tokens, every chunk with the same δ (a sweep point).  The
    registry holds one distinct canonical chunk per relocated chunk, packed
    back to back (chunks shorter than a block share blocks) over a random
    block permutation, so the call reads every registry row once.  Each
    request starts at a random offset inside its first destination block and
    lays its chunks back to back; all of its block-table entries are real
    blocks in a random permutation of the destination pool."""
    assert req_tokens % chunk_len == 0
    rng = np.random.default_rng(seed)
    per_req = req_tokens // chunk_len
    n_chunks = num_reqs * per_req
    reg_blocks = (n_chunks * chunk_len + block - 1) // block
    reg_perm = rng.permutation(reg_blocks).astype(np.int64)
    order = rng.permutation(n_chunks).astype(np.int64)     # registry chunk of each chunk
    pos = (order[:, None] * chunk_len + np.arange(chunk_len)[None, :]).reshape(-1)
    src_slots = (reg_perm[pos // block] * block + pos % block).astype(np.int32)
    chunk_req = np.repeat(np.arange(num_reqs), per_req).astype(np.int32)
    bases = rng.integers(0, block, size=num_reqs)
    chunk_dst_pos = (bases[chunk_req] +
                     np.tile(np.arange(per_req) * chunk_len, num_reqs)).astype(np.int32)
    max_blocks = (block - 1 + req_tokens + block - 1) // block
    bt = rng.permutation(num_reqs * max_blocks).astype(np.int32).reshape(num_reqs, max_blocks)
    return RelocateWorkload(
        src_slots_total=reg_blocks * block, dst_slots_total=num_reqs * max_blocks * block,
        tok_off=(np.arange(n_chunks + 1) * chunk_len).astype(np.int32), src_slots=src_slots,
        chunk_req=chunk_req, chunk_dst_pos=chunk_dst_pos,
        delta=np.full(n_chunks, delta, np.int32), block_tables=bt,
        chunk_len=np.full(n_chunks, chunk_len, np.int32))


# ---------------------------------------------------------------------------
# Splice workloads (Leyline §2.1-§2.3)
# ---------------------------------------------------------------------------

@dataclass
class SpliceSeqs:
    """Sequences stored in one paged pool, each with its own block table row."""
    num_slots: int
    block_tables: np.ndarray   # int32 [S][max_blocks]
    seq_lens: np.ndarray       # int32 [S]


def splice_seqs(seed: int, seq_lens: List[int], max_blocks: int, block: int = BLOCK,
                spare_blocks: int = 0) -> SpliceSeqs:
    """Random, distinct physical blocks for every block-table entry of every
    sequence (all ``max_blocks`` entries are real, so a splice may grow a
    sequence up to ``max_blocks * block`` tokens).  ``spare_blocks`` extra
    physical blocks are left unreferenced (they must never be touched)."""
    rng = np.random.default_rng(seed)
    S = len(seq_lens)
    total = S * max_blocks + spare_blocks
    perm = rng.permutation(total).astype(np.int32)
    bt = perm[:S * max_blocks].reshape(S, max_blocks).copy()
    return SpliceSeqs(num_slots=total * block, block_tables=bt,
                      seq_lens=np.asarray(seq_lens, dtype=np.int32))


@dataclass
class Directives:
    s_start: np.ndarray   # int32 [S]
    s_end: np.ndarray     # int32 [S]
    stub_len: np.ndarray  # int32 [S]


def random_directives(seed: int, seq_lens, span_lo: int, span_hi: int, stub_lo: int,
                      stub_hi: int) -> Directives:
    """One directive per sequence: a span of U[span_lo, span_hi] tokens at a
    uniform offset, replaced by a stub of U[stub_lo, stub_hi] rows."""
    rng = np.random.default_rng(seed)
    s0, s1, nr = [], [], []
    for n in seq_lens:
        n = int(n)
        span = int(rng.integers(min(span_lo, n), min(span_hi, n) + 1))
        off = int(rng.integers(0, n - span + 1))
        s0.append(off)
        s1.append(off + span)
        nr.append(int(rng.integers(stub_lo, stub_hi + 1)))
    return Directives(np.asarray(s0, np.int32), np.asarray(s1, np.int32), np.asarray(nr, np.int32))


def random_aligned_directives(seed: int, seq_lens, span_lo: int, span_hi: int, stub_lo: int,
                              stub_hi: int, block: int = BLOCK) -> Directives:
    """One block-aligned directive per sequence: a span of U[span_lo, span_hi]
    tokens rounded down to whole blocks, at a block-aligned uniform offset,
    replaced by a stub of U[stub_lo, stub_hi] whole blocks."""
    rng = np.random.default_rng(seed)
    s0, s1, nr = [], [], []
    for n in seq_lens:
        n = int(n)
        span = block * int(rng.integers(min(span_lo, n) // block, min(span_hi, n) // block + 1))
        off = block * int(rng.integers(0, (n - span) // block + 1))
        s0.append(off)
        s1.append(off + span)
        nr.append(block * int(rng.integers(stub_lo, stub_hi + 1)))
    return Directives(np.asarray(s0, np.int32), np.asarray(s1, np.int32), np.asarray(nr, np.int32))


def shard(n: int, rank: int, world: int) -> range:
    """Contiguous share of ``n`` independent units for ``rank`` of ``world``."""
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return range(lo, lo + base + (1 if rank < extra else 0))


@dataclass
class TokenStreams:
    stream_off: np.ndarray  # int64 [num_streams + 1], prefix offsets from 0
    tokens: np.ndarray      # int32 [total], token ids

    @property
    def num_streams(self) -> int:
        return len(self.stream_off) - 1


def token_streams(seed: int, lengths, vocab: int = 129280, shared_segments: int = 0,
                  segment_lo: int = 512, segment_hi: int = 4096) -> TokenStreams:
    """Token-id streams of the given lengths, ids U[0, vocab).  With
    `shared_segments` > 0, each stream also carries copies of segments drawn
    from a common pool, pasted at random offsets, so equal content recurs at
    shifted positions (the agentic traffic a content-keyed cache serves)."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    tokens = rng.integers(0, vocab, int(off[-1]), dtype=np.int64).astype(np.int32)
    if shared_segments > 0:
        pool = [rng.integers(0, vocab, int(rng.integers(segment_lo, segment_hi + 1)),
                             dtype=np.int64).astype(np.int32) for _ in range(shared_segments)]
        for s in range(len(lengths)):
            n = int(lengths[s])
            for _ in range(3):
                seg = pool[int(rng.integers(len(pool)))]
                if len(seg) >= n:
                    continue
                at = int(rng.integers(0, n - len(seg) + 1))
                tokens[off[s] + at: off[s] + at + len(seg)] = seg
    return TokenStreams(off, tokens)

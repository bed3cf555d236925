// kv_internal.h -- launch parameters shared by the host entry points and the
// kernels.  Not part of the public ABI (include/kvreloc.h is).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvr {

constexpr int kThreads = 256;         // threads per row-moving block
constexpr int kMaxSeqsPerLaunch = 64; // splice directives carried in one launch
constexpr int kMaxRank = 64;          // largest patch rank
constexpr int kHeaderBytes = 256;     // workspace header: status word, ticket counter
constexpr int kTileMla = 32;          // rows per tile for MLA rows (576 bf16)
constexpr int kTileGqa = 16;          // rows per tile for 8 x 128 GQA rows
constexpr int kTileGqa4 = 32;         // rows per tile for 4 x 128 GQA rows
constexpr int kTileMha = 4;           // rows per tile for 32 x 128 MHA rows

// Device status codes (same values as kv_status).
enum : uint32_t {
    kStatusOk = 0,
    kStatusOutOfRange = 2,
    kStatusCapacity = 3,
    kStatusTimeout = 5,
    kStatusOverlap = 8
};

// Row-moving kernels of a call made with the debug checks on read the
// status word first (`gate`; nullptr when the checks are off) and store
// nothing when a check found an overlap.
__device__ __forceinline__ bool gate_closed(const uint32_t *gate)
{
    return gate != nullptr && *reinterpret_cast<const volatile uint32_t *>(gate) == kStatusOverlap;
}

// A pool as the kernels see it: byte addresses and byte strides.
struct PoolView {
    char *copy;
    int64_t copy_ls, copy_ss;
    char *rot;
    int64_t rot_ls, rot_ss;
    int64_t num_slots;
    int64_t num_blocks;
    int32_t block;
    int32_t num_layers;
    int32_t il; // rotary pairs interleaved (x[2j], x[2j+1]) instead of rotate-half
};

struct PatchView {
    int32_t m;
    const float *u[2];
    int64_t u_ls[2], u_ts[2];
    const float *v[2];
    int64_t v_ls[2], v_cs[2], v_cols[2];
    const int64_t *u_chunk_tok; // per chunk: U row of its first token (nullptr: call order)
    const int32_t *v_chunk;     // per chunk: V slot (nullptr: call order)
    int64_t u_rows[2];          // extents of the factor arrays (0: unchecked)
    int64_t v_slots[2];
};

// True when U row `urow` and V slot `vslot` lie inside the extents of every
// patched channel (an extent of 0 is not checked).
__host__ __device__ __forceinline__ bool patch_rows_ok(const PatchView &pv, int64_t urow,
                                                       int64_t vslot)
{
    for (int ch = 0; ch < 2; ++ch) {
        if (pv.u[ch] == nullptr)
            continue;
        if (pv.u_rows[ch] > 0 && (urow < 0 || urow >= pv.u_rows[ch]))
            return false;
        if (pv.v_slots[ch] > 0 && (vslot < 0 || vslot >= pv.v_slots[ch]))
            return false;
    }
    return true;
}

// kv_relocate (in_place = 0) and kv_patch (in_place = 1: rows are read from
// and written back to the destination slots, without rotation).
struct RelocParams {
    PoolView src, dst;
    int32_t num_chunks;
    int64_t total_tokens;
    const int32_t *tok_off;
    const int32_t *src_slots;
    const int32_t *chunk_req;
    const int32_t *chunk_dst_pos;
    const int32_t *delta;
    const int32_t *block_tables;
    int32_t num_reqs, max_blocks;
    const float4 *table; // [num_chunks][head_dim/2]
    PatchView patch;
    int32_t patched;
    int32_t in_place;
    uint32_t *status;
    const uint32_t *gate; // debug checks: the status word (else nullptr)
};

// Host-side plan of one sequence of a splice launch.
struct SpliceSeq {
    int32_t s_start, s_end, seq_len, n_r;
    int32_t delta;   // n_r - (s_end - s_start)
    int32_t n_shift; // shift tiles (each covers all layers, in layer_groups units)
    int32_t n_stub;  // stub tiles
    int32_t bt_row;  // block-table row
    int64_t ticket_base;
    int64_t flag_base; // per-unit "layers read" counters of this sequence: [n_shift][groups]
    int64_t stub_base; // first stub row of this sequence
};

struct SpliceParams {
    PoolView pool;
    const int32_t *block_tables;
    int32_t max_blocks;
    const char *stub_copy; // [L][total_stub][copy_dim] bf16
    const char *stub_rot;  // [L][total_stub][rot width] bf16
    int64_t total_stub;
    const float4 *table; // [num_seqs][head_dim/2], row q for sequence q of this launch
    uint32_t *status;
    uint32_t *ticket;
    uint32_t *flags;
    int64_t total_tickets;
    int64_t wait_limit_ns;
    int64_t skip_publish; // test hook: this ticket does not publish its reads (-1: none)
    const uint32_t *gate;
    double rope_base;     // inline_table: every block forms its own cos/sin row
    int32_t inline_table; // 1: no δ-table kernel ran (small launches)
    int32_t layer_groups; // a tile's layers are cut into this many units ...
    int32_t group_layers; // ... of this many layers (the last may be shorter)
    int32_t num_seqs;
    SpliceSeq seq[kMaxSeqsPerLaunch];
};

// One tile of a composed splice (several directives per sequence applied as
// one edit): up to T rows that move from src_lo.. to dst_lo.. (logical
// positions of sequence `seq`, or stub rows when `stub`), turned by the
// δ-table row `unit` (-1: no rotation).  dep[0..1] and dep[2..3] are two
// inclusive ranges of earlier tiles whose source rows this tile's
// destination overlaps (-1: none).
struct SpliceTile {
    int64_t src_lo;
    int64_t dst_lo;
    int32_t n;
    int32_t seq;
    int32_t unit;
    int32_t stub;
    int32_t dep[4];
};

struct ComposedParams {
    PoolView pool;
    const int32_t *block_tables;
    int32_t max_blocks;
    const char *stub_copy; // [L][total_stub][copy_dim] bf16
    const char *stub_rot;  // [L][total_stub][rot width] bf16
    int64_t total_stub;
    const SpliceTile *tiles; // [num_tiles], in ticket order
    const float4 *table;     // [units][head_dim/2]
    uint32_t *status;
    uint32_t *ticket;
    uint32_t *flags; // [num_tiles] (layer, warp) read counters
    int64_t num_tiles;
    int64_t wait_limit_ns;
    int64_t skip_publish; // test hook (-1: none)
    const uint32_t *gate;
};

// Block-aligned splice by remapping (s_start, s_end, n_r multiples of the
// block size, Δ != 0): downstream rows keep their physical blocks, the
// block-table row is permuted, only the rotary part is rewritten in place.
struct RemapSeq {
    int32_t s_start, s_end, seq_len, n_r;
    int32_t delta;
    int32_t bt_row;
    int32_t n_down;   // tiles of downstream rows (rotated in place)
    int32_t n_stub;   // tiles of stub rows (written into the stub blocks)
    int64_t tile_base;
    int64_t stub_base; // first stub row of this sequence
};

struct RemapParams {
    PoolView pool;
    int32_t *block_tables; // rows are read by the data kernel, rewritten by the commit kernel
    int32_t max_blocks;
    const char *stub_copy;
    const char *stub_rot;
    int64_t total_stub;
    const float4 *table; // [num_seqs][head_dim/2]
    uint32_t *status;
    const uint32_t *gate;
    int64_t total_tiles;
    int32_t num_seqs;
    RemapSeq seq[kMaxSeqsPerLaunch];
};

// Debug check of a relocation in one pool: mark the source slots, then test
// the destination slots (bitmap of num_slots bits).
struct OverlapParams {
    const int32_t *tok_off;
    const int32_t *src_slots;
    const int32_t *chunk_req;
    const int32_t *chunk_dst_pos;
    const int32_t *block_tables;
    int32_t num_chunks, num_reqs, max_blocks, block;
    int64_t total_tokens;
    int64_t num_slots;  // of the destination pool
    int64_t num_blocks;
    uint32_t *bitmap;
    uint32_t *status;
};

// Debug check of a splice: every used block-table entry marked once.
struct DupBlockParams {
    const int32_t *block_tables;
    const int32_t *used; // entries used per block-table row [rows]
    int32_t rows, max_blocks;
    int64_t num_blocks;
    uint32_t *bitmap;
    uint32_t *status;
};

struct TableParams {
    const int32_t *d_delta;             // per-unit shifts in device memory, or ...
    int32_t h_delta[kMaxSeqsPerLaunch]; // ... carried in the launch (d_delta == nullptr)
    int32_t units;
    int32_t half;     // frequencies per head
    int32_t head_dim; // d
    double base;
    float4 *table;
};

// Content-defined chunking of token streams (kv_cdc).
struct CdcParams {
    const int64_t *stream_off; // [num_streams + 1]
    int32_t num_streams;
    int64_t total;             // tokens
    const int32_t *tokens;
    uint64_t gear_seed, threshold, fp_seed;
    int64_t max_chunks;
    int64_t *chunk_end;        // [max_chunks]
    uint64_t *fingerprint;     // [max_chunks]
    int64_t *num_chunks;       // device scalar
    uint32_t *status;
    uint32_t *flags;           // workspace: one word per 32 positions
    int64_t *block_count;      // workspace: chunk ends per block
    int64_t *block_last;       // workspace: last chunk end in the block, or -1
    int64_t *block_off;        // workspace: chunks before the block
    int64_t *block_prev_end;   // workspace: last chunk end before the block, or 0
    int32_t blocks;
};

// Fingerprints of token ranges (kv_fingerprint).
struct FingerprintParams {
    const int32_t *tokens;
    int64_t total;
    const int64_t *start;
    const int64_t *end;
    int64_t count;
    uint64_t seed;
    uint64_t *fingerprint;
    uint32_t *status;
};

} // namespace kvr

/*
 * kvreloc.h -- C ABI of the GB300 (sm_103a) KV relocation / splice / patch library.
 *
 * The library moves rows of a paged, bf16 KV cache on one GPU:
 *   - kv_relocate  copies cached rows into new slots.  The position-free part
 *                  of each row (the MLA latent c_KV, or the GQA V) is copied
 *                  verbatim; the RoPE part (MLA k_pe, or every head of the GQA
 *                  K) is rotated in closed form by R(δ), δ = p_target - p_source.
 *                  [Irminsul: MLA-native position-independent cache, §2.1 and
 *                  §2.2; Kamera: unified position-invariant KV cache, §2]
 *   - kv_splice    applies one Leyline directive D = (s_start, s_end, R, m) per
 *                  sequence: writes the prefilled stub R at s_start and shifts
 *                  every downstream row by Δ = |R| - |S| in place, rotating its
 *                  RoPE part by R(Δ).  [Leyline: KV-cache directives for agentic
 *                  inference, §2.1 directive, §2.2 δ-rotation, §2.3 integration]
 *   - kv_patch     adds Kamera's rank-m conditioning patch U_m V_mᵀ to stored
 *                  rows; the same patch can be fused into kv_relocate.
 *                  [Kamera §2: KV^(B|A) = R(δ)·KV(B|∅) + U_m V_mᵀ]
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers named d_* and every pointer inside kv_pool_desc / kv_patch_desc
 *    are DEVICE pointers; h_* pointers are host memory.
 *  - The caller owns all memory.  The library allocates nothing: its scratch
 *    state lives in the caller's workspace (size from kv_workspace_size()).
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *    Argument errors are reported synchronously, before anything is enqueued,
 *    and then nothing is modified.  Errors found on the device (an index
 *    outside its pool or table, a bounded wait that ran out) are recorded in
 *    the workspace status word and read with kv_get_device_status(); the
 *    offending rows are skipped, nothing outside the pools is touched, and no
 *    kernel traps.
 *  - One workspace serves one call at a time: calls that share a workspace
 *    must be ordered (same stream, or synchronised).
 *  - Rotation convention: "rotate-half" by default.  On a rotary vector of d
 *    elements, pair j is (x[j], x[j+d/2]), j < d/2, with frequency
 *    θ_j = base^(-2j/d); R(δ) turns pair j by the angle δ·θ_j:
 *       y[j] = x[j]·cos - x[j+d/2]·sin,  y[j+d/2] = x[j]·sin + x[j+d/2]·cos.
 *    A pool with pair_convention = 1 stores interleaved pairs (x[2j], x[2j+1])
 *    instead (same θ_j); source and destination pools must agree.
 *    The angle and its cosine/sine are formed in fp64 (one small table per
 *    call); the rotation runs in fp32 registers with compensated products and
 *    one round-to-nearest-even to bf16.  R(0) is the identity, bit for bit.
 *  - Layout: element e of the copy part of slot s in layer l is the bf16 at
 *       copy_base + l*copy_layer_stride + s*copy_slot_stride + e   (elements)
 *    and element (head h, i) of the rotary part is at
 *       rot_base + l*rot_layer_stride + s*rot_slot_stride + h*rot_head_dim + i.
 *    An MLA pool of rows c_KV[512] ‖ k_pe[64] is described by
 *    copy_base = pool, rot_base = pool + 512, both slot strides 576.
 *    Logical position p of request (or sequence) q is slot
 *       block_tables[q*max_blocks + p/block_size]*block_size + p%block_size.
 *  - Alignment: copy_base, rot_base and every stride must give 16-byte aligned
 *    rows (strides multiples of 8 elements); copy_dim % 8 == 0;
 *    rot_head_dim % 16 == 0.  Patch factors: 16-byte aligned, strides
 *    multiples of 4 floats, rank a multiple of 4.  Index arrays are naturally
 *    aligned (4 bytes for int32, 8 for int64); a misaligned one is rejected
 *    with KV_ERR_INVALID_ARG.
 */
#ifndef KVRELOC_H
#define KVRELOC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *kv_stream_t;

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, stride, alignment or directive */
    KV_ERR_OUT_OF_RANGE = 2, /* (device) a slot, block id or request index outside its pool/table */
    KV_ERR_CAPACITY = 3,     /* kv_splice: block table row too short for seq_len + Δ;
                                (device) kv_cdc: more chunks than max_chunks */
    KV_ERR_WORKSPACE = 4,    /* workspace NULL, misaligned or smaller than needed */
    KV_ERR_TIMEOUT = 5,      /* (device) a bounded inter-block wait ran out */
    KV_ERR_CUDA = 6,         /* a CUDA runtime call failed */
    KV_ERR_UNSUPPORTED = 7,  /* a layout the kernels do not handle */
    KV_ERR_OVERLAP = 8       /* (device, debug checks on) kv_relocate: a destination slot is
                                also a source slot of the call in the same pool; kv_splice,
                                kv_splice_composed: a block id appears twice among the
                                block-table entries the call uses.  Nothing is stored. */
} kv_status;

/* Leyline directive modes (Leyline §2.1). */
typedef enum {
    KV_AMORTIZE = 0,      /* splice in place, shift + rotate downstream rows */
    KV_FORGET = 1,        /* move nothing; truncate to s_start for a re-prefill */
    KV_AMORTIZE_REMAP = 2 /* AMORTIZE; block-aligned directives move whole blocks by
                             permuting the block-table row (see kv_splice) */
} kv_mode;

/* One paged KV pool (device memory, bf16 elements, strides in elements). */
typedef struct {
    int32_t num_layers;        /* L */
    int32_t block_size;        /* tokens per paged block (64 in the benchmarks) */
    int64_t num_slots;         /* slots per layer; a multiple of block_size */
    void *copy_base;           /* verbatim part: MLA c_KV, or GQA V */
    int64_t copy_layer_stride;
    int64_t copy_slot_stride;
    int32_t copy_dim;          /* 512 (MLA) or H*D (GQA) */
    void *rot_base;            /* rotated part: MLA k_pe, or GQA K */
    int64_t rot_layer_stride;
    int64_t rot_slot_stride;
    int32_t rot_heads;         /* 1 (MLA) or H (GQA) */
    int32_t rot_head_dim;      /* 64 (MLA) or 128 (GQA) */
    double rope_base;          /* 10000, 500000, ... */
    int32_t pair_convention;   /* 0: rotate-half pairs (x[j], x[j+d/2]);
                                  1: interleaved pairs (x[2j], x[2j+1]), same θ_j */
} kv_pool_desc;

/* Rank-m patch factors, one (U, V) pair per channel: index 0 patches the
 * copy part, index 1 the rotated part; a NULL u or v leaves that channel
 * unpatched (the same arrays may serve both channels).  fp32:
 *   U(l, t, r)      = u[l*u_layer_stride + t*u_tok_stride + r]
 *   V(l, c, col, r) = v[l*v_layer_stride + c*v_chunk_stride + col*v_col_stride + r]
 * t is the token's U row and c the chunk's V slot; col is the column inside
 * the channel (rotated part: head*rot_head_dim + i).  Each patched value
 * becomes rnd(x + Σ_r U(l,t,r)·V(l,c,col,r)), x the copied or (fused into
 * kv_relocate) the unrounded rotated value.  By default t is the token's
 * index in the call (tok_off[c] + offset in chunk c) and c the chunk's index
 * in the call.  Factors kept once per canonical chunk and reused by any
 * later call (Kamera §3: reorder under one orbit patch, recall of an evicted
 * chunk) are addressed through the optional device maps instead, for both
 * channels:
 *   d_u_chunk_tok[c]  U row of chunk c's first token (its tokens follow it),
 *   d_v_chunk[c]      V slot of chunk c;
 * u_rows[ch] and v_slots[ch], when nonzero, are the extents of channel ch's
 * factor arrays (U rows per layer, V slots per layer): a token whose U row
 * (mapped or in call order) or a chunk whose V slot falls outside them is
 * skipped and sets KV_ERR_OUT_OF_RANGE in the device status, like an index
 * outside a pool.  0 leaves that extent unchecked (the caller then keeps every
 * row and slot inside the arrays).  An MLA patch over the 576-wide row is one
 * factor pair: u[0] = u[1], v[1] = v[0] + 512*v_col_stride. */
typedef struct {
    int32_t rank; /* m: 4..64, a multiple of 4 */
    const float *u[2];
    int64_t u_layer_stride[2];
    int64_t u_tok_stride[2];
    const float *v[2];
    int64_t v_layer_stride[2];
    int64_t v_chunk_stride[2];
    int64_t v_col_stride[2];
    const int64_t *d_u_chunk_tok; /* NULL: the call's token order */
    const int32_t *d_v_chunk;     /* NULL: the call's chunk order */
    int64_t u_rows[2];            /* U rows per layer; 0 = unchecked */
    int64_t v_slots[2];           /* V slots per layer; 0 = unchecked */
} kv_patch_desc;

/* Bytes of device workspace needed by any call on `pool` that moves at most
 * `max_rows` rows per layer in total (relocate/patch: tokens; splice:
 * downstream rows plus stub rows over all sequences of the call) and has at
 * most `max_units` chunks (relocate, patch) or sequences (splice).  The
 * workspace must be 256-byte aligned.  Returns 0 for an invalid pool. */
size_t kv_workspace_size(const kv_pool_desc *pool, int64_t max_rows, int32_t max_units);

/* Gather chunks of cached rows from `src` into `dst` (Irminsul §2.2, Kamera §2).
 * Chunk c covers tokens t = d_tok_off[c] .. d_tok_off[c+1]-1 (d_tok_off has
 * num_chunks+1 non-decreasing entries, d_tok_off[0] = 0,
 * d_tok_off[num_chunks] = total_tokens).  Token t is read from source slot
 * d_src_slots[t] and written to logical position d_chunk_dst_pos[c] +
 * (t - d_tok_off[c]) of request d_chunk_req[c] in d_block_tables
 * ([num_reqs][max_blocks] int32).  Its copy part is copied verbatim; each
 * rotary head is turned by R(d_delta[c]).  `patch` (NULL = none) adds the
 * rank-m patch before the single rounding.
 * src and dst may be the same pool when no destination slot is also a source
 * slot: the call is not in place, and overlapping slots give undefined rows
 * unless the debug checks are on (kv_set_debug_checks), which then report
 * KV_ERR_OVERLAP and store nothing.
 * Shapes (num_layers, copy_dim, rot_heads, rot_head_dim, rope_base) of src
 * and dst must match. */
kv_status kv_relocate(const kv_pool_desc *src, const kv_pool_desc *dst, int32_t num_chunks,
                      int64_t total_tokens, const int32_t *d_tok_off, const int32_t *d_src_slots,
                      const int32_t *d_chunk_req, const int32_t *d_chunk_dst_pos,
                      const int32_t *d_delta, const int32_t *d_block_tables, int32_t num_reqs,
                      int32_t max_blocks, const kv_patch_desc *patch, void *d_workspace,
                      size_t workspace_bytes, kv_stream_t stream);

/* Apply one directive per sequence, in place (Leyline §2.1-§2.3).
 * Sequence q uses block-table row q of d_block_tables ([num_seqs][max_blocks]),
 * has h_seq_lens[q] tokens and the directive
 *   (h_s_start[q], h_s_end[q], R = h_stub_len[q] prefilled rows, mode)
 * with 0 <= s_start <= s_end <= seq_len (half-open span S = [s_start, s_end)).
 * The stub rows of all sequences are stored back to back, in sequence order:
 *   d_stub_copy [L][Σ h_stub_len][copy_dim],
 *   d_stub_rot  [L][Σ h_stub_len][rot_heads*rot_head_dim]
 * (contiguous bf16, 16-byte aligned; may be NULL when Σ h_stub_len = 0).
 * AMORTIZE: rows [0, s_start) stay; the stub is written verbatim at
 * [s_start, s_start+|R|); the row at s_end+k moves to s_end+Δ+k with its
 * copy part verbatim and its rotary part turned by R(Δ), Δ = |R| - |S|;
 * h_seq_lens[q] becomes seq_len + Δ.  Slots at or beyond the new length keep
 * whatever they held.  Needs ceil(max(seq_len, seq_len+Δ)/block_size) <=
 * max_blocks (else KV_ERR_CAPACITY); the caller owns the blocks of every
 * entry used, distinct across the whole call (checked, with KV_ERR_OVERLAP
 * and nothing stored, when the debug checks are on).  The in-place shift is
 * overlap-safe for Δ of either sign.
 * FORGET: moves nothing and sets h_seq_lens[q] = s_start (the caller
 * re-prefills from there); no device work.
 * AMORTIZE_REMAP: the logical result of AMORTIZE.  A sequence whose directive
 * is block-aligned (s_start, s_end and |R| multiples of block_size) and
 * shifts (Δ != 0) keeps its downstream rows in their physical blocks: only
 * their rotary part is rewritten (R(Δ) in place) and its block-table row is
 * permuted ON THE DEVICE -- with A = s_start/B, the row becomes [entries
 * 0..A) [|R|/B blocks for the stub: the span's blocks first, then the row's
 * entries after the downstream blocks] [the downstream blocks] [the entries
 * left, in order].  After the call the device row is authoritative; entries
 * at or beyond the new length remain the sequence's.  Other sequences (and
 * every sequence when max_blocks > 49152) take the AMORTIZE path and keep
 * their rows.  d_block_tables is only written in this mode.
 * h_seq_lens is updated when the call returns KV_OK (the data movement itself
 * completes in stream order). */
kv_status kv_splice(const kv_pool_desc *pool, int32_t num_seqs, int32_t *d_block_tables,
                    int32_t max_blocks, int32_t *h_seq_lens, const int32_t *h_s_start,
                    const int32_t *h_s_end, const int32_t *h_stub_len, const void *d_stub_copy,
                    const void *d_stub_rot, kv_mode mode, void *d_workspace,
                    size_t workspace_bytes, kv_stream_t stream);

/* Several directives per sequence applied as ONE in-place edit (Leyline
 * §2.1-§2.3 composed with the closure R(a)R(b) = R(a+b)).  Sequence q gets
 * num_dirs directives in order; directive i is
 *   (h_s_start[i*num_seqs + q], h_s_end[i*num_seqs + q], h_stub_len[i*num_seqs + q])
 * in the indexing that directives 0..i-1 left, exactly as num_dirs successive
 * kv_splice calls would take them.  Stub rows are stored directive by
 * directive and, within a directive, sequence by sequence (the stub arrays
 * of the successive calls back to back):
 *   d_stub_copy [L][Σ h_stub_len][copy_dim], d_stub_rot [L][Σ h_stub_len][rot width].
 * Every row of the final sequence is written once, from its origin (an
 * original row, or a stub row at the position its directive wrote it), its
 * rotary part turned by the total shift it underwent and rounded once --
 * where successive kv_splice calls round after every directive.  Rows whose
 * total shift is 0 are not touched.  Only the final length is checked
 * against max_blocks (KV_ERR_CAPACITY); h_seq_lens becomes the final
 * lengths when the call returns KV_OK.  AMORTIZE semantics only.  The
 * workspace size depends on the directives: kv_splice_composed_workspace_size
 * (0 when the directives are invalid).  The plan is built on the host and
 * copied into the workspace on `stream`. */
size_t kv_splice_composed_workspace_size(const kv_pool_desc *pool, int32_t num_seqs,
                                         int32_t num_dirs, const int32_t *h_seq_lens,
                                         const int32_t *h_s_start, const int32_t *h_s_end,
                                         const int32_t *h_stub_len);
kv_status kv_splice_composed(const kv_pool_desc *pool, int32_t num_seqs, int32_t num_dirs,
                             const int32_t *d_block_tables, int32_t max_blocks,
                             int32_t *h_seq_lens, const int32_t *h_s_start, const int32_t *h_s_end,
                             const int32_t *h_stub_len, const void *d_stub_copy,
                             const void *d_stub_rot, void *d_workspace, size_t workspace_bytes,
                             kv_stream_t stream);

/* One tile of a composed splice plan, as kv_splice_composed_plan reports it:
 * n (<= tile rows) rows moving from logical positions src_lo.. (or global
 * stub rows src_lo.. when stub = 1) to logical positions dst_lo.. of
 * sequence seq, rotary part turned by the shift h_deltas[unit] (unit = -1:
 * no rotation).  dep[0..1] and dep[2..3] are two inclusive ranges of tiles
 * (indices into the plan, all smaller than this tile's) whose source rows
 * this tile's destination overlaps; -1 = none.  Tiles run in index order of
 * their tickets. */
typedef struct {
    int64_t src_lo;
    int64_t dst_lo;
    int32_t n;
    int32_t seq;
    int32_t unit;
    int32_t stub;
    int32_t dep[4];
} kv_splice_tile;

/* The composed splice's plan, for inspection (host only, no device work):
 * writes up to max_tiles tiles to h_tiles and up to max_units shifts to
 * h_deltas (either may be NULL) and the counts to *n_tiles, *n_units.
 * Argument errors as kv_splice_composed (capacity is not checked here). */
kv_status kv_splice_composed_plan(const kv_pool_desc *pool, int32_t num_seqs, int32_t num_dirs,
                                  const int32_t *h_seq_lens, const int32_t *h_s_start,
                                  const int32_t *h_s_end, const int32_t *h_stub_len,
                                  kv_splice_tile *h_tiles, int64_t max_tiles, int32_t *h_deltas,
                                  int32_t max_units, int64_t *n_tiles, int32_t *n_units);

/* Add the rank-m patch to stored rows in place (Kamera §2), one rounding per
 * value.  Chunks are described as in kv_relocate: the tokens of chunk c sit
 * at logical positions d_chunk_dst_pos[c] + i of request d_chunk_req[c]. */
kv_status kv_patch(const kv_pool_desc *pool, int32_t num_chunks, int64_t total_tokens,
                   const int32_t *d_tok_off, const int32_t *d_chunk_req,
                   const int32_t *d_chunk_dst_pos, const int32_t *d_block_tables,
                   int32_t num_reqs, int32_t max_blocks, const kv_patch_desc *patch,
                   void *d_workspace, size_t workspace_bytes, kv_stream_t stream);

/* Allocation-free variant of kv_relocate.  The source pages have no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory: code running inside a runtime whose allocator owns all of the GPU
 * (for example a serving engine that hands out pre-reserved HBM to its
 * plugins and forbids further cudaMalloc), or latency-critical paths where an
 * allocation and its implicit synchronisation are not acceptable.  Such a
 * caller still passes the pools, index arrays and patch factors; the scratch
 * that kv_relocate takes from its workspace (a status word and the per-chunk
 * cos/sin table) comes instead from a fixed 2 MiB device array inside the
 * library.  Every GPU that loads the library holds that array until the
 * process exits.
 *  - Limit: the table holds up to 4095 chunks for MLA rows (64-dim k_pe) and
 *    2047 chunks for 8 x 128 GQA rows; larger num_chunks is rejected with
 *    KV_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents;
 *    each call clears its status word first.  Calls that overlap on the GPU
 *    (different streams, not ordered) race on the array: order them.
 *  - h_device_status: when non-NULL the call waits for `stream` and stores
 *    the device status (KV_OK, KV_ERR_OUT_OF_RANGE, or KV_ERR_OVERLAP with
 *    the debug checks on) there; when NULL the call stays asynchronous and
 *    device-side errors are not reported.
 *  - With the debug checks on (kv_set_debug_checks) and src, dst the same
 *    pool, the overlap bitmap (one bit per slot) must also fit in the array,
 *    else the call is rejected with KV_ERR_WORKSPACE.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments otherwise as kv_relocate. */
kv_status kv_relocate_noalloc(const kv_pool_desc *src, const kv_pool_desc *dst,
                              int32_t num_chunks, int64_t total_tokens, const int32_t *d_tok_off,
                              const int32_t *d_src_slots, const int32_t *d_chunk_req,
                              const int32_t *d_chunk_dst_pos, const int32_t *d_delta,
                              const int32_t *d_block_tables, int32_t num_reqs,
                              int32_t max_blocks, const kv_patch_desc *patch,
                              int32_t *h_device_status, kv_stream_t stream);

/* Wait for `stream`, then return the device status of the last call that
 * used this workspace (KV_OK, KV_ERR_OUT_OF_RANGE, KV_ERR_CAPACITY from
 * kv_cdc, KV_ERR_TIMEOUT, or KV_ERR_OVERLAP with the debug checks on), or
 * KV_ERR_CUDA if the synchronisation or the read failed. */
kv_status kv_get_device_status(const void *d_workspace, kv_stream_t stream);

/* ---------------------------------------------------------------------
 * Content-defined chunking of token streams
 * [Irminsul: MLA-native position-independent cache, §2.2, content hash
 * keying with CDC and the fixed-window fallback S1]
 *
 * The registry that kv_relocate serves is keyed by content: a Gear rolling
 * hash over windows of 64 tokens ends a chunk where it falls below a
 * threshold, so chunk boundaries follow the tokens, not their offsets, and
 * each chunk is named by its xxHash64 fingerprint.  The pages fix neither the
 * Gear table nor the threshold; this library defines them as follows:
 *   h(i) = 2*h(i-1) + G(x_i) modulo 2^64, with h = 0 before the first token of
 *          every stream, so h(i) holds exactly the last 64 tokens;
 *   G(x) = output number x (counting from 0) of the SplitMix64 generator seeded
 *          with gear_seed (token ids read as unsigned 32-bit numbers);
 *   a chunk ends after token i when h(i) < threshold (mean chunk length
 *          2^64 / threshold tokens), and at the end of its stream;
 *   fingerprint = XXH64 of the chunk's token ids as 4-byte little-endian
 *          words, seeded with fp_seed.
 * ------------------------------------------------------------------- */

/* Workspace bytes kv_cdc needs for `total_tokens` tokens (256-byte aligned). */
size_t kv_cdc_workspace_size(int64_t total_tokens);

/* Chunk num_streams token streams, concatenated in d_tokens: stream s is
 * tokens d_stream_off[s] .. d_stream_off[s+1]-1 (num_streams+1 int64 device
 * entries, non-decreasing, first 0, last total_tokens; empty streams have no
 * chunk).  Writes, in stream order, each chunk's exclusive end (a global
 * token offset; a chunk starts where the previous one ends, the first at 0)
 * to d_chunk_end[k] and its fingerprint to d_fingerprint[k], for
 * k < max_chunks, and the number of chunks to the device scalar
 * *d_num_chunks.  More chunks than max_chunks set the device status
 * KV_ERR_CAPACITY (total_tokens chunks always fit); offsets that do not start
 * at 0 or end at total_tokens set KV_ERR_OUT_OF_RANGE.  Three kernels. */
kv_status kv_cdc(int32_t num_streams, const int64_t *d_stream_off, int64_t total_tokens,
                 const int32_t *d_tokens, uint64_t gear_seed, uint64_t threshold,
                 uint64_t fp_seed, int64_t max_chunks, int64_t *d_chunk_end,
                 uint64_t *d_fingerprint, int64_t *d_num_chunks, void *d_workspace,
                 size_t workspace_bytes, kv_stream_t stream);

/* Fingerprints of arbitrary token ranges: d_fingerprint[k] = XXH64 of tokens
 * d_start[k] .. d_end[k]-1 (device int64 arrays, 0 <= start <= end <=
 * total_tokens), seeded with fp_seed.  The fixed-window fallback passes
 * consecutive windows of 128 tokens.  A range outside the tokens is skipped
 * and sets KV_ERR_OUT_OF_RANGE in the workspace status word (only the
 * 256-byte header of the workspace is used).  One kernel. */
kv_status kv_fingerprint(int64_t num_ranges, const int64_t *d_start, const int64_t *d_end,
                         int64_t total_tokens, const int32_t *d_tokens, uint64_t fp_seed,
                         uint64_t *d_fingerprint, void *d_workspace, size_t workspace_bytes,
                         kv_stream_t stream);

/* Debug checks of the caller contracts that the in-place kernels rely on
 * (process-wide; off by default).  When on:
 *  - kv_relocate (and kv_relocate_noalloc) on a source and destination that
 *    are the same pool (the same copy_base or the same rot_base) first marks
 *    every source slot in a bitmap, then tests every destination slot against
 *    it: a destination slot that is also a source slot of the call would be
 *    read and written by different blocks in no fixed order (Irminsul §2.2:
 *    the relocation gathers stored rows into new slots);
 *  - kv_splice and kv_splice_composed mark every block-table entry the call
 *    uses (ceil(max(old length, new length) / block_size) per sequence): a
 *    block id that appears twice would make two logical positions share a
 *    slot, and the in-place shift (Leyline §2.1-§2.3) would race on it.
 * Either finding sets KV_ERR_OVERLAP in the device status, and the call's
 * row-moving kernels then store nothing (the pools and block tables stay bit
 * for bit as they were).  Cost when on: the workspace grows by one bit per
 * slot of the destination pool, rounded up to 256 bytes (kv_workspace_size
 * and kv_splice_composed_workspace_size always include it), plus one memset
 * of that bitmap and one or two scan kernels over the call's index arrays (a
 * few bytes per token or block-table entry, against the kilobytes per token
 * that the rows move).  Cost when off: none -- the scans are not launched and
 * no kernel reads anything more. */
void kv_set_debug_checks(int32_t on);

/* Upper bound, in nanoseconds, of every inter-block wait inside kv_splice
 * (default 2e9).  Values <= 0 restore the default.  Process-wide. */
void kv_set_wait_limit_ns(int64_t limit_ns);

/* Test hook for the failure path of the in-place splices (process-wide; -1,
 * the default, turns it off).  The tile of each kv_splice / kv_splice_composed
 * launch that draws ticket `ticket` does not publish that it has read its
 * rows; the tiles whose destination overlaps those rows then wait in vain
 * until the wait limit, record KV_ERR_TIMEOUT, skip their stores and keep
 * publishing, so the launch still finishes.  Lets a test run the kernels' own
 * timeout branch without faulting or hanging a GPU (give it a short
 * kv_set_wait_limit_ns). */
void kv_set_splice_skip_publish(int64_t ticket);

/* Run the bounded wait used by kv_splice on a workspace flag that nothing
 * sets, with the given limit; the device status afterwards is
 * KV_ERR_TIMEOUT.  Exercises the failure path without faulting a GPU. */
kv_status kv_check_wait_timeout(void *d_workspace, size_t workspace_bytes, int64_t limit_ns,
                                kv_stream_t stream);

/* Timing hook.  When both are non-NULL (cudaEvent_t handles), every later
 * call on this thread records `start_event` on its stream just before its
 * row-moving kernel(s) and `stop_event` just after, so the caller can time
 * that kernel alone with cudaEventElapsedTime.  NULL, NULL turns it off. */
void kv_set_kernel_events(void *start_event, void *stop_event);

/* Number of kernels the most recent successful call on this thread enqueued. */
int32_t kv_last_launch_count(void);

/* Short English name of a status code (static storage). */
const char *kv_status_string(kv_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t kv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVRELOC_H */

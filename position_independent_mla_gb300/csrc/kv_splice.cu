// kv_splice.cu -- the in-place, overlap-safe Leyline splice (AMORTIZE).
//
// Leyline §2.2-§2.3: with Δ = |R| - |S|, every downstream row s_end + k moves
// to s_end + Δ + k; its verbatim part is kept and its rotary part turned by
// R(Δ); the prefilled stub R is written verbatim at s_start.
//
// The shift happens in place through the sequence's block table, so a row
// may only be overwritten after the row that lived there has been read.
// The downstream rows of a sequence are cut into tiles of T rows, numbered
// in the order that makes all hazards point backwards: ascending positions
// for Δ < 0 (rows move down), descending for Δ > 0 (rows move up).  The stub
// tiles come last.  A tile's destination range overlaps the source range of
// at most two earlier tiles.  Each block takes a ticket from an atomic
// counter (so tickets are handed out in launch order, and every tile a block
// waits for belongs to a block that is already running).  Every shift tile
// owns a counter of layer reads: once the eight row-moving warps' loads of a
// layer have landed, a ninth warp of the block, which moves no rows and so
// has no stores of its own in flight for its release to wait on, adds 8
// with a release reduction, so layer l is read when the counter reaches
// 8 (l + 1).  The warps signal it through a named barrier without waiting,
// and it publishes at once: reading needs nothing, since a tile's source
// rows are overwritten only by itself and by later tiles.  Then thread 0
// makes sure (acquire, bounded) that the tiles
// it overwrites have read this layer -- a value seen once covers all layers
// up to it, so a dependency far behind costs one poll for the whole tile --
// and after one barrier the rows are stored.  Because reads are published before any wait,
// a tile's wait chain runs back through at most one earlier tile per layer
// (its length is bounded by the layer count, not by the number of tiles).
// The earliest unfinished tile never waits on an unfinished one, so the
// protocol cannot deadlock; the bound on each wait turns any unforeseen
// stall into KV_ERR_TIMEOUT instead of a hang.
#include "kv_launch.h"
#include "kv_tiles.cuh"

namespace kvr {

constexpr uint32_t kWarps = kThreads / 32; // row-moving warps of a splice block
// threads of a splice block: the row-moving warps, then the publishing warp
constexpr int kSpliceThreads = kThreads + 32;
constexpr uint32_t kReadBar = 1; // named barrier: the warps' loads of a layer have landed
// resident blocks per SM to aim for: three 288-thread blocks leave each
// thread enough registers to hold its rows without local-memory spills
constexpr int kSpliceMinBlocks = 3;

// The publishing warp's part of one layer: wait until every row-moving warp
// has read the layer, add their 8 reads to `flag` with a release reduction
// (one lane; none when flag is null), then join the block's barrier.
__device__ __forceinline__ void publish_layer(uint32_t *flag)
{
    bar_wait_all(kReadBar, kSpliceThreads);
    if (flag != nullptr && (threadIdx.x & 31) == 0)
        red_release_add(flag, kWarps);
    __syncthreads();
}

// GR: the launch cuts tiles into layer groups (p.layer_groups > 1); without
// it the unit is the whole tile and the loop runs over every layer.
template <class G, bool IL, bool GR>
__global__ void __launch_bounds__(kSpliceThreads, kSpliceMinBlocks) splice_kernel(const __grid_constant__ SpliceParams p)
{
    __shared__ uint32_t s_ticket;
    __shared__ volatile int32_t s_abort; // 0 -> 1 once a wait ran out; never reset
    __shared__ int64_t s_dep[2];
    __shared__ uint32_t s_seen[2];
    __shared__ int64_t s_src[G::T];
    __shared__ int64_t s_dst[G::T];
    __shared__ int32_t s_ident[G::T];
    __shared__ float4 s_cs[G::kHalf];
    __shared__ uint32_t s_sink;

    if (gate_closed(p.gate))
        return; // a debug check found a duplicate block: every block leaves
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_ticket = atomicAdd(p.ticket, 1u);
        s_abort = 0;
    }
    __syncthreads();
    const int64_t t = s_ticket;
    if (t >= p.total_tickets)
        return;

    int q = 0;
    while (q + 1 < p.num_seqs && p.seq[q + 1].ticket_base <= t)
        ++q;
    const SpliceSeq &S = p.seq[q];
    // this unit: tile k of the sequence, layers [l0, l1) (group g of its layers)
    const int64_t u = t - S.ticket_base;
    const int32_t NG = GR ? p.layer_groups : 1;
    const int64_t shift_units = (int64_t)S.n_shift * NG;
    const bool shift = u < shift_units;
    const int64_t k = shift ? u / NG : S.n_shift + (u - shift_units) / NG;
    const int g = (int)(shift ? u % NG : (u - shift_units) % NG);
    const int32_t *bt = p.block_tables + (int64_t)S.bt_row * p.max_blocks;
    const int32_t B = p.pool.block;
    const int64_t nb = p.pool.num_blocks;
    const int l0 = GR ? g * p.group_layers : 0;
    const int l1 = GR ? min(p.pool.num_layers, l0 + p.group_layers) : p.pool.num_layers;

    // positions (shift tile) or stub rows (stub tile) covered: [lo, hi)
    int64_t lo, hi;
    if (shift) {
        if (S.delta < 0) {
            lo = S.s_end + k * G::T;
            hi = min(lo + (int64_t)G::T, (int64_t)S.seq_len);
        } else {
            hi = S.seq_len - k * G::T;
            lo = max(hi - (int64_t)G::T, (int64_t)S.s_end);
        }
    } else {
        lo = (k - S.n_shift) * G::T;
        hi = min(lo + (int64_t)G::T, (int64_t)S.n_r);
    }

    if (tid < G::T) {
        const int64_t i = lo + tid;
        int64_t src = -1, dst = -1;
        if (i < hi) {
            if (shift) {
                src = slot_of(bt, p.max_blocks, B, nb, i);
                dst = slot_of(bt, p.max_blocks, B, nb, i + S.delta);
            } else {
                src = S.stub_base + i;
                dst = slot_of(bt, p.max_blocks, B, nb, (int64_t)S.s_start + i);
            }
            if (src < 0 || dst < 0) {
                set_status(p.status, kStatusOutOfRange);
                src = dst = -1;
            }
        }
        s_src[tid] = src;
        s_dst[tid] = dst;
        s_ident[tid] = shift ? 0 : 1;
    }
    if (tid == 0) {
        // earlier tiles whose source rows this tile's destination overlaps
        s_dep[0] = s_dep[1] = -1;
        s_seen[0] = s_seen[1] = 0u;
        const int64_t dlo = shift ? lo + S.delta : (int64_t)S.s_start + lo;
        const int64_t dhi = shift ? hi + S.delta : (int64_t)S.s_start + hi;
        const int64_t a = max(dlo, (int64_t)S.s_end), b = min(dhi, (int64_t)S.seq_len);
        if (S.delta != 0 && S.n_shift > 0 && a < b) {
            int64_t j0, j1;
            if (S.delta < 0) {
                j0 = (a - S.s_end) / G::T;
                j1 = (b - 1 - S.s_end) / G::T;
            } else {
                j0 = (S.seq_len - b) / G::T;
                j1 = (S.seq_len - 1 - a) / G::T;
            }
            int n = 0;
            for (int64_t j = j0; j <= j1 && n < 2; ++j)
                if (!(shift && j == k))
                    s_dep[n++] = j;
        }
    }
    if (!p.inline_table)
        for (int j = tid; j < G::kHalf; j += kThreads)
            stage_cs<G, CsOrder<G, false, IL>::kPacked>(s_cs, j,
                                                     p.table[(int64_t)q * G::kHalf + j]);
    __syncthreads();

    if (tid >= kThreads) {
        // the publishing warp: a launch without a δ table has it form this
        // unit's cos/sin rows (fp64 angle reduction) while the row-moving
        // warps' first loads are in flight -- the rows reach shared memory
        // before the first layer's barrier, which the stores wait for --
        // then this unit's read counter, once per layer
        if (p.inline_table && shift)
            for (int j = tid - kThreads; j < G::kHalf; j += 32)
                stage_cs<G, CsOrder<G, false, IL>::kPacked>(
                    s_cs, j, delta_entry_call(S.delta, j, 2 * G::kHalf, p.rope_base));
        uint32_t *flag = shift && t != p.skip_publish ? p.flags + S.flag_base + k * NG + g
                                                       : nullptr;
        for (int l = l0; l < l1; ++l)
            publish_layer(flag);
        return;
    }
    const int64_t copy_row_bytes = (int64_t)G::CV * 16, rot_row_bytes = (int64_t)G::kRotW * 16;
    PatchAt none{nullptr, 0, nullptr, nullptr};
    for (int l = l0; l < l1; ++l) {
        const RowsAt pool_l{p.pool.copy + l * p.pool.copy_ls, p.pool.copy_ss,
                            p.pool.rot + l * p.pool.rot_ls, p.pool.rot_ss};
        const RowsAt from = shift ? pool_l
                                  : RowsAt{p.stub_copy + l * p.total_stub * copy_row_bytes,
                                           copy_row_bytes,
                                           p.stub_rot + l * p.total_stub * rot_row_bytes,
                                           rot_row_bytes};
        TileRegs<G> regs;
        if (!s_abort)
            load_tile<G>(from, s_src, regs);
        else
            regs = TileRegs<G>{};
        // make every load complete before the barrier (see fold_tile)
        const uint32_t f = fold_tile<G>(regs);
        if (p.total_tickets < 0)
            s_sink = f;
        // this warp's share of layer l is in registers: let the publishing
        // warp count it now, before waiting on anyone, so that a tile's
        // progress never waits on the tiles behind it (its source rows are
        // overwritten only by itself and by later tiles)
        bar_arrive(kReadBar, kSpliceThreads);
        // every warp of the same layer group of a tile has read layer l
        const uint32_t want = ((uint32_t)(l - l0) + 1u) * kWarps;
        if (tid == 0 && !s_abort) {
            // the tiles this one overwrites must have read layer l
            for (int d = 0; d < 2; ++d) {
                if (s_dep[d] < 0 || s_seen[d] >= want)
                    continue;
                const uint32_t seen = wait_count(p.flags + S.flag_base + s_dep[d] * NG + g, want,
                                                 p.wait_limit_ns);
                if (seen < want) {
                    set_status(p.status, kStatusTimeout);
                    s_abort = 1;
                    break;
                }
                s_seen[d] = seen;
            }
        }
        __syncthreads();
        if (!s_abort)
            store_tile<G, false, true, IL>(pool_l, s_dst, regs, s_cs, 0, s_ident, none);
    }
}

cudaError_t launch_splice(const SpliceParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.total_tickets == 0)
        return cudaSuccess;
    if (p.total_tickets > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    const unsigned blocks = (unsigned)p.total_tickets;
    return with_inplace_geo(kind, [&](auto g) {
        return with_bool(p.pool.il != 0, [&](auto il) {
            return with_bool(p.layer_groups > 1, [&](auto gr) {
                splice_kernel<typename decltype(g)::type, decltype(il)::value,
                              decltype(gr)::value><<<blocks, kSpliceThreads, 0, stream>>>(p);
                return cudaGetLastError();
            });
        });
    });
}

// ---------------------------------------------------------------------------
// Composed splice: several directives per sequence as one in-place edit.
//
// The host turns the directives into a table of tiles (each: T rows moving by
// one constant shift, or stub rows landing at their final positions) ordered
// so that every tile a tile overwrites comes earlier: rows moving down in
// ascending order, rows moving up in descending order, stubs last (the map
// is monotone, so rows moving down and rows moving up never overlap).  The
// protocol is the splice's: tickets, release counts of the layers read (from
// the publishing warp), bounded acquire waits on the (at most two ranges of)
// earlier tiles a tile overwrites, one barrier per layer.  Every row is read once and rounded
// once, its rotary part turned by its total shift.
// ---------------------------------------------------------------------------

template <class G, bool IL>
__global__ void __launch_bounds__(kSpliceThreads, kSpliceMinBlocks)
splice_composed_kernel(const __grid_constant__ ComposedParams p)
{
    __shared__ uint32_t s_ticket;
    __shared__ volatile int32_t s_abort;
    __shared__ uint32_t s_min[2]; // smallest count seen over each dependency range
    __shared__ int64_t s_src[G::T];
    __shared__ int64_t s_dst[G::T];
    __shared__ int32_t s_ident[G::T];
    __shared__ float4 s_cs[G::kHalf];
    __shared__ uint32_t s_sink;

    if (gate_closed(p.gate))
        return; // a debug check found a duplicate block: every block leaves
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_ticket = atomicAdd(p.ticket, 1u);
        s_abort = 0;
        s_min[0] = s_min[1] = 0u;
    }
    __syncthreads();
    const int64_t t = s_ticket;
    if (t >= p.num_tiles)
        return;
    const SpliceTile tile = p.tiles[t];
    const int32_t *bt = p.block_tables + (int64_t)tile.seq * p.max_blocks;
    const int32_t B = p.pool.block;
    const int64_t nb = p.pool.num_blocks;
    const int L = p.pool.num_layers;
    if (tid < G::T) {
        int64_t src = -1, dst = -1;
        if (tid < tile.n) {
            src = tile.stub ? tile.src_lo + tid : slot_of(bt, p.max_blocks, B, nb, tile.src_lo + tid);
            dst = slot_of(bt, p.max_blocks, B, nb, tile.dst_lo + tid);
            if (src < 0 || dst < 0 || (tile.stub && src >= p.total_stub)) {
                set_status(p.status, kStatusOutOfRange);
                src = dst = -1;
            }
        }
        s_src[tid] = src;
        s_dst[tid] = dst;
        s_ident[tid] = tile.unit < 0;
    }
    if (tile.unit >= 0)
        for (int j = tid; j < G::kHalf; j += kThreads)
            stage_cs<G, CsOrder<G, false, IL>::kPacked>(s_cs, j,
                                                     p.table[(int64_t)tile.unit * G::kHalf + j]);
    __syncthreads();

    if (tid >= kThreads) {
        // the publishing warp: this tile's read counter, once per layer
        uint32_t *flag = !tile.stub && t != p.skip_publish ? p.flags + t : nullptr;
        for (int l = 0; l < L; ++l)
            publish_layer(flag);
        return;
    }
    const int64_t copy_row_bytes = (int64_t)G::CV * 16, rot_row_bytes = (int64_t)G::kRotW * 16;
    PatchAt none{nullptr, 0, nullptr, nullptr};
    for (int l = 0; l < L; ++l) {
        const RowsAt pool_l{p.pool.copy + l * p.pool.copy_ls, p.pool.copy_ss,
                            p.pool.rot + l * p.pool.rot_ls, p.pool.rot_ss};
        const RowsAt from = tile.stub ? RowsAt{p.stub_copy + l * p.total_stub * copy_row_bytes,
                                               copy_row_bytes,
                                               p.stub_rot + l * p.total_stub * rot_row_bytes,
                                               rot_row_bytes}
                                      : pool_l;
        TileRegs<G> regs;
        if (!s_abort)
            load_tile<G>(from, s_src, regs);
        else
            regs = TileRegs<G>{};
        const uint32_t f = fold_tile<G>(regs);
        if (p.num_tiles < 0)
            s_sink = f;
        // this warp's share of layer l is read: counted before any wait
        bar_arrive(kReadBar, kSpliceThreads);
        const uint32_t want = ((uint32_t)l + 1u) * kWarps;
        if (tid == 0 && !s_abort) {
            for (int r = 0; r < 2 && !s_abort; ++r) {
                const int32_t lo = tile.dep[2 * r], hi = tile.dep[2 * r + 1];
                if (lo < 0 || s_min[r] >= want)
                    continue;
                uint32_t mn = 0xFFFFFFFFu;
                for (int32_t j = lo; j <= hi; ++j) {
                    const uint32_t seen = wait_count(p.flags + j, want, p.wait_limit_ns);
                    if (seen < want) {
                        set_status(p.status, kStatusTimeout);
                        s_abort = 1;
                        break;
                    }
                    mn = min(mn, seen);
                }
                s_min[r] = mn;
            }
        }
        __syncthreads();
        if (!s_abort)
            store_tile<G, false, true, IL>(pool_l, s_dst, regs, s_cs, 0, s_ident, none);
    }
}

cudaError_t launch_splice_composed(const ComposedParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.num_tiles == 0)
        return cudaSuccess;
    if (p.num_tiles > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    const unsigned blocks = (unsigned)p.num_tiles;
    return with_inplace_geo(kind, [&](auto g) {
        return with_bool(p.pool.il != 0, [&](auto il) {
            splice_composed_kernel<typename decltype(g)::type, decltype(il)::value>
                <<<blocks, kSpliceThreads, 0, stream>>>(p);
            return cudaGetLastError();
        });
    });
}

// ---------------------------------------------------------------------------
// Block-aligned splice by remapping the block table.
//
// With s_start, s_end and |R| multiples of the block size B and Δ != 0, the
// downstream rows keep their offsets inside their blocks, so whole blocks can
// change logical position instead of moving their bytes.  In blocks, with
// A = s_start / B, Sb span blocks, Nb = |R| / B stub blocks and Db downstream
// blocks, the row becomes
//   [old 0..A) [Nb stub blocks] [the Db downstream blocks] [the rest],
// where the stub blocks are taken first from the span's blocks, then from the
// row's spare entries past the downstream ones, and "the rest" is what is
// left of those, in order -- a permutation of the row.  The downstream rows
// stay where they are physically; only their rotary part is turned by R(Δ)
// in place (MLA: 256 of 2304 bytes per row and layer).  The stub rows are
// written into the stub blocks.  Nothing is read that another tile writes,
// so the tiles need no ordering; the commit kernel rewrites the rows after
// the data kernel has finished reading them.
// ---------------------------------------------------------------------------

// Entry j of the permuted row, from the old row.
__device__ __forceinline__ int32_t remapped_entry(const int32_t *old, int32_t j, int32_t A,
                                                  int32_t Sb, int32_t Nb, int32_t Db)
{
    auto spare = [&](int32_t k) { return k < Sb ? old[A + k] : old[A + Sb + Db + (k - Sb)]; };
    if (j < A)
        return old[j];
    if (j < A + Nb)
        return spare(j - A);
    if (j < A + Nb + Db)
        return old[A + Sb + (j - A - Nb)];
    return spare(Nb + (j - A - Nb - Db));
}

template <class G, bool IL>
__global__ void __launch_bounds__(kThreads, G::kMinBlocks) remap_data_kernel(const __grid_constant__ RemapParams p)
{
    __shared__ int64_t s_idx[G::T]; // slot of each row (in place, or the stub's target)
    __shared__ int64_t s_src[G::T]; // stub tiles: row of the tile's stub rows
    __shared__ int32_t s_ident[G::T];
    __shared__ float4 s_cs[G::kHalf];

    if (gate_closed(p.gate))
        return;
    const int tid = threadIdx.x;
    const int64_t t = blockIdx.x;
    int q = 0;
    while (q + 1 < p.num_seqs && p.seq[q + 1].tile_base <= t)
        ++q;
    const RemapSeq &S = p.seq[q];
    const int64_t k = t - S.tile_base;
    const bool down = k < S.n_down;
    const int32_t *old = p.block_tables + (int64_t)S.bt_row * p.max_blocks;
    const int32_t B = p.pool.block;
    const int64_t nb = p.pool.num_blocks;
    const int32_t A = S.s_start / B, Sb = (S.s_end - S.s_start) / B, Nb = S.n_r / B;
    const int32_t Db = (int32_t)((S.seq_len - S.s_end + B - 1) / B);
    if (tid < G::T) {
        int64_t slot = -1;
        if (down) {
            const int64_t pos = S.s_end + k * G::T + tid;
            if (pos < S.seq_len)
                slot = slot_of(old, p.max_blocks, B, nb, pos); // stays where it is
        } else {
            const int64_t j = (k - S.n_down) * G::T + tid; // stub row
            if (j < S.n_r) {
                const int32_t blk = remapped_entry(old, A + (int32_t)(j / B), A, Sb, Nb, Db);
                slot = (blk >= 0 && blk < nb) ? (int64_t)blk * B + j % B : -1;
                if (slot < 0)
                    set_status(p.status, kStatusOutOfRange);
            }
        }
        s_idx[tid] = slot;
        s_src[tid] = (!down && slot >= 0) ? tid : -1;
        s_ident[tid] = down ? 0 : 1;
    }
    // downstream tiles turn only the rotary part: pair-packed for every row
    // kind; stub tiles are written unrotated (identity rows)
    constexpr bool kPack = CsOrder<G, false, IL, true>::kPacked;
    if (down)
        for (int j = tid; j < G::kHalf; j += kThreads)
            stage_cs<G, kPack>(s_cs, j, p.table[(int64_t)q * G::kHalf + j]);
    __syncthreads();

    const int64_t copy_row_bytes = (int64_t)G::CV * 16, rot_row_bytes = (int64_t)G::kRotW * 16;
    PatchAt none{nullptr, 0, nullptr, nullptr};
    auto layer_rows = [&](int l) {
        return RowsAt{p.pool.copy + l * p.pool.copy_ls, p.pool.copy_ss,
                      p.pool.rot + l * p.pool.rot_ls, p.pool.rot_ss};
    };
    if (down) {
        // rotary part only, in place; rows of different layers are
        // independent, so LB layers of loads are in flight at once (four
        // 16-byte loads per thread: with the pair-packed rotation eight
        // layers spilled registers and measured slower)
        constexpr int LB = G::kRotPer >= 4 ? 1 : 4 / G::kRotPer;
        const int Lc = p.pool.num_layers;
        for (int l0 = 0; l0 < Lc; l0 += LB) {
            TileRegs<G> regs[LB];
#pragma unroll
            for (int b = 0; b < LB; ++b)
                if (l0 + b < Lc)
                    load_tile<G, false>(layer_rows(l0 + b), s_idx, regs[b]);
#pragma unroll
            for (int b = 0; b < LB; ++b)
                if (l0 + b < Lc)
                    store_tile<G, false, false, IL, kPack>(layer_rows(l0 + b), s_idx, regs[b],
                                                           s_cs, 0, s_ident, none);
        }
        return;
    }
    for (int l = 0; l < p.pool.num_layers; ++l) {
        const RowsAt pool_l = layer_rows(l);
        TileRegs<G> regs;
        {
            const int64_t j0 = S.stub_base;
            const RowsAt stub_l{p.stub_copy + (l * p.total_stub + j0 + (k - S.n_down) * G::T) *
                                                  copy_row_bytes,
                                copy_row_bytes,
                                p.stub_rot + (l * p.total_stub + j0 + (k - S.n_down) * G::T) *
                                                 rot_row_bytes,
                                rot_row_bytes};
            // the tile's rows are stub rows 0..T-1 counted from stub_l
            load_tile<G>(stub_l, s_src, regs);
            store_tile<G, false, true, IL>(pool_l, s_idx, regs, s_cs, 0, s_ident, none);
        }
    }
}

// One block per sequence: the whole old row into shared memory, then the
// permuted row written back over it.
__global__ void remap_commit_kernel(const __grid_constant__ RemapParams p)
{
    extern __shared__ int32_t s_old[];
    if (gate_closed(p.gate))
        return; // the block-table rows stay as they were
    const RemapSeq &S = p.seq[blockIdx.x];
    int32_t *row = p.block_tables + (int64_t)S.bt_row * p.max_blocks;
    const int32_t B = p.pool.block;
    for (int j = threadIdx.x; j < p.max_blocks; j += blockDim.x)
        s_old[j] = row[j];
    __syncthreads();
    const int32_t A = S.s_start / B, Sb = (S.s_end - S.s_start) / B, Nb = S.n_r / B;
    const int32_t Db = (int32_t)((S.seq_len - S.s_end + B - 1) / B);
    for (int j = threadIdx.x; j < p.max_blocks; j += blockDim.x)
        row[j] = remapped_entry(s_old, j, A, Sb, Nb, Db);
}

cudaError_t launch_remap(const RemapParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.num_seqs == 0)
        return cudaSuccess;
    if (p.total_tiles > 0) {
        if (p.total_tiles > 0x7FFFFFFFll)
            return cudaErrorInvalidConfiguration;
        cudaError_t e = with_inplace_geo(kind, [&](auto g) {
            return with_bool(p.pool.il != 0, [&](auto il) {
                remap_data_kernel<typename decltype(g)::type, decltype(il)::value>
                    <<<(unsigned)p.total_tiles, kThreads, 0, stream>>>(p);
                return cudaGetLastError();
            });
        });
        if (e != cudaSuccess)
            return e;
    }
    const size_t smem = (size_t)p.max_blocks * sizeof(int32_t);
    cudaError_t e = cudaFuncSetAttribute(remap_commit_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    remap_commit_kernel<<<p.num_seqs, 256, smem, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Failure-path check: the same bounded wait on a flag nothing sets.
// ---------------------------------------------------------------------------

__global__ void wait_check_kernel(const uint32_t *flag, uint32_t *status, int64_t limit_ns)
{
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        if (!wait_flag(flag, limit_ns))
            set_status(status, kStatusTimeout);
    }
}

cudaError_t launch_wait_check(uint32_t *flag, uint32_t *status, int64_t limit_ns,
                              cudaStream_t stream)
{
    wait_check_kernel<<<1, 32, 0, stream>>>(flag, status, limit_ns);
    return cudaGetLastError();
}

} // namespace kvr

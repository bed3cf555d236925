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
// owns a counter of (layer, warp) reads, each warp adding one with a release
// reduction once its loads of a layer have landed, so layer l is read when
// the counter reaches 8 (l + 1).  A warp publishes at once: reading needs
// nothing, since a tile's source rows are overwritten only by itself and by
// later tiles.  Then thread 0 makes sure (acquire, bounded) that the tiles
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

constexpr uint32_t kWarps = kThreads / 32;

template <class G>
__global__ void __launch_bounds__(kThreads, G::kMinBlocks) splice_kernel(const __grid_constant__ SpliceParams p)
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
    const int64_t k = t - S.ticket_base;
    const bool shift = k < S.n_shift;
    const int32_t *bt = p.block_tables + (int64_t)S.bt_row * p.max_blocks;
    const int32_t B = p.pool.block;
    const int64_t nb = p.pool.num_blocks;
    const int L = p.pool.num_layers;

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
    for (int j = tid; j < G::kHalf; j += kThreads)
        s_cs[G::cs_index(j)] = p.table[(int64_t)q * G::kHalf + j];
    __syncthreads();

    const int64_t copy_row_bytes = (int64_t)G::CV * 16, rot_row_bytes = (int64_t)G::kRotW * 16;
    PatchAt none{nullptr, 0, nullptr, nullptr};
    for (int l = 0; l < L; ++l) {
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
        // this warp's share of layer l is in registers: publish it now (one
        // increment per warp), before waiting on anyone, so that a tile's
        // progress never waits on the tiles behind it (its source rows are
        // overwritten only by itself and by later tiles)
        __syncwarp();
        if (shift && (tid & 31) == 0)
            red_release_add(p.flags + S.flag_base + k, 1u);
        const uint32_t want = ((uint32_t)l + 1u) * kWarps; // every warp has read layer l
        if (tid == 0 && !s_abort) {
            // the tiles this one overwrites must have read layer l
            for (int d = 0; d < 2; ++d) {
                if (s_dep[d] < 0 || s_seen[d] >= want)
                    continue;
                const uint32_t seen =
                    wait_count(p.flags + S.flag_base + s_dep[d], want, p.wait_limit_ns);
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
            store_tile<G, false>(pool_l, s_dst, regs, s_cs, 0, s_ident, none);
    }
}

cudaError_t launch_splice(const SpliceParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.total_tickets == 0)
        return cudaSuccess;
    if (p.total_tickets > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    const unsigned blocks = (unsigned)p.total_tickets;
    if (kind == RowKind::Mla)
        splice_kernel<GeoMla><<<blocks, kThreads, 0, stream>>>(p);
    else
        splice_kernel<GeoGqa><<<blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Composed splice: several directives per sequence as one in-place edit.
//
// The host turns the directives into a table of tiles (each: T rows moving by
// one constant shift, or stub rows landing at their final positions) ordered
// so that every tile a tile overwrites comes earlier: rows moving down in
// ascending order, rows moving up in descending order, stubs last (the map
// is monotone, so rows moving down and rows moving up never overlap).  The
// protocol is the splice's: tickets, per-warp release counts of the layers
// read, bounded acquire waits on the (at most two ranges of) earlier tiles a
// tile overwrites, one barrier per layer.  Every row is read once and rounded
// once, its rotary part turned by its total shift.
// ---------------------------------------------------------------------------

template <class G>
__global__ void __launch_bounds__(kThreads, G::kMinBlocks)
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
            s_cs[G::cs_index(j)] = p.table[(int64_t)tile.unit * G::kHalf + j];
    __syncthreads();

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
        // this warp's share of layer l is read: publish before waiting
        __syncwarp();
        if (!tile.stub && (tid & 31) == 0)
            red_release_add(p.flags + t, 1u);
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
            store_tile<G, false>(pool_l, s_dst, regs, s_cs, 0, s_ident, none);
    }
}

cudaError_t launch_splice_composed(const ComposedParams &p, RowKind kind, cudaStream_t stream)
{
    if (p.num_tiles == 0)
        return cudaSuccess;
    if (p.num_tiles > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    const unsigned blocks = (unsigned)p.num_tiles;
    if (kind == RowKind::Mla)
        splice_composed_kernel<GeoMla><<<blocks, kThreads, 0, stream>>>(p);
    else
        splice_composed_kernel<GeoGqa><<<blocks, kThreads, 0, stream>>>(p);
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

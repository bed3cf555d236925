// kv_api.cu -- the extern "C" entry points declared in include/kvreloc.h.
//
// Host side only: argument checks (synchronous, before anything is
// enqueued), workspace carving, per-call planning of the splice tiles, and
// the launches.  Every step of the data path runs in the kernels.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "kvreloc.h"
#include "kv_launch.h"

using namespace kvr;

namespace {

constexpr int64_t kDefaultWaitLimitNs = 2000000000ll;
// A splice launch of few tiles cuts every tile's layers into groups (units of
// their own) until it has about this many units: some 7 waves of 4 blocks on
// each of 152 SMs, so that the last, partly filled wave costs little.
constexpr int64_t kUnitsTarget = 4096;
// Splice launches of at most this many tiles (a wave or two) form their
// cos/sin rows inside the splice kernel instead of launching the δ-table
// kernel: each block spends a few fp64 sincos on its prologue, which only
// pays off while the launch is short.
constexpr int64_t kInlineTableTiles = 1024;
std::atomic<int64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int32_t> g_debug_checks{0};   // kv_set_debug_checks
std::atomic<int64_t> g_skip_publish{-1};  // kv_set_splice_skip_publish (test hook)
thread_local int32_t t_launches = 0;
thread_local cudaEvent_t t_ev_start = nullptr, t_ev_stop = nullptr;

cudaError_t mark(cudaEvent_t ev, cudaStream_t stream)
{
    return (t_ev_start && t_ev_stop) ? cudaEventRecord(ev, stream) : cudaSuccess;
}

constexpr size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Natural alignment of a device array of n-byte elements (NULL passes: the
// callers check presence separately).
bool aligned_to(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

// Shape and layout checks shared by every call.
bool pool_ok(const kv_pool_desc *p)
{
    if (!p)
        return false;
    if (p->num_layers <= 0 || p->block_size <= 0 || p->num_slots <= 0 ||
        p->num_slots % p->block_size != 0)
        return false;
    if (p->copy_dim <= 0 || p->copy_dim % 8 != 0 || p->rot_heads <= 0 || p->rot_head_dim <= 0 ||
        p->rot_head_dim % 16 != 0)
        return false;
    if (!(p->rope_base > 0.0) || (p->pair_convention != 0 && p->pair_convention != 1))
        return false;
    if (!p->copy_base || !p->rot_base || !aligned16(p->copy_base) || !aligned16(p->rot_base))
        return false;
    const int64_t strides[4] = {p->copy_layer_stride, p->copy_slot_stride, p->rot_layer_stride,
                                p->rot_slot_stride};
    for (int64_t s : strides)
        if (s < 0 || s % 8 != 0)
            return false;
    return true;
}

bool row_kind(const kv_pool_desc *p, RowKind *kind)
{
    if (p->copy_dim == 512 && p->rot_heads == 1 && p->rot_head_dim == 64) {
        *kind = RowKind::Mla;
        return true;
    }
    if (p->copy_dim == 1024 && p->rot_heads == 8 && p->rot_head_dim == 128) {
        *kind = RowKind::Gqa;
        return true;
    }
    if (p->copy_dim == 512 && p->rot_heads == 4 && p->rot_head_dim == 128) {
        *kind = RowKind::Gqa4;
        return true;
    }
    if (p->copy_dim == 4096 && p->rot_heads == 32 && p->rot_head_dim == 128) {
        *kind = RowKind::Mha;
        return true;
    }
    return false;
}

PoolView view_of(const kv_pool_desc *p)
{
    PoolView v;
    v.copy = static_cast<char *>(p->copy_base);
    v.copy_ls = p->copy_layer_stride * 2;
    v.copy_ss = p->copy_slot_stride * 2;
    v.rot = static_cast<char *>(p->rot_base);
    v.rot_ls = p->rot_layer_stride * 2;
    v.rot_ss = p->rot_slot_stride * 2;
    v.num_slots = p->num_slots;
    v.num_blocks = p->num_slots / p->block_size;
    v.block = p->block_size;
    v.num_layers = p->num_layers;
    v.il = p->pair_convention;
    return v;
}

size_t table_bytes(const kv_pool_desc *p, int64_t units)
{
    return align256((size_t)units * (size_t)(p->rot_head_dim / 2) * sizeof(float4));
}

// Debug checks: a bitmap of `bits` bits, and the per-sequence entry counts of
// a splice.
size_t bitmap_bytes(int64_t bits) { return align256((size_t)((bits + 31) / 32) * 4u); }

size_t debug_bytes(const kv_pool_desc *p, int64_t seqs)
{
    return bitmap_bytes(p->num_slots) + align256((size_t)std::max<int64_t>(seqs, 0) * 4u);
}

// Source and destination share their slots (a relocation inside one pool).
bool same_pool(const kv_pool_desc *a, const kv_pool_desc *b)
{
    return a->copy_base == b->copy_base || a->rot_base == b->rot_base;
}

// Debug check of a splice's block-table entries: `used[q]` entries of row q
// must name distinct blocks.  Copies the counts into the workspace at `at`
// (pageable host memory: the call returns once the driver holds its copy)
// and launches the scan; returns the gate for the row-moving kernels.
cudaError_t launch_dup_check(const kv_pool_desc *pool, const int32_t *d_block_tables,
                             int32_t max_blocks, const std::vector<int32_t> &used, char *at,
                             uint32_t *status, cudaStream_t stream)
{
    const int64_t nb = pool->num_slots / pool->block_size;
    uint32_t *bm = reinterpret_cast<uint32_t *>(at);
    int32_t *d_used = reinterpret_cast<int32_t *>(at + bitmap_bytes(pool->num_slots));
    cudaError_t e = cudaMemsetAsync(bm, 0, bitmap_bytes(nb), stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_used, used.data(), used.size() * sizeof(int32_t),
                            cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return e;
    DupBlockParams dp{};
    dp.block_tables = d_block_tables;
    dp.used = d_used;
    dp.rows = (int32_t)used.size();
    dp.max_blocks = max_blocks;
    dp.num_blocks = nb;
    dp.bitmap = bm;
    dp.status = status;
    return launch_dup_block_check(dp, stream);
}

// Factor checks; fills `pv` and tells whether any channel is patched.
kv_status patch_view(const kv_patch_desc *d, PatchView *pv, bool *any)
{
    std::memset(pv, 0, sizeof *pv);
    *any = false;
    if (!d)
        return KV_OK;
    if (d->rank < 4 || d->rank > kMaxRank || d->rank % 4 != 0)
        return KV_ERR_INVALID_ARG;
    pv->m = d->rank;
    if (!aligned_to(d->d_u_chunk_tok, 8) || !aligned_to(d->d_v_chunk, 4))
        return KV_ERR_INVALID_ARG;
    pv->u_chunk_tok = d->d_u_chunk_tok;
    pv->v_chunk = d->d_v_chunk;
    for (int ch = 0; ch < 2; ++ch) {
        if (!d->u[ch] || !d->v[ch])
            continue;
        if (!aligned16(d->u[ch]) || !aligned16(d->v[ch]))
            return KV_ERR_INVALID_ARG;
        const int64_t s[5] = {d->u_layer_stride[ch], d->u_tok_stride[ch], d->v_layer_stride[ch],
                              d->v_chunk_stride[ch], d->v_col_stride[ch]};
        for (int64_t x : s)
            if (x < 0 || x % 4 != 0)
                return KV_ERR_INVALID_ARG;
        pv->u[ch] = d->u[ch];
        pv->v[ch] = d->v[ch];
        pv->u_ls[ch] = d->u_layer_stride[ch];
        pv->u_ts[ch] = d->u_tok_stride[ch];
        pv->v_ls[ch] = d->v_layer_stride[ch];
        pv->v_cs[ch] = d->v_chunk_stride[ch];
        pv->v_cols[ch] = d->v_col_stride[ch];
        if (d->u_rows[ch] < 0 || d->v_slots[ch] < 0)
            return KV_ERR_INVALID_ARG;
        pv->u_rows[ch] = d->u_rows[ch];
        pv->v_slots[ch] = d->v_slots[ch];
        *any = true;
    }
    return KV_OK;
}

kv_status ws_ok(const void *ws, size_t have, size_t need)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || have < need)
        return KV_ERR_WORKSPACE;
    return KV_OK;
}

#define KV_CUDA(call)                                                                              \
    do {                                                                                           \
        if ((call) != cudaSuccess)                                                                 \
            return KV_ERR_CUDA;                                                                    \
    } while (0)

// Shared body of kv_relocate (in_place = false) and kv_patch (in_place = true).
kv_status relocate_impl(const kv_pool_desc *src, const kv_pool_desc *dst, int32_t num_chunks,
                        int64_t total_tokens, const int32_t *tok_off, const int32_t *src_slots,
                        const int32_t *chunk_req, const int32_t *chunk_dst_pos,
                        const int32_t *delta, const int32_t *block_tables, int32_t num_reqs,
                        int32_t max_blocks, const kv_patch_desc *patch, void *ws,
                        size_t ws_bytes, cudaStream_t stream, bool in_place)
{
    t_launches = 0;
    if (!pool_ok(src) || !pool_ok(dst))
        return KV_ERR_INVALID_ARG;
    if (src->num_layers != dst->num_layers || src->copy_dim != dst->copy_dim ||
        src->rot_heads != dst->rot_heads || src->rot_head_dim != dst->rot_head_dim ||
        src->rope_base != dst->rope_base || src->pair_convention != dst->pair_convention)
        return KV_ERR_INVALID_ARG;
    RowKind kind;
    if (!row_kind(src, &kind))
        return KV_ERR_UNSUPPORTED;
    if (num_chunks < 0 || total_tokens < 0 || total_tokens > 0x7FFFFFFFll)
        return KV_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (num_chunks == 0 || !tok_off || !chunk_req || !chunk_dst_pos || !block_tables)
            return KV_ERR_INVALID_ARG;
        if (!in_place && (!src_slots || !delta))
            return KV_ERR_INVALID_ARG;
        if (num_reqs <= 0 || max_blocks <= 0)
            return KV_ERR_INVALID_ARG;
        const void *i32s[6] = {tok_off, src_slots, chunk_req, chunk_dst_pos, delta, block_tables};
        for (const void *a : i32s)
            if (!aligned_to(a, 4))
                return KV_ERR_INVALID_ARG;
    }
    PatchView pv;
    bool patched = false;
    kv_status st = patch_view(patch, &pv, &patched);
    if (st != KV_OK)
        return st;
    if (in_place && !patched)
        return KV_ERR_INVALID_ARG;
    const size_t need = kHeaderBytes + (in_place ? 0 : table_bytes(src, num_chunks));
    // debug check: a relocation inside one pool must not write a slot it reads
    const bool check = !in_place && g_debug_checks.load() != 0 && same_pool(src, dst);
    const size_t check_bytes = check ? bitmap_bytes(dst->num_slots) : 0;
    if ((st = ws_ok(ws, ws_bytes, need + check_bytes)) != KV_OK)
        return st;

    char *w = static_cast<char *>(ws);
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes, stream));
    if (total_tokens == 0)
        return KV_OK;
    const uint32_t *gate = nullptr;
    if (check) {
        uint32_t *bm = reinterpret_cast<uint32_t *>(w + need);
        KV_CUDA(cudaMemsetAsync(bm, 0, check_bytes, stream));
        OverlapParams op{};
        op.tok_off = tok_off;
        op.src_slots = src_slots;
        op.chunk_req = chunk_req;
        op.chunk_dst_pos = chunk_dst_pos;
        op.block_tables = block_tables;
        op.num_chunks = num_chunks;
        op.num_reqs = num_reqs;
        op.max_blocks = max_blocks;
        op.block = dst->block_size;
        op.total_tokens = total_tokens;
        op.num_slots = dst->num_slots;
        op.num_blocks = dst->num_slots / dst->block_size;
        op.bitmap = bm;
        op.status = reinterpret_cast<uint32_t *>(w);
        KV_CUDA(launch_overlap_check(op, stream));
        t_launches += 2;
        gate = reinterpret_cast<uint32_t *>(w);
    }
    float4 *table = reinterpret_cast<float4 *>(w + kHeaderBytes);
    if (!in_place) {
        TableParams tp{};
        tp.d_delta = delta;
        tp.units = num_chunks;
        tp.half = src->rot_head_dim / 2;
        tp.head_dim = src->rot_head_dim;
        tp.base = src->rope_base;
        tp.table = table;
        KV_CUDA(launch_delta_table(tp, stream));
        ++t_launches;
    }
    RelocParams rp{};
    rp.src = view_of(src);
    rp.dst = view_of(dst);
    rp.num_chunks = num_chunks;
    rp.total_tokens = total_tokens;
    rp.tok_off = tok_off;
    rp.src_slots = src_slots;
    rp.chunk_req = chunk_req;
    rp.chunk_dst_pos = chunk_dst_pos;
    rp.delta = delta;
    rp.block_tables = block_tables;
    rp.num_reqs = num_reqs;
    rp.max_blocks = max_blocks;
    rp.table = table;
    rp.patch = pv;
    rp.patched = patched ? 1 : 0;
    rp.in_place = in_place ? 1 : 0;
    rp.status = reinterpret_cast<uint32_t *>(w);
    rp.gate = gate;
    KV_CUDA(mark(t_ev_start, stream));
    if (patch_tc_supported(rp, kind)) {
        KV_CUDA(launch_patch_tc(rp, kind, stream));
        t_launches += patch_tc_launches(rp, kind);
    } else {
        KV_CUDA(launch_relocate(rp, kind, stream));
        ++t_launches;
    }
    KV_CUDA(mark(t_ev_stop, stream));
    return KV_OK;
}


// ---------------------------------------------------------------------------
// Composed splice planning (host)
// ---------------------------------------------------------------------------

// A run of len logical rows whose content comes from src.. (original
// positions, or global stub rows when `stub`) and was last rounded at
// positions written..; within a run both advance with the position.
struct Seg {
    int64_t src, written, len;
    bool stub;
};

struct ComposedPlan {
    std::vector<SpliceTile> tiles;
    std::vector<int32_t> deltas;   // δ-table unit -> shift
    std::vector<int64_t> final_len; // per sequence
    int64_t total_stub = 0;
};

// Pieces of the logical range [from, to) of `segs`, in order.
void cut_range(const std::vector<Seg> &segs, int64_t from, int64_t to, std::vector<Seg> &out)
{
    int64_t pos = 0;
    for (const Seg &g : segs) {
        const int64_t lo = std::max(pos, from), hi = std::min(pos + g.len, to);
        if (lo < hi)
            out.push_back(Seg{g.src + (lo - pos), g.written + (lo - pos), hi - lo, g.stub});
        pos += g.len;
    }
}

// Inclusive run [first, last] of the tiles in tiles[b, e) -- sorted by
// source position, ascending or descending, and non-overlapping -- whose
// source rows meet [d, d + n), with `self` trimmed off the run's ends (a
// tile may overwrite its own rows; no other position of self is possible).
// Returns false when no other tile qualifies.
bool overlapping_run(const std::vector<SpliceTile> &tiles, size_t b, size_t e, bool ascending,
                     int64_t d, int64_t n, int64_t self, int32_t &first, int32_t &last)
{
    first = last = -1;
    if (b >= e)
        return false;
    auto below = [&](const SpliceTile &u) { return u.src_lo + u.n <= d; }; // entirely before
    auto above = [&](const SpliceTile &u) { return u.src_lo >= d + n; };  // entirely after
    size_t lo, hi; // [lo, hi) meets the range
    if (ascending) {
        lo = (size_t)(std::partition_point(tiles.begin() + b, tiles.begin() + e, below) -
                      tiles.begin());
        hi = (size_t)(std::partition_point(tiles.begin() + lo, tiles.begin() + e,
                                           [&](const SpliceTile &u) { return !above(u); }) -
                      tiles.begin());
    } else {
        lo = (size_t)(std::partition_point(tiles.begin() + b, tiles.begin() + e, above) -
                      tiles.begin());
        hi = (size_t)(std::partition_point(tiles.begin() + lo, tiles.begin() + e,
                                           [&](const SpliceTile &u) { return !below(u); }) -
                      tiles.begin());
    }
    if (lo < hi && (int64_t)lo == self)
        ++lo;
    if (lo < hi && (int64_t)(hi - 1) == self)
        --hi;
    if (lo >= hi)
        return false;
    first = (int32_t)lo;
    last = (int32_t)(hi - 1);
    return true;
}

kv_status plan_composed(RowKind kind, int32_t num_seqs, int32_t num_dirs, int64_t capacity,
                        const int32_t *lens, const int32_t *s0, const int32_t *s1,
                        const int32_t *nr, ComposedPlan &plan)
{
    const int64_t T = inplace_tile_rows(kind);
    // validate every directive in the indexing the previous ones leave
    plan.total_stub = 0;
    for (int32_t q = 0; q < num_seqs; ++q) {
        int64_t len = lens[q];
        if (len < 0)
            return KV_ERR_INVALID_ARG;
        for (int32_t i = 0; i < num_dirs; ++i) {
            const int64_t k = (int64_t)i * num_seqs + q;
            if (s0[k] < 0 || s0[k] > s1[k] || s1[k] > len || nr[k] < 0)
                return KV_ERR_INVALID_ARG;
            len += (int64_t)nr[k] - (s1[k] - s0[k]);
            plan.total_stub += nr[k];
        }
        if (len > 0x7FFFFFFFll)
            return KV_ERR_CAPACITY;
        if (capacity >= 0 && std::max<int64_t>(len, lens[q]) > capacity)
            return KV_ERR_CAPACITY;
    }
    std::map<int64_t, int32_t> unit_of;
    auto unit = [&](int64_t shift) -> int32_t {
        if (shift == 0)
            return -1;
        auto it = unit_of.find(shift);
        if (it != unit_of.end())
            return it->second;
        const int32_t u = (int32_t)plan.deltas.size();
        plan.deltas.push_back((int32_t)shift);
        unit_of.emplace(shift, u);
        return u;
    };
    int64_t stub_row = 0;
    std::vector<int64_t> stub_first((size_t)num_dirs * num_seqs);
    for (int32_t i = 0; i < num_dirs; ++i)
        for (int32_t q = 0; q < num_seqs; ++q) {
            stub_first[(size_t)i * num_seqs + q] = stub_row;
            stub_row += nr[(int64_t)i * num_seqs + q];
        }
    plan.final_len.assign(num_seqs, 0);
    for (int32_t q = 0; q < num_seqs; ++q) {
        std::vector<Seg> segs;
        int64_t len = lens[q];
        if (len > 0)
            segs.push_back(Seg{0, 0, len, false});
        for (int32_t i = 0; i < num_dirs; ++i) {
            const int64_t k = (int64_t)i * num_seqs + q;
            std::vector<Seg> next;
            cut_range(segs, 0, s0[k], next);
            if (nr[k] > 0)
                next.push_back(Seg{stub_first[(size_t)k], s0[k], nr[k], true});
            cut_range(segs, s1[k], len, next);
            segs.swap(next);
            len += (int64_t)nr[k] - (s1[k] - s0[k]);
        }
        plan.final_len[q] = len;
        // final positions and shifts; tiles: rows moving down (ascending),
        // rows moving up (descending), stub rows
        std::vector<int64_t> at(segs.size());
        int64_t pos = 0;
        for (size_t g = 0; g < segs.size(); ++g) {
            at[g] = pos;
            pos += segs[g].len;
        }
        const size_t base = plan.tiles.size();
        for (size_t g = 0; g < segs.size(); ++g) {
            const int64_t shift = at[g] - segs[g].written;
            if (segs[g].stub || shift >= 0)
                continue;
            for (int64_t o = 0; o < segs[g].len; o += T)
                plan.tiles.push_back(SpliceTile{segs[g].src + o, at[g] + o,
                                                (int32_t)std::min(T, segs[g].len - o), q,
                                                unit(shift), 0, {-1, -1, -1, -1}});
        }
        const size_t down_end = plan.tiles.size();
        for (size_t g = segs.size(); g-- > 0;) {
            const int64_t shift = at[g] - segs[g].written;
            if (segs[g].stub || shift <= 0)
                continue;
            for (int64_t hi = segs[g].len; hi > 0; hi -= T) {
                const int64_t lo = std::max<int64_t>(0, hi - T);
                plan.tiles.push_back(SpliceTile{segs[g].src + lo, at[g] + lo, (int32_t)(hi - lo),
                                                q, unit(shift), 0, {-1, -1, -1, -1}});
            }
        }
        const size_t up_end = plan.tiles.size();
        for (size_t g = 0; g < segs.size(); ++g) {
            if (!segs[g].stub)
                continue;
            const int64_t shift = at[g] - segs[g].written;
            for (int64_t o = 0; o < segs[g].len; o += T)
                plan.tiles.push_back(SpliceTile{segs[g].src + o, at[g] + o,
                                                (int32_t)std::min(T, segs[g].len - o), q,
                                                unit(shift), 1, {-1, -1, -1, -1}});
        }
        // dependencies: the earlier tiles whose source rows each destination meets
        for (size_t j = base; j < plan.tiles.size(); ++j) {
            SpliceTile &tl = plan.tiles[j];
            int32_t f, l;
            int r = 0;
            if (overlapping_run(plan.tiles, base, down_end, true, tl.dst_lo, tl.n, (int64_t)j, f, l)) {
                tl.dep[2 * r] = f;
                tl.dep[2 * r + 1] = l;
                ++r;
            }
            if (overlapping_run(plan.tiles, down_end, up_end, false, tl.dst_lo, tl.n, (int64_t)j, f,
                                l)) {
                tl.dep[2 * r] = f;
                tl.dep[2 * r + 1] = l;
                ++r;
            }
            // every wait must point backwards, or the protocol could deadlock
            for (int d = 0; d < 2 * r; ++d)
                if (tl.dep[d] >= (int32_t)j)
                    return KV_ERR_UNSUPPORTED;
        }
    }
    if (plan.tiles.size() > 0x7FFFFFFFull)
        return KV_ERR_CAPACITY;
    return KV_OK;
}

// Workspace of a composed splice: header, δ-table, tiles, unit shifts, counters.
size_t composed_bytes(const kv_pool_desc *pool, const ComposedPlan &plan)
{
    return kHeaderBytes + table_bytes(pool, (int64_t)plan.deltas.size()) +
           align256(plan.tiles.size() * sizeof(SpliceTile)) +
           align256(plan.deltas.size() * sizeof(int32_t)) + align256(plan.tiles.size() * 4u);
}

} // namespace

extern "C" {

size_t kv_workspace_size(const kv_pool_desc *pool, int64_t max_rows, int32_t max_units)
{
    RowKind kind;
    if (!pool_ok(pool) || !row_kind(pool, &kind) || max_rows < 0 || max_units < 0)
        return 0;
    // the splices' tiles are the smaller ones (one flag each)
    const int64_t T = std::min(tile_rows(kind), inplace_tile_rows(kind));
    const int64_t units = std::max<int64_t>(max_units, 1);
    const int64_t flags = (int64_t)pool->num_layers * ((max_rows + T - 1) / T + units);
    // the last part serves the debug checks (kv_set_debug_checks)
    return (size_t)kHeaderBytes + table_bytes(pool, units) + align256((size_t)flags * 4u) +
           debug_bytes(pool, units);
}

kv_status kv_relocate(const kv_pool_desc *src, const kv_pool_desc *dst, int32_t num_chunks,
                      int64_t total_tokens, const int32_t *d_tok_off, const int32_t *d_src_slots,
                      const int32_t *d_chunk_req, const int32_t *d_chunk_dst_pos,
                      const int32_t *d_delta, const int32_t *d_block_tables, int32_t num_reqs,
                      int32_t max_blocks, const kv_patch_desc *patch, void *d_workspace,
                      size_t workspace_bytes, kv_stream_t stream)
{
    return relocate_impl(src, dst, num_chunks, total_tokens, d_tok_off, d_src_slots, d_chunk_req,
                         d_chunk_dst_pos, d_delta, d_block_tables, num_reqs, max_blocks, patch,
                         d_workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                         false);
}

kv_status kv_patch(const kv_pool_desc *pool, int32_t num_chunks, int64_t total_tokens,
                   const int32_t *d_tok_off, const int32_t *d_chunk_req,
                   const int32_t *d_chunk_dst_pos, const int32_t *d_block_tables,
                   int32_t num_reqs, int32_t max_blocks, const kv_patch_desc *patch,
                   void *d_workspace, size_t workspace_bytes, kv_stream_t stream)
{
    return relocate_impl(pool, pool, num_chunks, total_tokens, d_tok_off, nullptr, d_chunk_req,
                         d_chunk_dst_pos, nullptr, d_block_tables, num_reqs, max_blocks, patch,
                         d_workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                         true);
}

kv_status kv_splice(const kv_pool_desc *pool, int32_t num_seqs, int32_t *d_block_tables,
                    int32_t max_blocks, int32_t *h_seq_lens, const int32_t *h_s_start,
                    const int32_t *h_s_end, const int32_t *h_stub_len, const void *d_stub_copy,
                    const void *d_stub_rot, kv_mode mode, void *d_workspace,
                    size_t workspace_bytes, kv_stream_t stream_)
{
    t_launches = 0;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!pool_ok(pool) || num_seqs < 0 ||
        (mode != KV_AMORTIZE && mode != KV_FORGET && mode != KV_AMORTIZE_REMAP))
        return KV_ERR_INVALID_ARG;
    RowKind kind;
    if (!row_kind(pool, &kind))
        return KV_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return KV_OK;
    if (!h_seq_lens || !h_s_start || !h_s_end || !h_stub_len)
        return KV_ERR_INVALID_ARG;
    int64_t total_stub = 0;
    for (int q = 0; q < num_seqs; ++q) {
        if (h_seq_lens[q] < 0 || h_s_start[q] < 0 || h_s_start[q] > h_s_end[q] ||
            h_s_end[q] > h_seq_lens[q] || h_stub_len[q] < 0)
            return KV_ERR_INVALID_ARG;
        total_stub += h_stub_len[q];
    }
    if (mode == KV_FORGET) {
        for (int q = 0; q < num_seqs; ++q)
            h_seq_lens[q] = h_s_start[q];
        return KV_OK;
    }
    if (!d_block_tables || !aligned_to(d_block_tables, 4) || max_blocks <= 0)
        return KV_ERR_INVALID_ARG;
    if (total_stub > 0 && (!d_stub_copy || !d_stub_rot || !aligned16(d_stub_copy) ||
                           !aligned16(d_stub_rot)))
        return KV_ERR_INVALID_ARG;
    const int64_t B = pool->block_size;
    for (int q = 0; q < num_seqs; ++q) {
        const int64_t delta = (int64_t)h_stub_len[q] - (h_s_end[q] - h_s_start[q]);
        const int64_t new_len = h_seq_lens[q] + delta;
        if (new_len > 0x7FFFFFFFll)
            return KV_ERR_CAPACITY;
        const int64_t span = std::max<int64_t>(h_seq_lens[q], new_len);
        if ((span + B - 1) / B > max_blocks)
            return KV_ERR_CAPACITY;
    }

    // KV_AMORTIZE_REMAP: block-aligned directives that shift move by
    // permuting the block-table row; the others take the data-moving path
    std::vector<char> remap((size_t)num_seqs, 0);
    if (mode == KV_AMORTIZE_REMAP && max_blocks <= kMaxRemapBlocks)
        for (int q = 0; q < num_seqs; ++q)
            remap[q] = h_s_start[q] % B == 0 && h_s_end[q] % B == 0 && h_stub_len[q] % B == 0 &&
                       h_stub_len[q] != h_s_end[q] - h_s_start[q];

    // plan: launches of up to kMaxSeqsPerLaunch sequences each; a launch of
    // few tiles cuts every tile's layers into groups, each its own ticketed
    // unit, so that short edits still fill the GPU (max_groups 1: whole tiles)
    const int T = inplace_tile_rows(kind);
    std::vector<SpliceParams> plans;
    int64_t stub_base = 0, max_flags = 0;
    auto make_plans = [&](int32_t max_groups) {
        plans.clear();
        stub_base = 0;
        max_flags = 0;
        for (int q0 = 0; q0 < num_seqs; q0 += kMaxSeqsPerLaunch) {
            SpliceParams sp{};
            sp.num_seqs = std::min(kMaxSeqsPerLaunch, num_seqs - q0);
            int64_t tickets = 0, flags = 0;
            for (int i = 0; i < sp.num_seqs; ++i) {
                const int q = q0 + i;
                SpliceSeq &S = sp.seq[i];
                S.s_start = h_s_start[q];
                S.s_end = h_s_end[q];
                S.seq_len = h_seq_lens[q];
                S.n_r = h_stub_len[q];
                S.delta = S.n_r - (S.s_end - S.s_start);
                const int64_t down = S.seq_len - S.s_end;
                S.n_shift = (S.delta == 0 || remap[q]) ? 0 : (int32_t)((down + T - 1) / T);
                S.n_stub = remap[q] ? 0 : (S.n_r + T - 1) / T;
                S.bt_row = q;
                S.stub_base = stub_base;
                stub_base += S.n_r;
                tickets += S.n_shift + S.n_stub;
            }
            // layer groups: enough units for about kUnitsTarget blocks
            const int32_t L = pool->num_layers;
            int32_t groups = (int32_t)std::min<int64_t>(
                std::min<int64_t>(L, max_groups),
                std::max<int64_t>(1, (kUnitsTarget + std::max<int64_t>(tickets, 1) - 1) /
                                         std::max<int64_t>(tickets, 1)));
            const int32_t per = (L + groups - 1) / groups;
            groups = (L + per - 1) / per;
            sp.layer_groups = groups;
            sp.group_layers = per;
            tickets = 0;
            for (int i = 0; i < sp.num_seqs; ++i) {
                SpliceSeq &S = sp.seq[i];
                S.ticket_base = tickets;
                S.flag_base = flags;
                tickets += (int64_t)(S.n_shift + S.n_stub) * groups;
                flags += (int64_t)S.n_shift * groups;
            }
            sp.total_tickets = tickets;
            max_flags = std::max(max_flags, flags);
            plans.push_back(sp);
        }
    };
    make_plans(pool->num_layers);
    const bool check = g_debug_checks.load() != 0;
    {
        // a workspace too small for these groups' counters: whole tiles
        const size_t tb = table_bytes(pool, std::min(num_seqs, kMaxSeqsPerLaunch));
        if (workspace_bytes < kHeaderBytes + tb + align256((size_t)max_flags * 4u) +
                                  (check ? debug_bytes(pool, num_seqs) : 0))
            make_plans(1);
    }
    const size_t tbytes = table_bytes(pool, std::min(num_seqs, kMaxSeqsPerLaunch));
    const size_t need = kHeaderBytes + tbytes + align256((size_t)max_flags * 4u);
    kv_status st =
        ws_ok(d_workspace, workspace_bytes, need + (check ? debug_bytes(pool, num_seqs) : 0));
    if (st != KV_OK)
        return st;

    // workspace: header, the tiles' read counters, the δ-table (then the
    // debug-check part); the header and the first launch's counters are
    // cleared by one memset
    char *w = static_cast<char *>(d_workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(w);
    uint32_t *ticket = status + 1;
    uint32_t *flags = reinterpret_cast<uint32_t *>(w + kHeaderBytes);
    float4 *table = reinterpret_cast<float4 *>(w + kHeaderBytes + align256((size_t)max_flags * 4u));
    size_t first_flags = 0;
    for (const SpliceParams &sp : plans)
        if (sp.total_tickets > 0) {
            for (int i = 0; i < sp.num_seqs; ++i)
                first_flags += (size_t)sp.seq[i].n_shift * (size_t)sp.layer_groups;
            break;
        }
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes + first_flags * 4u, stream));
    const uint32_t *gate = nullptr;
    if (check) {
        // the entries each sequence uses, before and after its directive
        std::vector<int32_t> used((size_t)num_seqs);
        for (int q = 0; q < num_seqs; ++q) {
            const int64_t new_len =
                (int64_t)h_seq_lens[q] + h_stub_len[q] - (h_s_end[q] - h_s_start[q]);
            used[q] = (int32_t)((std::max<int64_t>(h_seq_lens[q], new_len) + B - 1) / B);
        }
        KV_CUDA(launch_dup_check(pool, d_block_tables, max_blocks, used, w + need, status,
                                 stream));
        ++t_launches;
        gate = status;
    }
    const int64_t limit = g_wait_limit_ns.load();
    const int64_t skip = g_skip_publish.load();
    bool marked = false, first = true;
    for (SpliceParams &sp : plans) {
        if (sp.total_tickets == 0)
            continue;
        int64_t nflags = 0;
        for (int i = 0; i < sp.num_seqs; ++i)
            nflags += (int64_t)sp.seq[i].n_shift * sp.layer_groups;
        if (!first) {
            KV_CUDA(cudaMemsetAsync(ticket, 0, sizeof(uint32_t), stream));
            if (nflags > 0)
                KV_CUDA(cudaMemsetAsync(flags, 0, (size_t)nflags * 4u, stream));
        }
        first = false;
        // a launch of at most kInlineTableTiles tiles forms its cos/sin rows
        // in the blocks themselves (no δ-table kernel); larger ones share the
        // table, built once
        sp.inline_table = sp.total_tickets <= kInlineTableTiles ? 1 : 0;
        sp.rope_base = pool->rope_base;
        if (!sp.inline_table) {
            TableParams tp{};
            tp.d_delta = nullptr;
            for (int i = 0; i < sp.num_seqs; ++i)
                tp.h_delta[i] = sp.seq[i].delta;
            tp.units = sp.num_seqs;
            tp.half = pool->rot_head_dim / 2;
            tp.head_dim = pool->rot_head_dim;
            tp.base = pool->rope_base;
            tp.table = table;
            KV_CUDA(launch_delta_table(tp, stream));
            ++t_launches;
        }
        sp.pool = view_of(pool);
        sp.block_tables = d_block_tables;
        sp.max_blocks = max_blocks;
        sp.stub_copy = static_cast<const char *>(d_stub_copy);
        sp.stub_rot = static_cast<const char *>(d_stub_rot);
        sp.total_stub = total_stub;
        sp.table = table;
        sp.status = status;
        sp.ticket = ticket;
        sp.flags = flags;
        sp.wait_limit_ns = limit;
        sp.skip_publish = skip;
        sp.gate = gate;
        if (!marked) {
            KV_CUDA(mark(t_ev_start, stream));
            marked = true;
        }
        KV_CUDA(launch_splice(sp, kind, stream));
        ++t_launches;
    }
    // remapped sequences: rotary parts in place, stubs into their blocks,
    // then the permuted block-table rows
    int64_t remap_stub = 0;
    std::vector<RemapParams> rplans;
    {
        RemapParams rp{};
        int64_t stub_base = 0;
        for (int q = 0; q < num_seqs; ++q) {
            if (remap[q]) {
                if (rp.num_seqs == kMaxSeqsPerLaunch) {
                    rplans.push_back(rp);
                    rp = RemapParams{};
                }
                RemapSeq &R = rp.seq[rp.num_seqs++];
                R.s_start = h_s_start[q];
                R.s_end = h_s_end[q];
                R.seq_len = h_seq_lens[q];
                R.n_r = h_stub_len[q];
                R.delta = R.n_r - (R.s_end - R.s_start);
                R.bt_row = q;
                R.n_down = (int32_t)((R.seq_len - R.s_end + T - 1) / T);
                R.n_stub = (R.n_r + T - 1) / T;
                R.tile_base = rp.total_tiles;
                R.stub_base = stub_base;
                rp.total_tiles += R.n_down + R.n_stub;
                ++remap_stub;
            }
            stub_base += h_stub_len[q];
        }
        if (rp.num_seqs > 0)
            rplans.push_back(rp);
    }
    for (RemapParams &rp : rplans) {
        TableParams tp{};
        tp.d_delta = nullptr;
        for (int i = 0; i < rp.num_seqs; ++i)
            tp.h_delta[i] = rp.seq[i].delta;
        tp.units = rp.num_seqs;
        tp.half = pool->rot_head_dim / 2;
        tp.head_dim = pool->rot_head_dim;
        tp.base = pool->rope_base;
        tp.table = table;
        KV_CUDA(launch_delta_table(tp, stream));
        ++t_launches;
        rp.pool = view_of(pool);
        rp.block_tables = d_block_tables;
        rp.max_blocks = max_blocks;
        rp.stub_copy = static_cast<const char *>(d_stub_copy);
        rp.stub_rot = static_cast<const char *>(d_stub_rot);
        rp.total_stub = total_stub;
        rp.table = table;
        rp.status = status;
        rp.gate = gate;
        if (!marked) {
            KV_CUDA(mark(t_ev_start, stream));
            marked = true;
        }
        KV_CUDA(launch_remap(rp, kind, stream));
        t_launches += rp.total_tiles > 0 ? 2 : 1;
    }
    (void)remap_stub;
    if (marked)
        KV_CUDA(mark(t_ev_stop, stream));
    for (int q = 0; q < num_seqs; ++q)
        h_seq_lens[q] += h_stub_len[q] - (h_s_end[q] - h_s_start[q]);
    return KV_OK;
}

size_t kv_splice_composed_workspace_size(const kv_pool_desc *pool, int32_t num_seqs,
                                         int32_t num_dirs, const int32_t *h_seq_lens,
                                         const int32_t *h_s_start, const int32_t *h_s_end,
                                         const int32_t *h_stub_len)
{
    RowKind kind;
    if (!pool_ok(pool) || !row_kind(pool, &kind) || num_seqs < 0 || num_dirs < 0)
        return 0;
    if (num_seqs > 0 && (!h_seq_lens || (num_dirs > 0 && (!h_s_start || !h_s_end || !h_stub_len))))
        return 0;
    ComposedPlan plan;
    if (plan_composed(kind, num_seqs, num_dirs, -1, h_seq_lens, h_s_start, h_s_end, h_stub_len,
                      plan) != KV_OK)
        return 0;
    // the last part serves the debug checks (kv_set_debug_checks)
    return composed_bytes(pool, plan) + debug_bytes(pool, num_seqs);
}

kv_status kv_splice_composed(const kv_pool_desc *pool, int32_t num_seqs, int32_t num_dirs,
                             const int32_t *d_block_tables, int32_t max_blocks,
                             int32_t *h_seq_lens, const int32_t *h_s_start, const int32_t *h_s_end,
                             const int32_t *h_stub_len, const void *d_stub_copy,
                             const void *d_stub_rot, void *d_workspace, size_t workspace_bytes,
                             kv_stream_t stream_)
{
    t_launches = 0;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!pool_ok(pool))
        return KV_ERR_INVALID_ARG;
    RowKind kind;
    if (!row_kind(pool, &kind))
        return KV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_dirs < 0)
        return KV_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_dirs == 0)
        return KV_OK;
    if (!h_seq_lens || !h_s_start || !h_s_end || !h_stub_len || !d_block_tables ||
        !aligned_to(d_block_tables, 4) || max_blocks <= 0)
        return KV_ERR_INVALID_ARG;
    ComposedPlan plan;
    kv_status st = plan_composed(kind, num_seqs, num_dirs, (int64_t)max_blocks * pool->block_size,
                                 h_seq_lens, h_s_start, h_s_end, h_stub_len, plan);
    if (st != KV_OK)
        return st;
    if (plan.total_stub > 0 && (!d_stub_copy || !d_stub_rot || !aligned16(d_stub_copy) ||
                                !aligned16(d_stub_rot)))
        return KV_ERR_INVALID_ARG;
    const size_t need = composed_bytes(pool, plan);
    const bool check = g_debug_checks.load() != 0;
    if ((st = ws_ok(d_workspace, workspace_bytes,
                    need + (check ? debug_bytes(pool, num_seqs) : 0))) != KV_OK)
        return st;

    char *w = static_cast<char *>(d_workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(w);
    const size_t tbytes = table_bytes(pool, (int64_t)plan.deltas.size());
    float4 *table = reinterpret_cast<float4 *>(w + kHeaderBytes);
    SpliceTile *tiles = reinterpret_cast<SpliceTile *>(w + kHeaderBytes + tbytes);
    const size_t tiles_bytes = align256(plan.tiles.size() * sizeof(SpliceTile));
    int32_t *deltas = reinterpret_cast<int32_t *>(w + kHeaderBytes + tbytes + tiles_bytes);
    uint32_t *flags = reinterpret_cast<uint32_t *>(
        w + kHeaderBytes + tbytes + tiles_bytes + align256(plan.deltas.size() * sizeof(int32_t)));
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes, stream));
    const uint32_t *gate = nullptr;
    if (check) {
        const int64_t B = pool->block_size;
        std::vector<int32_t> used((size_t)num_seqs);
        for (int32_t q = 0; q < num_seqs; ++q)
            used[q] = (int32_t)((std::max<int64_t>(h_seq_lens[q], plan.final_len[q]) + B - 1) / B);
        KV_CUDA(launch_dup_check(pool, d_block_tables, max_blocks, used, w + need, status,
                                 stream));
        ++t_launches;
        gate = status;
    }
    if (!plan.tiles.empty()) {
        // the plan is copied from pageable host memory: the call returns once
        // the driver holds its own copy, so the vectors may go out of scope
        KV_CUDA(cudaMemcpyAsync(tiles, plan.tiles.data(), plan.tiles.size() * sizeof(SpliceTile),
                                cudaMemcpyHostToDevice, stream));
        KV_CUDA(cudaMemsetAsync(flags, 0, plan.tiles.size() * 4u, stream));
    }
    if (!plan.deltas.empty()) {
        KV_CUDA(cudaMemcpyAsync(deltas, plan.deltas.data(), plan.deltas.size() * sizeof(int32_t),
                                cudaMemcpyHostToDevice, stream));
        TableParams tp{};
        tp.d_delta = deltas;
        tp.units = (int32_t)plan.deltas.size();
        tp.half = pool->rot_head_dim / 2;
        tp.head_dim = pool->rot_head_dim;
        tp.base = pool->rope_base;
        tp.table = table;
        KV_CUDA(launch_delta_table(tp, stream));
        ++t_launches;
    }
    if (!plan.tiles.empty()) {
        ComposedParams cp{};
        cp.pool = view_of(pool);
        cp.block_tables = d_block_tables;
        cp.max_blocks = max_blocks;
        cp.stub_copy = static_cast<const char *>(d_stub_copy);
        cp.stub_rot = static_cast<const char *>(d_stub_rot);
        cp.total_stub = plan.total_stub;
        cp.tiles = tiles;
        cp.table = table;
        cp.status = status;
        cp.ticket = status + 1;
        cp.flags = flags;
        cp.num_tiles = (int64_t)plan.tiles.size();
        cp.wait_limit_ns = g_wait_limit_ns.load();
        cp.skip_publish = g_skip_publish.load();
        cp.gate = gate;
        KV_CUDA(mark(t_ev_start, stream));
        KV_CUDA(launch_splice_composed(cp, kind, stream));
        KV_CUDA(mark(t_ev_stop, stream));
        ++t_launches;
    }
    for (int32_t q = 0; q < num_seqs; ++q)
        h_seq_lens[q] = (int32_t)plan.final_len[q];
    return KV_OK;
}

kv_status kv_splice_composed_plan(const kv_pool_desc *pool, int32_t num_seqs, int32_t num_dirs,
                                  const int32_t *h_seq_lens, const int32_t *h_s_start,
                                  const int32_t *h_s_end, const int32_t *h_stub_len,
                                  kv_splice_tile *h_tiles, int64_t max_tiles, int32_t *h_deltas,
                                  int32_t max_units, int64_t *n_tiles, int32_t *n_units)
{
    static_assert(sizeof(kv_splice_tile) == sizeof(SpliceTile), "tile layout");
    if (!pool_ok(pool))
        return KV_ERR_INVALID_ARG;
    RowKind kind;
    if (!row_kind(pool, &kind))
        return KV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_dirs < 0 || !n_tiles || !n_units)
        return KV_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!h_seq_lens || (num_dirs > 0 && (!h_s_start || !h_s_end || !h_stub_len))))
        return KV_ERR_INVALID_ARG;
    ComposedPlan plan;
    if (num_dirs > 0) {
        const kv_status st = plan_composed(kind, num_seqs, num_dirs, -1, h_seq_lens, h_s_start,
                                           h_s_end, h_stub_len, plan);
        if (st != KV_OK)
            return st;
    }
    *n_tiles = (int64_t)plan.tiles.size();
    *n_units = (int32_t)plan.deltas.size();
    if (h_tiles)
        std::memcpy(h_tiles, plan.tiles.data(),
                    std::min<size_t>(plan.tiles.size(), (size_t)std::max<int64_t>(max_tiles, 0)) *
                        sizeof(SpliceTile));
    if (h_deltas)
        std::memcpy(h_deltas, plan.deltas.data(),
                    std::min<size_t>(plan.deltas.size(), (size_t)std::max<int32_t>(max_units, 0)) *
                        sizeof(int32_t));
    return KV_OK;
}

size_t kv_cdc_workspace_size(int64_t total_tokens)
{
    if (total_tokens < 0)
        return 0;
    const int64_t blocks = cdc_blocks(total_tokens);
    return kHeaderBytes + align256((size_t)blocks * kThreads * sizeof(uint32_t)) +
           4 * align256((size_t)blocks * sizeof(int64_t));
}

kv_status kv_cdc(int32_t num_streams, const int64_t *d_stream_off, int64_t total_tokens,
                 const int32_t *d_tokens, uint64_t gear_seed, uint64_t threshold,
                 uint64_t fp_seed, int64_t max_chunks, int64_t *d_chunk_end,
                 uint64_t *d_fingerprint, int64_t *d_num_chunks, void *d_workspace,
                 size_t workspace_bytes, kv_stream_t stream_)
{
    t_launches = 0;
    if (num_streams < 0 || total_tokens < 0 || max_chunks < 0 || !d_stream_off ||
        !d_num_chunks || (total_tokens > 0 && !d_tokens) ||
        (max_chunks > 0 && (!d_chunk_end || !d_fingerprint)) ||
        (num_streams == 0 && total_tokens > 0) || cdc_blocks(total_tokens) > 0x7FFFFFFF)
        return KV_ERR_INVALID_ARG;
    if (!aligned_to(d_stream_off, 8) || !aligned_to(d_tokens, 4) || !aligned_to(d_chunk_end, 8) ||
        !aligned_to(d_fingerprint, 8) || !aligned_to(d_num_chunks, 8))
        return KV_ERR_INVALID_ARG;
    kv_status st = ws_ok(d_workspace, workspace_bytes, kv_cdc_workspace_size(total_tokens));
    if (st != KV_OK)
        return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    char *w = static_cast<char *>(d_workspace);
    const int64_t blocks = cdc_blocks(total_tokens);
    CdcParams p{};
    p.stream_off = d_stream_off;
    p.num_streams = num_streams;
    p.total = total_tokens;
    p.tokens = d_tokens;
    p.gear_seed = gear_seed;
    p.threshold = threshold;
    p.fp_seed = fp_seed;
    p.max_chunks = max_chunks;
    p.chunk_end = d_chunk_end;
    p.fingerprint = d_fingerprint;
    p.num_chunks = d_num_chunks;
    p.status = reinterpret_cast<uint32_t *>(w);
    p.flags = reinterpret_cast<uint32_t *>(w + kHeaderBytes);
    p.block_count = reinterpret_cast<int64_t *>(
        w + kHeaderBytes + align256((size_t)blocks * kThreads * sizeof(uint32_t)));
    const size_t per = align256((size_t)blocks * sizeof(int64_t)) / sizeof(int64_t);
    p.block_last = p.block_count + per;
    p.block_off = p.block_last + per;
    p.block_prev_end = p.block_off + per;
    p.blocks = (int32_t)blocks;
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes, stream));
    if (blocks == 0) {
        KV_CUDA(cudaMemsetAsync(d_num_chunks, 0, sizeof(int64_t), stream));
        return KV_OK;
    }
    KV_CUDA(mark(t_ev_start, stream));
    KV_CUDA(launch_cdc(p, stream));
    KV_CUDA(mark(t_ev_stop, stream));
    t_launches = kCdcLaunches;
    return KV_OK;
}

kv_status kv_fingerprint(int64_t num_ranges, const int64_t *d_start, const int64_t *d_end,
                         int64_t total_tokens, const int32_t *d_tokens, uint64_t fp_seed,
                         uint64_t *d_fingerprint, void *d_workspace, size_t workspace_bytes,
                         kv_stream_t stream_)
{
    t_launches = 0;
    if (num_ranges < 0 || total_tokens < 0 ||
        (num_ranges > 0 && (!d_start || !d_end || !d_fingerprint || (total_tokens > 0 && !d_tokens))))
        return KV_ERR_INVALID_ARG;
    if (!aligned_to(d_start, 8) || !aligned_to(d_end, 8) || !aligned_to(d_tokens, 4) ||
        !aligned_to(d_fingerprint, 8))
        return KV_ERR_INVALID_ARG;
    kv_status st = ws_ok(d_workspace, workspace_bytes, kHeaderBytes);
    if (st != KV_OK)
        return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    KV_CUDA(cudaMemsetAsync(d_workspace, 0, kHeaderBytes, stream));
    if (num_ranges == 0)
        return KV_OK;
    FingerprintParams f{};
    f.tokens = d_tokens;
    f.total = total_tokens;
    f.start = d_start;
    f.end = d_end;
    f.count = num_ranges;
    f.seed = fp_seed;
    f.fingerprint = d_fingerprint;
    f.status = static_cast<uint32_t *>(d_workspace);
    KV_CUDA(mark(t_ev_start, stream));
    KV_CUDA(launch_fingerprint(f, stream));
    KV_CUDA(mark(t_ev_stop, stream));
    t_launches = 1;
    return KV_OK;
}

kv_status kv_get_device_status(const void *d_workspace, kv_stream_t stream)
{
    if (!d_workspace)
        return KV_ERR_WORKSPACE;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KV_ERR_CUDA;
    uint32_t st = 0;
    if (cudaMemcpy(&st, d_workspace, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess)
        return KV_ERR_CUDA;
    return static_cast<kv_status>(st);
}

void kv_set_wait_limit_ns(int64_t limit_ns)
{
    g_wait_limit_ns.store(limit_ns > 0 ? limit_ns : kDefaultWaitLimitNs);
}

void kv_set_debug_checks(int32_t on) { g_debug_checks.store(on != 0 ? 1 : 0); }

void kv_set_splice_skip_publish(int64_t ticket) { g_skip_publish.store(ticket >= 0 ? ticket : -1); }

kv_status kv_check_wait_timeout(void *d_workspace, size_t workspace_bytes, int64_t limit_ns,
                                kv_stream_t stream_)
{
    t_launches = 0;
    kv_status st = ws_ok(d_workspace, workspace_bytes, kHeaderBytes);
    if (st != KV_OK)
        return st;
    if (limit_ns <= 0)
        return KV_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    uint32_t *w = static_cast<uint32_t *>(d_workspace);
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes, stream));
    KV_CUDA(launch_wait_check(w + 2, w, limit_ns, stream));
    ++t_launches;
    return KV_OK;
}

void kv_set_kernel_events(void *start_event, void *stop_event)
{
    t_ev_start = static_cast<cudaEvent_t>(start_event);
    t_ev_stop = static_cast<cudaEvent_t>(stop_event);
}

int32_t kv_last_launch_count(void) { return t_launches; }

const char *kv_status_string(kv_status s)
{
    switch (s) {
    case KV_OK:
        return "ok";
    case KV_ERR_INVALID_ARG:
        return "invalid argument";
    case KV_ERR_OUT_OF_RANGE:
        return "index out of range";
    case KV_ERR_CAPACITY:
        return "block table too short";
    case KV_ERR_WORKSPACE:
        return "workspace missing, misaligned or too small";
    case KV_ERR_TIMEOUT:
        return "bounded wait ran out";
    case KV_ERR_CUDA:
        return "CUDA runtime error";
    case KV_ERR_UNSUPPORTED:
        return "unsupported layout";
    case KV_ERR_OVERLAP:
        return "overlapping slots or duplicate blocks (debug check)";
    }
    return "unknown status";
}

int32_t kv_version(void) { return 200; }

} // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free relocation
// ---------------------------------------------------------------------------
//
// kv_relocate needs a little device scratch (a status word and the per-chunk
// cos/sin table).  Callers that cannot allocate device memory themselves get
// it from this fixed array instead of a workspace argument.  The array is a
// device global: every GPU that loads the library keeps these bytes until
// the process exits.  Host code may not use its name as an address (on the
// host it only names a stand-in object), so its device address is fetched
// once per device with cudaGetSymbolAddress and passed to the kernels.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20; // 2 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call made with that device current).
kv_status noalloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
        return KV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return KV_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return KV_OK;
}

} // namespace

extern "C" kv_status kv_relocate_noalloc(const kv_pool_desc *src, const kv_pool_desc *dst,
                                         int32_t num_chunks, int64_t total_tokens,
                                         const int32_t *d_tok_off, const int32_t *d_src_slots,
                                         const int32_t *d_chunk_req,
                                         const int32_t *d_chunk_dst_pos, const int32_t *d_delta,
                                         const int32_t *d_block_tables, int32_t num_reqs,
                                         int32_t max_blocks, const kv_patch_desc *patch,
                                         int32_t *h_device_status, kv_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    void *scratch = nullptr;
    kv_status st = noalloc_scratch(&scratch);
    if (st != KV_OK)
        return st;
    // the shared relocation path; it clears the status word before launching
    st = relocate_impl(src, dst, num_chunks, total_tokens, d_tok_off, d_src_slots, d_chunk_req,
                       d_chunk_dst_pos, d_delta, d_block_tables, num_reqs, max_blocks, patch,
                       scratch, kNoAllocScratchBytes, stream, false);
    if (st != KV_OK || h_device_status == nullptr)
        return st;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return KV_ERR_CUDA;
    *h_device_status = static_cast<int32_t>(word);
    return KV_OK;
}

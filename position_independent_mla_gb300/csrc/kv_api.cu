// kv_api.cu -- the extern "C" entry points declared in include/kvreloc.h.
//
// Host side only: argument checks (synchronous, before anything is
// enqueued), workspace carving, per-call planning of the splice tiles, and
// the launches.  Every step of the data path runs in the kernels.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvreloc.h"
#include "kv_launch.h"

using namespace kvr;

namespace {

constexpr int64_t kDefaultWaitLimitNs = 2000000000ll;
std::atomic<int64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
thread_local int32_t t_launches = 0;
thread_local cudaEvent_t t_ev_start = nullptr, t_ev_stop = nullptr;

cudaError_t mark(cudaEvent_t ev, cudaStream_t stream)
{
    return (t_ev_start && t_ev_stop) ? cudaEventRecord(ev, stream) : cudaSuccess;
}

constexpr size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
    if (!(p->rope_base > 0.0))
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
    return v;
}

size_t table_bytes(const kv_pool_desc *p, int64_t units)
{
    return align256((size_t)units * (size_t)(p->rot_head_dim / 2) * sizeof(float4));
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
        src->rope_base != dst->rope_base)
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
    }
    PatchView pv;
    bool patched = false;
    kv_status st = patch_view(patch, &pv, &patched);
    if (st != KV_OK)
        return st;
    if (in_place && !patched)
        return KV_ERR_INVALID_ARG;
    const size_t need = kHeaderBytes + (in_place ? 0 : table_bytes(src, num_chunks));
    if ((st = ws_ok(ws, ws_bytes, need)) != KV_OK)
        return st;

    char *w = static_cast<char *>(ws);
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes, stream));
    if (total_tokens == 0)
        return KV_OK;
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
    KV_CUDA(mark(t_ev_start, stream));
    if (patch_tc_supported(rp, kind)) {
        KV_CUDA(launch_patch_tc(rp, kind, stream));
        t_launches += patch_tc_launches(kind);
    } else {
        KV_CUDA(launch_relocate(rp, kind, stream));
        ++t_launches;
    }
    KV_CUDA(mark(t_ev_stop, stream));
    return KV_OK;
}

} // namespace

extern "C" {

size_t kv_workspace_size(const kv_pool_desc *pool, int64_t max_rows, int32_t max_units)
{
    RowKind kind;
    if (!pool_ok(pool) || !row_kind(pool, &kind) || max_rows < 0 || max_units < 0)
        return 0;
    const int64_t T = tile_rows(kind);
    const int64_t units = std::max<int64_t>(max_units, 1);
    const int64_t flags = (int64_t)pool->num_layers * ((max_rows + T - 1) / T + units);
    return (size_t)kHeaderBytes + table_bytes(pool, units) + align256((size_t)flags * 4u);
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

kv_status kv_splice(const kv_pool_desc *pool, int32_t num_seqs, const int32_t *d_block_tables,
                    int32_t max_blocks, int32_t *h_seq_lens, const int32_t *h_s_start,
                    const int32_t *h_s_end, const int32_t *h_stub_len, const void *d_stub_copy,
                    const void *d_stub_rot, kv_mode mode, void *d_workspace,
                    size_t workspace_bytes, kv_stream_t stream_)
{
    t_launches = 0;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!pool_ok(pool) || num_seqs < 0 || (mode != KV_AMORTIZE && mode != KV_FORGET))
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
    if (!d_block_tables || max_blocks <= 0)
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

    // plan: launches of up to kMaxSeqsPerLaunch sequences each
    const int T = tile_rows(kind);
    const int L = pool->num_layers;
    std::vector<SpliceParams> plans;
    int64_t stub_base = 0, max_flags = 0;
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
            S.n_shift = S.delta == 0 ? 0 : (int32_t)((down + T - 1) / T);
            S.n_stub = (S.n_r + T - 1) / T;
            S.bt_row = q;
            S.ticket_base = tickets;
            S.flag_base = flags;
            S.stub_base = stub_base;
            tickets += S.n_shift + S.n_stub;
            flags += S.n_shift;
            stub_base += S.n_r;
        }
        sp.total_tickets = tickets;
        max_flags = std::max(max_flags, flags);
        plans.push_back(sp);
    }
    const size_t tbytes = table_bytes(pool, std::min(num_seqs, kMaxSeqsPerLaunch));
    const size_t need = kHeaderBytes + tbytes + align256((size_t)max_flags * 4u);
    kv_status st = ws_ok(d_workspace, workspace_bytes, need);
    if (st != KV_OK)
        return st;

    char *w = static_cast<char *>(d_workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(w);
    uint32_t *ticket = status + 1;
    float4 *table = reinterpret_cast<float4 *>(w + kHeaderBytes);
    uint32_t *flags = reinterpret_cast<uint32_t *>(w + kHeaderBytes + tbytes);
    KV_CUDA(cudaMemsetAsync(w, 0, kHeaderBytes, stream));
    const int64_t limit = g_wait_limit_ns.load();
    bool marked = false;
    for (SpliceParams &sp : plans) {
        if (sp.total_tickets == 0)
            continue;
        int64_t nflags = 0;
        for (int i = 0; i < sp.num_seqs; ++i)
            nflags += sp.seq[i].n_shift;
        KV_CUDA(cudaMemsetAsync(ticket, 0, sizeof(uint32_t), stream));
        if (nflags > 0)
            KV_CUDA(cudaMemsetAsync(flags, 0, (size_t)nflags * 4u, stream));
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
        if (!marked) {
            KV_CUDA(mark(t_ev_start, stream));
            marked = true;
        }
        KV_CUDA(launch_splice(sp, kind, stream));
        ++t_launches;
    }
    if (marked)
        KV_CUDA(mark(t_ev_stop, stream));
    for (int q = 0; q < num_seqs; ++q)
        h_seq_lens[q] += h_stub_len[q] - (h_s_end[q] - h_s_start[q]);
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
    }
    return "unknown status";
}

int32_t kv_version(void) { return 100; }

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

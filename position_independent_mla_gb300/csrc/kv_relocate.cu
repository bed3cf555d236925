// kv_relocate.cu -- δ-table construction and the relocation / patch kernels.
//
// Relocation (Irminsul §2.2, Kamera §2): every token of every chunk is read
// from its source slot and written to the slot of its target position; the
// verbatim part is copied, each rotary head is turned by R(δ_chunk), and an
// optional rank-m patch U_m V_mᵀ is added before the single rounding.  One
// block handles T consecutive tokens of the call for all layers, so the
// per-token index work (chunk search, block-table lookup) and the cos/sin
// rows are set up once and reused for every layer.
#include <algorithm>

#include "kv_launch.h"
#include "kv_tiles.cuh"

namespace kvr {

// ---------------------------------------------------------------------------
// δ-table: cos/sin of δ_u·θ_j in fp64, stored as two-part fp32
// ---------------------------------------------------------------------------

__global__ void delta_table_kernel(const __grid_constant__ TableParams p)
{
    // 64-bit indices and a grid-stride loop: units * half may exceed 2^31
    const int64_t n = (int64_t)p.units * p.half;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t u = i / p.half;
        const int j = (int)(i % p.half);
        const int32_t delta = p.d_delta ? p.d_delta[u] : p.h_delta[u];
        p.table[i] = delta_entry(delta, j, p.head_dim, p.base);
    }
}

cudaError_t launch_delta_table(const TableParams &p, cudaStream_t stream)
{
    const int64_t n = (int64_t)p.units * p.half;
    if (n <= 0)
        return cudaSuccess;
    // at most 152 SMs x 16 blocks of 256 threads; larger tables loop
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
    delta_table_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Relocation / in-place patch
// ---------------------------------------------------------------------------

template <class G, bool PATCH, bool IL>
__global__ void __launch_bounds__(kThreads, G::kMinBlocks) relocate_kernel(const __grid_constant__ RelocParams p)
{
    __shared__ int64_t s_src[G::T];
    __shared__ int64_t s_dst[G::T];
    __shared__ int64_t s_tok[G::T];   // U row of the row's token (patch)
    __shared__ int32_t s_chunk[G::T]; // chunk of the row (δ-table row)
    __shared__ int32_t s_vslot[G::T]; // V slot of the row's chunk (patch)
    __shared__ int32_t s_ident[G::T];
    __shared__ float4 s_cs[G::T][G::kCsRow];

    if (gate_closed(p.gate))
        return; // a debug check found an overlap: store nothing
    const int tid = threadIdx.x;
    const int64_t tile0 = (int64_t)blockIdx.x * G::T;

    if (blockIdx.x == 0 && tid == 0) {
        if (p.tok_off[0] != 0 || p.tok_off[p.num_chunks] != p.total_tokens)
            set_status(p.status, kStatusOutOfRange);
    }
    if (tid < G::T) {
        const int64_t t = tile0 + tid;
        int64_t src = -1, dst = -1;
        int32_t c = 0, ident = 1;
        if (t < p.total_tokens) {
            // chunk holding token t: the largest c with tok_off[c] <= t
            int lo = 0, hi = p.num_chunks - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.tok_off[mid] <= t)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            c = lo;
            const int64_t off = t - p.tok_off[c];
            const int32_t req = p.chunk_req[c];
            bool ok = off >= 0 && t < p.tok_off[c + 1] && req >= 0 && req < p.num_reqs;
            if (ok) {
                dst = slot_of(p.block_tables + (int64_t)req * p.max_blocks, p.max_blocks,
                              p.dst.block, p.dst.num_blocks, (int64_t)p.chunk_dst_pos[c] + off);
                if (p.in_place) {
                    src = dst;
                } else {
                    const int64_t s = p.src_slots[t];
                    src = (s >= 0 && s < p.src.num_slots) ? s : -1;
                }
                ok = src >= 0 && dst >= 0;
            }
            if (!ok) {
                set_status(p.status, kStatusOutOfRange);
                src = dst = -1;
            }
            ident = p.in_place ? 1 : (p.delta[c] == 0);
        }
        s_src[tid] = src;
        s_dst[tid] = dst;
        // the patch's U row and V slot: call order, or the caller's maps
        const bool live = t < p.total_tokens;
        const int64_t urow = (live && p.patch.u_chunk_tok)
                                 ? p.patch.u_chunk_tok[c] + (t - p.tok_off[c])
                                 : t;
        const int32_t vslot = (live && p.patch.v_chunk) ? p.patch.v_chunk[c] : c;
        if (PATCH && src >= 0 && !patch_rows_ok(p.patch, urow, vslot)) {
            // a factor row or slot outside the caller's stated extents
            set_status(p.status, kStatusOutOfRange);
            s_src[tid] = s_dst[tid] = -1;
        }
        s_tok[tid] = urow;
        s_chunk[tid] = c;
        s_vslot[tid] = vslot;
        s_ident[tid] = ident;
    }
    __syncthreads();
    if (!p.in_place) {
        for (int i = tid; i < G::T * G::kHalf; i += kThreads) {
            const int r = i / G::kHalf, j = i % G::kHalf;
            stage_cs<G, CsOrder<G, PATCH, IL>::kPacked>(
                s_cs[r], j, (s_src[r] >= 0 && !s_ident[r])
                                ? p.table[(int64_t)s_chunk[r] * G::kHalf + j]
                                : make_float4(1.f, 0.f, 0.f, 0.f));
        }
        __syncthreads();
    }

    PatchAt pa{&p.patch, 0, s_tok, s_vslot};
    for (int l = 0; l < p.src.num_layers; ++l) {
        const RowsAt from{p.src.copy + l * p.src.copy_ls, p.src.copy_ss,
                          p.src.rot + l * p.src.rot_ls, p.src.rot_ss};
        const RowsAt to{p.dst.copy + l * p.dst.copy_ls, p.dst.copy_ss,
                        p.dst.rot + l * p.dst.rot_ls, p.dst.rot_ss};
        TileRegs<G> regs;
        load_tile<G>(from, s_src, regs);
        pa.layer = l;
        store_tile<G, PATCH, true, IL>(to, s_dst, regs, &s_cs[0][0], G::kCsRow, s_ident, pa);
    }
}

template <class G>
static cudaError_t launch_reloc_shape(const RelocParams &p, cudaStream_t stream)
{
    const int64_t tiles = (p.total_tokens + G::T - 1) / G::T;
    if (tiles == 0)
        return cudaSuccess;
    if (tiles > 0x7FFFFFFFll)
        return cudaErrorInvalidConfiguration;
    return with_bool(p.dst.il != 0, [&](auto il) {
        constexpr bool IL = decltype(il)::value;
        if (p.patched)
            relocate_kernel<G, true, IL><<<(unsigned)tiles, kThreads, 0, stream>>>(p);
        else
            relocate_kernel<G, false, IL><<<(unsigned)tiles, kThreads, 0, stream>>>(p);
        return cudaGetLastError();
    });
}

cudaError_t launch_relocate(const RelocParams &p, RowKind kind, cudaStream_t stream)
{
    return with_geo(kind, [&](auto g) {
        return launch_reloc_shape<typename decltype(g)::type>(p, stream);
    });
}

} // namespace kvr
